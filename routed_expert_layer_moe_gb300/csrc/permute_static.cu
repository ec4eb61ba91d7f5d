// Dispatch without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: an inference-engine plugin whose enqueue step must not allocate, code
// that runs while its stream is being captured into a CUDA graph (cudaMalloc is
// not an operation a capture can record), or a host framework whose device
// memory is owned entirely by its own pool.  moe_permute_no_workspace serves
// them: it runs the same kernels as moe_permute, but its scratch lives in a
// fixed array compiled into this library, so the caller passes only its inputs
// and outputs.
//
// The array is a file-scope __device__ variable.  Every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Host code
// may not hand the symbol itself to a kernel (on the host it names a host-side
// stand-in, not device memory), so the first call on each device looks up the
// device address with cudaGetSymbolAddress while that device is current and
// keeps it.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB

__device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  void* ptr[kMaxDevices] = {};
  std::mutex mu;
};

ScratchAddress& scratch_address() {
  static ScratchAddress a;
  return a;
}

// Device address of g_permute_scratch on the current device, looked up once per device.
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  ScratchAddress& a = scratch_address();
  std::lock_guard<std::mutex> lock(a.mu);
  if (!a.ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    a.ptr[dev] = p;
  }
  *out = a.ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_no_workspace(const moe_problem* p, const int32_t* ids, const void* x,
                                               const int32_t* phys_to_log, int32_t* masked_m, int32_t* offsets,
                                               int32_t* row_of, int32_t* src_of, void* xg, float* xg_scales,
                                               int32_t* err_flag, moe_stream_t stream) {
  const moe_status st = moe_check_problem(p);
  if (st != MOE_OK) return st;
  if (!masked_m || !offsets || !err_flag) return MOE_ERR_INVALID;
  if (p->T > 0 && (!ids || !x || !row_of || !src_of || !xg)) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && p->T > 0 && !xg_scales) return MOE_ERR_INVALID;
  if (!phys_to_log && p->P != p->E) return MOE_ERR_INVALID;
  if (p->T > 0 && (!aligned16(x) || !aligned16(xg))) return MOE_ERR_UNSUPPORTED;
  // the scratch this problem needs must fit in the fixed array
  if (permute_workspace_bytes(*p) > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return (moe_status)launch_permute(*p, ids, x, phys_to_log, masked_m, offsets, row_of, src_of, xg, xg_scales,
                                    err_flag, scratch, (cudaStream_t)stream);
}

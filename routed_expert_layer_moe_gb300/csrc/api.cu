// The extern "C" entry points of moe.h: argument checks on the host, then the
// launches.  Nothing here allocates device memory or synchronises.
#include <mutex>

#include "common.cuh"

namespace moe {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCache {
  DeviceInfo info[kMaxDevices];
  bool valid[kMaxDevices] = {};
  std::mutex mu;
};

DeviceCache& cache() {
  static DeviceCache c;
  return c;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

const DeviceInfo& device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  DeviceCache& c = cache();
  if (dev >= 0 && dev < kMaxDevices && c.valid[dev]) return c.info[dev];
  std::lock_guard<std::mutex> lock(c.mu);
  static DeviceInfo fallback{};
  if (dev < 0 || dev >= kMaxDevices) {
    cudaDeviceGetAttribute(&fallback.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&fallback.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return fallback;
  }
  DeviceInfo d{};
  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  c.info[dev] = d;
  c.valid[dev] = true;
  return c.info[dev];
}

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint64_t inner, uint64_t outer,
                           uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, const void* base) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace moe

using namespace moe;

namespace {

int check_problem(const moe_problem* p) {
  if (!p) return MOE_ERR_INVALID;
  const moe_problem& q = *p;
  if (q.T < 0 || q.H <= 0 || q.I <= 0 || q.E <= 0 || q.E > 1024 || q.K <= 0 || q.K > 32 || q.K > q.E)
    return MOE_ERR_INVALID;
  if (q.P < q.E || q.has_shared < 0 || q.has_shared > 1 || q.P + q.has_shared > 1024) return MOE_ERR_INVALID;
  if (q.layout != MOE_LAYOUT_MASKED && q.layout != MOE_LAYOUT_CONTIG) return MOE_ERR_INVALID;
  if (q.layout == MOE_LAYOUT_MASKED) {
    if (q.M_max <= 0) return MOE_ERR_INVALID;
    if (q.has_shared && q.M_max < q.T) return MOE_ERR_INVALID;
  }
  if (q.act < MOE_F32 || q.act > MOE_E4M3 || q.wt < MOE_F32 || q.wt > MOE_E2M1 || q.out < MOE_F32 ||
      q.out > MOE_E4M3)
    return MOE_ERR_INVALID;
  // products that must fit the 32-bit row and element indices used on the device
  if ((int64_t)q.T * q.K > (1 << 30) || grouped_rows(q) * (int64_t)(q.H > q.I ? q.H : q.I) > (1LL << 40))
    return MOE_ERR_INVALID;
  if (grouped_rows(q) >= (1LL << 31)) return MOE_ERR_INVALID;
  // supported dtype combinations
  const bool f32 = q.act == MOE_F32 && q.wt == MOE_F32 && q.out == MOE_F32;
  const bool bf16 = q.act == MOE_BF16 && q.wt == MOE_BF16 && q.out == MOE_BF16;
  const bool f8 = q.act == MOE_BF16 && fp8_acts(q) && q.out == MOE_BF16;  // FP8 or FP4 weights
  if (!(f32 || bf16 || f8)) return MOE_ERR_UNSUPPORTED;
  if (f32 && (q.H % 4 || q.I % 4)) return MOE_ERR_UNSUPPORTED;
  if ((bf16 || f8) && (q.H % 128 || q.I % 128)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t ws_bytes(const moe_problem& p) {
  const size_t a = permute_workspace_bytes(p);
  const size_t b = gemm_workspace_bytes(p);
  return a > b ? a : b;
}

moe_status launched(int r) {
  if (r != MOE_OK) return (moe_status)r;
  return MOE_OK;
}

}  // namespace

extern "C" {

int32_t moe_version(void) { return (1 << 16) | 0; }

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK:
      return "ok";
    case MOE_ERR_INVALID:
      return "invalid argument";
    case MOE_ERR_UNSUPPORTED:
      return "unsupported problem";
    case MOE_ERR_CUDA:
      return "CUDA error";
    case MOE_ERR_WORKSPACE:
      return "workspace too small";
    default:
      return "unknown status";
  }
}

moe_status moe_check_problem(const moe_problem* p) { return (moe_status)check_problem(p); }

int64_t moe_grouped_rows(const moe_problem* p) {
  if (check_problem(p) != MOE_OK) return -1;
  return grouped_rows(*p);
}

size_t moe_workspace_bytes(const moe_problem* p) {
  if (check_problem(p) != MOE_OK) return 0;
  return ws_bytes(*p);
}

int32_t moe_gemm_tile_rows(const moe_problem* p, int32_t step) {
  if (check_problem(p) != MOE_OK || (step != 3 && step != 4)) return 0;
  return gemm_tile_rows(*p, step == 3 ? MODE_SWIGLU : MODE_DOWN);
}

moe_status moe_route_topk(const moe_problem* p, const float* logits, int32_t* ids, float* w, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (p->T > 0 && (!logits || !ids || !w)) return MOE_ERR_INVALID;
  return launched(launch_route(*p, logits, ids, w, (cudaStream_t)stream));
}

moe_status moe_route_grouped_topk(const moe_problem* p, const float* logits, const float* bias, int32_t n_group,
                                  int32_t topk_group, int32_t renormalize, float scale, int32_t* ids, float* w,
                                  moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (n_group < 1 || n_group > 32 || p->E % n_group || topk_group < 1 || topk_group > n_group ||
      p->K > topk_group * (p->E / n_group))
    return MOE_ERR_INVALID;
  if (p->T > 0 && (!logits || !ids || !w)) return MOE_ERR_INVALID;
  return launched(launch_route_grouped(*p, logits, bias, n_group, topk_group, renormalize != 0, scale, ids, w,
                                       (cudaStream_t)stream));
}

moe_status moe_permute(const moe_problem* p, const int32_t* ids, const void* x, const int32_t* phys_to_log,
                       int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                       float* xg_scales, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!masked_m || !offsets || !err_flag || !workspace) return MOE_ERR_INVALID;
  if (p->T > 0 && (!ids || !x || !row_of || !src_of || !xg)) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && p->T > 0 && !xg_scales) return MOE_ERR_INVALID;
  if (!phys_to_log && p->P != p->E) return MOE_ERR_INVALID;
  if (p->T > 0 && (!aligned16(x) || !aligned16(xg))) return MOE_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_bytes(*p)) return MOE_ERR_WORKSPACE;
  return launched(launch_permute(*p, ids, x, phys_to_log, masked_m, offsets, row_of, src_of, xg, xg_scales,
                                 err_flag, workspace, (cudaStream_t)stream));
}

static moe_status gemm_call(const moe_problem* p, int mode, const void* act, const float* act_scales,
                            const void* w, const float* w_scales, const int32_t* masked_m, const int32_t* offsets,
                            void* out, float* out_scales, int32_t* err_flag, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!act || !w || !masked_m || !offsets || !out || !err_flag) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && (!act_scales || !w_scales)) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && mode == MODE_SWIGLU && !out_scales) return MOE_ERR_INVALID;
  if (!aligned16(act) || !aligned16(w) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
  // packed 4-bit tensor maps want a 32-byte aligned base
  if (p->wt == MOE_E2M1 && (reinterpret_cast<uintptr_t>(w) & 31u)) return MOE_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_bytes(*p) || (ws_bytes(*p) > 0 && !workspace)) return MOE_ERR_WORKSPACE;
  return launched(launch_gemm(*p, mode, act, act_scales, w, w_scales, masked_m, offsets, out, out_scales, err_flag,
                              workspace, (cudaStream_t)stream));
}

moe_status moe_grouped_swiglu_gemm(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                                   const float* w13_scales, const int32_t* masked_m, const int32_t* offsets,
                                   void* hg, float* hg_scales, int32_t* err_flag, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream) {
  return gemm_call(p, MODE_SWIGLU, xg, xg_scales, w13, w13_scales, masked_m, offsets, hg, hg_scales, err_flag,
                   workspace, workspace_bytes, stream);
}

moe_status moe_grouped_down_gemm(const moe_problem* p, const void* hg, const float* hg_scales, const void* w2,
                                 const float* w2_scales, const int32_t* masked_m, const int32_t* offsets,
                                 void* yg, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  return gemm_call(p, MODE_DOWN, hg, hg_scales, w2, w2_scales, masked_m, offsets, yg, nullptr, err_flag, workspace,
                   workspace_bytes, stream);
}

moe_status moe_grouped_ffn(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                           const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                           const int32_t* offsets, void* hg, float* hg_scales, void* yg, int32_t* err_flag,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!xg || !w13 || !w2 || !masked_m || !offsets || !hg || !yg || !err_flag) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && (!xg_scales || !w13_scales || !w2_scales || !hg_scales)) return MOE_ERR_INVALID;
  if (!aligned16(xg) || !aligned16(w13) || !aligned16(w2) || !aligned16(hg) || !aligned16(yg))
    return MOE_ERR_UNSUPPORTED;
  if (p->wt == MOE_E2M1 && ((reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2)) & 31u))
    return MOE_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_bytes(*p) || (ws_bytes(*p) > 0 && !workspace)) return MOE_ERR_WORKSPACE;
  return launched(launch_grouped_ffn(*p, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, hg,
                                     hg_scales, yg, err_flag, workspace, (cudaStream_t)stream));
}

moe_status moe_route_permute(const moe_problem* p, const float* logits, const void* x, const int32_t* phys_to_log,
                             int32_t* ids, float* w, int32_t* masked_m, int32_t* offsets, int32_t* row_of,
                             int32_t* src_of, void* xg, float* xg_scales, int32_t* err_flag, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!masked_m || !offsets || !err_flag || !workspace) return MOE_ERR_INVALID;
  if (p->T > 0 && (!logits || !ids || !w || !x || !row_of || !src_of || !xg)) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && p->T > 0 && !xg_scales) return MOE_ERR_INVALID;
  if (!phys_to_log && p->P != p->E) return MOE_ERR_INVALID;
  if (p->T > 0 && (!aligned16(x) || !aligned16(xg))) return MOE_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_bytes(*p)) return MOE_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  if (route_permute_one_launch(*p, phys_to_log))
    return launched(launch_route_permute_small(*p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg,
                                               xg_scales, err_flag, st));
  r = launch_route(*p, logits, ids, w, st);
  if (r) return (moe_status)r;
  return launched(launch_permute(*p, ids, x, phys_to_log, masked_m, offsets, row_of, src_of, xg, xg_scales, err_flag,
                                 workspace, st));
}

moe_status moe_ffn_combine(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                           const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                           const int32_t* offsets, const int32_t* row_of, const float* w, void* hg, float* hg_scales,
                           void* yg, void* out, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!xg || !w13 || !w2 || !masked_m || !offsets || !hg || !yg || !err_flag) return MOE_ERR_INVALID;
  if (p->T > 0 && (!row_of || !w || !out)) return MOE_ERR_INVALID;
  if (fp8_acts(*p) && (!xg_scales || !w13_scales || !w2_scales || !hg_scales)) return MOE_ERR_INVALID;
  if (!aligned16(xg) || !aligned16(w13) || !aligned16(w2) || !aligned16(hg) || !aligned16(yg) ||
      (p->T > 0 && !aligned16(out)))
    return MOE_ERR_UNSUPPORTED;
  if (p->wt == MOE_E2M1 && ((reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2)) & 31u))
    return MOE_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_bytes(*p) || (ws_bytes(*p) > 0 && !workspace)) return MOE_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  const CombineArgs comb{row_of, w, out};
  if (p->wt == MOE_BF16)  // one launch for both GEMMs
    return launched(launch_grouped_ffn(*p, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, hg,
                                       hg_scales, yg, err_flag, workspace, st, &comb));
  r = launch_gemm(*p, MODE_SWIGLU, xg, xg_scales, w13, w13_scales, masked_m, offsets, hg, hg_scales, err_flag,
                  workspace, st);
  if (r) return (moe_status)r;
  return launched(launch_gemm(*p, MODE_DOWN, hg, hg_scales, w2, w2_scales, masked_m, offsets, yg, nullptr, err_flag,
                              workspace, st, &comb));
}

moe_status moe_combine(const moe_problem* p, const void* yg, const int32_t* row_of, const float* w, void* out,
                       moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (p->T > 0 && (!yg || !row_of || !w || !out)) return MOE_ERR_INVALID;
  if (p->T > 0 && (!aligned16(yg) || !aligned16(out))) return MOE_ERR_UNSUPPORTED;
  return launched(launch_combine(*p, yg, row_of, w, out, (cudaStream_t)stream));
}

moe_status moe_eplb_record(const moe_problem* p, const int32_t* masked_m, int64_t pass, int32_t window,
                           int32_t* load_window, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!masked_m || !load_window || window < 1 || pass < 0) return MOE_ERR_INVALID;
  return launched(launch_eplb_record(*p, masked_m, pass, window, load_window, (cudaStream_t)stream));
}

moe_status moe_eplb_rebalance(const moe_problem* p, const int32_t* load_window, int32_t window,
                              const int32_t* phys_to_log, int64_t* logical_load, int32_t* new_phys_to_log,
                              int32_t* err_flag, moe_stream_t stream) {
  int r = check_problem(p);
  if (r) return (moe_status)r;
  if (!load_window || window < 1 || !logical_load || !new_phys_to_log || !err_flag) return MOE_ERR_INVALID;
  if (!phys_to_log && p->P != p->E) return MOE_ERR_INVALID;
  if (p->P - p->E > p->E) return MOE_ERR_INVALID;  // each extra slot holds a different expert
  return launched(launch_eplb_rebalance(*p, load_window, window, phys_to_log, logical_load, new_phys_to_log,
                                        err_flag, (cudaStream_t)stream));
}

moe_status moe_selftest_bounded_wait(int64_t cycles, int32_t* err_flag, moe_stream_t stream) {
  if (!err_flag || cycles < 1 || cycles > 4000000000LL) return MOE_ERR_INVALID;
  return launched(launch_bounded_wait_selftest((long long)cycles, err_flag, (cudaStream_t)stream));
}

int32_t moe_eplb_invert(int32_t P, int32_t E, const int32_t* p2l, int32_t R, int32_t* l2p, int32_t* rc) {
  if (P < 0 || E <= 0 || R <= 0 || !p2l || !l2p || !rc) return MOE_ERR_INVALID;
  for (int e = 0; e < E; ++e) {
    rc[e] = 0;
    for (int j = 0; j < R; ++j) l2p[(size_t)e * R + j] = -1;
  }
  int32_t maxr = 0;
  for (int s = 0; s < P; ++s) {
    const int e = p2l[s];
    if (e < 0 || e >= E || rc[e] >= R) return MOE_ERR_INVALID;
    l2p[(size_t)e * R + rc[e]] = s;
    rc[e] += 1;
    if (rc[e] > maxr) maxr = rc[e];
  }
  return maxr;
}

}  // extern "C"

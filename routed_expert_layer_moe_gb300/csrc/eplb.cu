// EPLB load statistics on the device.
//
// "vLLM EPLB", section 1.2: expert_load_pass holds each physical slot's token
// count of one forward pass (here the per-slot row counts masked_m written by
// the dispatch), expert_load_window keeps the passes of a window, and a
// rebalance folds the window's physical loads onto the logical experts through
// physical_to_logical_map before re-assigning replicas.  Replica policy on one
// GPU: slots 0..E-1 keep experts 0..E-1, the P-E extra slots hold the P-E
// experts with the largest load (descending, ties to the lower index).
#include "common.cuh"

namespace moe {
namespace {

__global__ void eplb_record_kernel(const int32_t* __restrict__ masked_m, int P, int row, int32_t* __restrict__ window) {
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < P; s += gridDim.x * blockDim.x)
    window[(size_t)row * P + s] = masked_m[s];
}

// One CTA of 1024 threads; E <= 1024.
__global__ void __launch_bounds__(1024) eplb_rebalance_kernel(const int32_t* __restrict__ window, int W, int P, int E,
                                                             const int32_t* __restrict__ p2l,
                                                             int64_t* __restrict__ logical_load,
                                                             int32_t* __restrict__ new_p2l, int32_t* err) {
  __shared__ unsigned long long load[1024];
  for (int e = threadIdx.x; e < E; e += blockDim.x) load[e] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < P; s += blockDim.x) {
    const int e = p2l ? p2l[s] : s;
    if (e < 0 || e >= E) {
      atomicOr(err, MOE_FLAG_BAD_MAP);
      continue;
    }
    long long sum = 0;
    for (int w = 0; w < W; ++w) sum += window[(size_t)w * P + s];
    atomicAdd(&load[e], (unsigned long long)sum);  // integer sums: the order does not matter
  }
  __syncthreads();
  const int R = P - E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const unsigned long long v = load[e];
    logical_load[e] = (int64_t)v;
    new_p2l[e] = e;
    int rank = 0;  // experts ahead of e: larger load, or equal load and lower index
    for (int f = 0; f < E; ++f) {
      const unsigned long long u = load[f];
      rank += (u > v) || (u == v && f < e);
    }
    if (rank < R) new_p2l[E + rank] = e;
  }
}

}  // namespace

int launch_eplb_record(const moe_problem& p, const int32_t* masked_m, int64_t pass, int window, int32_t* load_window,
                       cudaStream_t st) {
  const int row = (int)(pass % window);
  eplb_record_kernel<<<(p.P + 255) / 256, 256, 0, st>>>(masked_m, p.P, row, load_window);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_eplb_rebalance(const moe_problem& p, const int32_t* load_window, int window, const int32_t* p2l,
                          int64_t* logical_load, int32_t* new_p2l, int32_t* err, cudaStream_t st) {
  eplb_rebalance_kernel<<<1, 1024, 0, st>>>(load_window, window, p.P, p.E, p2l, logical_load, new_p2l, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Diagnostic: the bounded wait every kernel of the library uses, run to its limit.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

// One thread waits on an mbarrier that nothing completes, with a bound of `cycles` SM
// cycles; on expiry it reports MOE_FLAG_TIMEOUT as the layer kernels do, and returns.
__global__ void bounded_wait_kernel(long long cycles, int32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0, &abort_flag, cycles)) atomicOr(err, MOE_FLAG_TIMEOUT);
}

}  // namespace

int launch_bounded_wait_selftest(long long cycles, int32_t* err, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>(cycles, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

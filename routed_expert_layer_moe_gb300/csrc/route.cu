// Step 1: softmax top-K routing, one warp per token.
//
// "MoE inference and expert parallelism" (blog.vllbc.top), routing section,
// Table 3-1: softmax scoring, top-K, renormalize=True.  Selection is made on
// the fp32 logits themselves (softmax is strictly increasing, so the chosen
// set is the same and no rounding of exp can create new ties); ties go to the
// lower expert index.  Weights: exp(l_k - l_max) / sum over the chosen K.
#include "common.cuh"

namespace moe {
namespace {

template <int PER>  // logits held per lane: E <= 32 * PER
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  float v[PER];
  uint32_t avail = 0;  // bit i: expert lane + 32*i not yet chosen
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(l + e) : -INFINITY;
    if (e < E) avail |= 1u << i;
  }
  int my_id = 0;
  float my_val = 0.0f;
  for (int k = 0; k < K; ++k) {
    // best remaining candidate of this lane: largest value, lowest index on ties
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if ((avail >> i) & 1u) {
        if (be == 0x7fffffff || v[i] > bv) {
          bv = v[i];
          be = lane + 32 * i;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
    if (lane == k) {
      my_id = be;
      my_val = bv;
    }
  }
  const float lmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = (lane < K) ? expf(my_val - lmax) : 0.0f;
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);  // fixed order k = 0..K-1
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_id;
    w[(size_t)t * K + lane] = ex / sum;
  }
}

template <int PER>
void launch_route_per(const moe_problem& p, const float* logits, int32_t* ids, float* w, cudaStream_t st) {
  const int threads = 256;
  const int blocks = (int)(((int64_t)p.T * 32 + threads - 1) / threads);
  route_topk_kernel<PER><<<blocks, threads, 0, st>>>(logits, p.T, p.E, p.K, ids, w);
}

}  // namespace

int launch_route(const moe_problem& p, const float* logits, int32_t* ids, float* w, cudaStream_t st) {
  if (p.T == 0) return MOE_OK;
  const int per = (p.E + 31) / 32;
  if (per <= 1)
    launch_route_per<1>(p, logits, ids, w, st);
  else if (per <= 2)
    launch_route_per<2>(p, logits, ids, w, st);
  else if (per <= 4)
    launch_route_per<4>(p, logits, ids, w, st);
  else if (per <= 8)
    launch_route_per<8>(p, logits, ids, w, st);
  else if (per <= 16)
    launch_route_per<16>(p, logits, ids, w, st);
  else
    launch_route_per<32>(p, logits, ids, w, st);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// Softmax top-K of one token by one warp, shared by the router kernel and the
// fused route + dispatch kernel (both produce the same ids and weights).
//
// "MoE inference and expert parallelism" (blog.vllbc.top), routing section,
// Table 3-1: softmax scoring, top-K, renormalize=True.  Selection is made on the
// fp32 logits (softmax is strictly increasing, so the chosen set is the same and
// no rounding of exp can create new ties); ties go to the lower expert index.
// Weights: exp(l_k - l_max) / sum over the chosen K, summed in k order.
#pragma once

#include "common.cuh"

namespace moe {

// Logits of one token, PER per lane: v[i] = l[lane + 32 i] (-inf past E); bit i of the result
// marks an expert that exists.
template <int PER>
__device__ __forceinline__ uint32_t route_load(const float* __restrict__ l, int E, int lane, float (&v)[PER]) {
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(l + e) : -INFINITY;
    if (e < E) avail |= 1u << i;
  }
  return avail;
}

// K rounds of a warp-wide arg-max over the experts still marked in avail (largest value,
// lowest index on ties); lane k < K ends with the k-th chosen expert and its logit.
template <int PER>
__device__ __forceinline__ void route_select(const float (&v)[PER], uint32_t avail, int K, int lane, int& my_id,
                                             float& my_val) {
  my_id = 0;
  my_val = 0.0f;
  for (int k = 0; k < K; ++k) {
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
}

// Weight of lane k < K's expert: exp(l_k - l_0) / sum_{j<K} exp(l_j - l_0) (l_0 the largest).
__device__ __forceinline__ float route_weight(float my_val, int K, int lane) {
  const float lmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = (lane < K) ? expf(my_val - lmax) : 0.0f;
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);  // fixed order k = 0..K-1
  return ex / sum;
}

}  // namespace moe

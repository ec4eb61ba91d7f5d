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

// "MoE inference and expert parallelism", routing section, Table 3-1 (DeepSeek-V3):
// sigmoid scores, e_score_correction_bias used for the choice only, grouped
// top-k (the best topk_group of n_group contiguous expert groups, a group
// scored by its best biased score, then the K best experts inside them).  The
// keys are formed and compared in fp64 (ties to the lower index); weights are
// the unbiased scores of the chosen experts, renormalised if asked, times
// `scale`.  One CTA per token: its 128 threads evaluate the E fp64 sigmoids
// (fp64 throughput is low, so they are spread over the whole CTA), then warp 0
// makes the choices from shared memory.
constexpr int GROUPED_THREADS = 128;

template <int PER>  // keys held per lane of warp 0: E <= 32 * PER
__global__ void __launch_bounds__(GROUPED_THREADS) route_grouped_kernel(const float* __restrict__ logits,
                                                                        const float* __restrict__ bias, int T, int E,
                                                                        int K, int n_group, int topk_group,
                                                                        int renorm, float scale,
                                                                        int32_t* __restrict__ ids,
                                                                        float* __restrict__ w) {
  __shared__ double s_sc[1024], s_key[1024];
  const int t = blockIdx.x;
  const float* l = logits + (size_t)t * E;
  for (int e = threadIdx.x; e < E; e += GROUPED_THREADS) {
    const double sc = 1.0 / (1.0 + exp(-(double)__ldg(l + e)));
    s_sc[e] = sc;
    s_key[e] = sc + (bias ? (double)__ldg(bias + e) : 0.0);
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int gs = E / n_group;
  double key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? s_key[e] : -INFINITY;
  }
  // group maxima: lane g keeps the score of group g
  double gmine = -INFINITY;
  for (int g = 0; g < n_group; ++g) {
    double m = -INFINITY;
    const int e_lo = g * gs, e_hi = e_lo + gs;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e >= e_lo && e < e_hi) m = fmax(m, key[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == g) gmine = m;
  }
  // the topk_group best groups (ties to the lower group index)
  uint32_t gsel = 0;
  for (int r = 0; r < topk_group; ++r) {
    const bool cand = lane < n_group && !((gsel >> lane) & 1u);
    double bv = cand ? gmine : -INFINITY;
    int bg = cand ? lane : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const double ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int og = __shfl_xor_sync(0xffffffffu, bg, off);
      if (og != 0x7fffffff && (bg == 0x7fffffff || ov > bv || (ov == bv && og < bg))) {
        bv = ov;
        bg = og;
      }
    }
    gsel |= 1u << bg;
  }
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    if (e < E && ((gsel >> (e / gs)) & 1u)) avail |= 1u << i;
  }
  int my_id = 0;
  for (int k = 0; k < K; ++k) {
    double bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if ((avail >> i) & 1u) {
        if (be == 0x7fffffff || key[i] > bv) {
          bv = key[i];
          be = lane + 32 * i;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const double ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
    if (lane == k) my_id = be;
  }
  const double my_sc = (lane < K) ? s_sc[my_id] : 0.0;
  double sum = 0.0;
  for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, my_sc, k);  // fixed order
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_id;
    w[(size_t)t * K + lane] = (float)((renorm ? my_sc / sum : my_sc) * (double)scale);
  }
}

template <int PER>
void launch_grouped_per(const moe_problem& p, const float* logits, const float* bias, int n_group, int topk_group,
                        int renorm, float scale, int32_t* ids, float* w, cudaStream_t st) {
  route_grouped_kernel<PER><<<p.T, GROUPED_THREADS, 0, st>>>(logits, bias, p.T, p.E, p.K, n_group, topk_group,
                                                             renorm, scale, ids, w);
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

int launch_route_grouped(const moe_problem& p, const float* logits, const float* bias, int n_group, int topk_group,
                         int renorm, float scale, int32_t* ids, float* w, cudaStream_t st) {
  if (p.T == 0) return MOE_OK;
  const int per = (p.E + 31) / 32;
  if (per <= 1)
    launch_grouped_per<1>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  else if (per <= 2)
    launch_grouped_per<2>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  else if (per <= 4)
    launch_grouped_per<4>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  else if (per <= 8)
    launch_grouped_per<8>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  else if (per <= 16)
    launch_grouped_per<16>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  else
    launch_grouped_per<32>(p, logits, bias, n_group, topk_group, renorm, scale, ids, w, st);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

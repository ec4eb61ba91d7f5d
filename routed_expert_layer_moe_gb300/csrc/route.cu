// Step 1: softmax top-K routing, one warp per token.
//
// "MoE inference and expert parallelism" (blog.vllbc.top), routing section,
// Table 3-1: softmax scoring, top-K, renormalize=True.  Selection is made on
// the fp32 logits themselves (softmax is strictly increasing, so the chosen
// set is the same and no rounding of exp can create new ties); ties go to the
// lower expert index.  Weights: exp(l_k - l_max) / sum over the chosen K.
#include "route_select.cuh"

namespace moe {
namespace {

// (value, expert) a is ordered before b: larger value, or equal value and lower expert index.
__device__ __forceinline__ bool before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Sorts one (value, expert) pair per lane across the warp, lane 0 first in the order above
// (a bitonic network: 15 compare-exchange stages over lane pairs).
__device__ __forceinline__ void warp_sort(float& v, int& e, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oe = __shfl_xor_sync(0xffffffffu, e, j);
      const bool first = (((lane & k) == 0) == ((lane & j) == 0));  // this lane keeps the earlier one
      if (first ? before(ov, oe, v, e) : before(v, e, ov, oe)) {
        v = ov;
        e = oe;
      }
    }
  }
}

// PER: logits held per lane (E <= 32 * PER).  CAND (PER >= 4, large batches): the candidate
// filter below first; it takes fewer instructions per token but a longer chain of shuffles,
// so small batches, bound by that latency, go without it.
template <int PER, bool CAND>
__global__ void __launch_bounds__(256, CAND ? (PER >= 32 ? 2 : 4) : 1) route_topk_kernel(const float* __restrict__ logits, int T,
                                                                       int E, int K, int32_t* __restrict__ ids,
                                                                       float* __restrict__ w) {
  __shared__ float cand_v[CAND ? 8 : 1][32];  // per warp: the candidates, when at most 32
  __shared__ int cand_e[CAND ? 8 : 1][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int t = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  float v[PER];
  uint32_t avail = route_load<PER>(l, E, lane, v);  // bit i: expert lane + 32*i not yet chosen
  if constexpr (CAND) {
    static_assert(PER >= 4, "every lane must hold an expert");
    // Candidates first: tau, the K-th of the 32 lane maxima in the order above, has K
    // elements at or before it, so every one of the top K is at or before tau.  When at most
    // 32 elements are, they are sorted across the warp and the first K taken; otherwise the
    // selection below runs over them.  (E > 96: every lane holds at least one expert.)
    float mv = -INFINITY;
    int me = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (((avail >> i) & 1u) && (me == 0x7fffffff || v[i] > mv)) {
        mv = v[i];
        me = lane + 32 * i;
      }
    warp_sort(mv, me, lane);
    const float tv = __shfl_sync(0xffffffffu, mv, K - 1);
    const int te = __shfl_sync(0xffffffffu, me, K - 1);
    uint32_t cand = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (((avail >> i) & 1u) && !before(tv, te, v[i], e)) cand |= 1u << i;
    }
    const int c = __popc(cand);
    int pos = c;  // inclusive prefix over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, pos, o);
      if (lane >= o) pos += u;
    }
    const int total = __shfl_sync(0xffffffffu, pos, 31);
    avail = cand;
    if (total <= 32) {
      pos -= c;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        if ((cand >> i) & 1u) {
          cand_v[wib][pos] = v[i];
          cand_e[wib][pos] = lane + 32 * i;
          ++pos;
        }
      }
      __syncwarp();
      float sv = (lane < total) ? cand_v[wib][lane] : -INFINITY;
      int se = (lane < total) ? cand_e[wib][lane] : 0x7fffffff;
      warp_sort(sv, se, lane);
      const float lmax = __shfl_sync(0xffffffffu, sv, 0);
      const float ex = (lane < K) ? expf(sv - lmax) : 0.0f;
      float sum = 0.0f;
      for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);  // fixed order k = 0..K-1
      if (lane < K) {
        ids[(size_t)t * K + lane] = se;
        w[(size_t)t * K + lane] = ex / sum;
      }
      return;
    }
  }
  int my_id;
  float my_val;
  route_select<PER>(v, avail, K, lane, my_id, my_val);
  const float wt = route_weight(my_val, K, lane);
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_id;
    w[(size_t)t * K + lane] = wt;
  }
}

template <int PER>
void launch_route_per(const moe_problem& p, const float* logits, int32_t* ids, float* w, cudaStream_t st) {
  const int threads = 256;
  const int blocks = (int)(((int64_t)p.T * 32 + threads - 1) / threads);
  if constexpr (PER >= 4) {
    if (p.T >= 2048 && p.E > 96) {
      route_topk_kernel<PER, true><<<blocks, threads, 0, st>>>(logits, p.T, p.E, p.K, ids, w);
      return;
    }
  }
  route_topk_kernel<PER, false><<<blocks, threads, 0, st>>>(logits, p.T, p.E, p.K, ids, w);
}

// "MoE inference and expert parallelism", routing section, Table 3-1 (DeepSeek-V3):
// sigmoid scores, e_score_correction_bias used for the choice only, grouped
// top-k (the best topk_group of n_group contiguous expert groups, a group
// scored by its best biased score, then the K best experts inside them; ties to
// the lower index); weights are the unbiased scores of the chosen experts,
// renormalised if asked, times `scale`.
//
// The choice is defined on fp64 keys sigmoid(l) + bias.  GB300's fp64 rate is
// low, so each token (one warp) first chooses on fp32 keys, whose error against
// the fp64 keys is below 2^-20 (1 + |key|) (a few ulps of the fp32 sigmoid plus
// the rounding of the sum).  Every decision the choice makes -- the last kept
// group against the best dropped one, each chosen expert against the next in
// the list, and the last chosen against the best one left -- compares two keys;
// when all those gaps exceed 2^-16 (1 + |key|) the fp64 keys order the same way
// and the fp32 choice is the fp64 choice.  Otherwise (near-ties, exact ties) the
// token is chosen again on fp64 keys.  The weights are the fp32 sigmoids of the
// chosen experts (expf and an IEEE division: a few ulps), summed in k order.
template <typename KT>
__device__ __forceinline__ KT key_lowest() {
  if constexpr (sizeof(KT) == 8) return (KT)0;  // order images of fp64 keys (below every real key)
  else return -INFINITY;
}

// fp64 key of one expert, kept out of line: the fallback is rare and its code stays small.
__device__ __noinline__ double key_fp64(const float* l, const float* bias, int e) {
  return 1.0 / (1.0 + exp(-(double)__ldg(l + e))) + (bias ? (double)__ldg(bias + e) : 0.0);
}

// Order-preserving image of an fp64 key as an unsigned integer (larger key, larger image).
__device__ __forceinline__ uint64_t order_image(double k) {
  const uint64_t u = (uint64_t)__double_as_longlong(k);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// The grouped choice on one warp's keys (float keys, or order images of fp64 keys).
// With float keys it also reports whether every decision had a decisive gap
// (`clear`) and the lowest key a decision touched (`cut`).
template <int PER, typename KT>
__device__ __forceinline__ void grouped_choice(const KT (&key)[PER], int lane, int E, int gs, int n_group,
                                               int topk_group, int K, int& my_id, bool& clear, KT& cut) {
  constexpr bool F = sizeof(KT) == 4;
  const KT NEG = key_lowest<KT>();
  auto kmax = [](KT a, KT b) { return a > b ? a : b; };
  auto gap_ok = [](KT a, KT b) {  // a is ordered before b: is the gap decisive?
    if constexpr (F) return a - b > 0x1p-16f * (1.0f + fabsf(a));  // a - b is exact when the two are close
    else return true;
  };
  // group maxima: lane g keeps the score of group g
  KT gmine = NEG;
  for (int g = 0; g < n_group; ++g) {
    KT m = NEG;
    const int e_lo = g * gs, e_hi = e_lo + gs;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e >= e_lo && e < e_hi) m = kmax(m, key[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = kmax(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == g) gmine = m;
  }
  clear = true;
  // the topk_group best groups (ties to the lower group index), then the best group left
  uint32_t gsel = 0;
  KT last = NEG;
  for (int r = 0; r <= topk_group && r < n_group; ++r) {
    const bool cand = lane < n_group && !((gsel >> lane) & 1u);
    KT bv = cand ? gmine : NEG;
    int bg = cand ? lane : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const KT ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int og = __shfl_xor_sync(0xffffffffu, bg, off);
      if (og != 0x7fffffff && (bg == 0x7fffffff || ov > bv || (ov == bv && og < bg))) {
        bv = ov;
        bg = og;
      }
    }
    if (r == topk_group) {  // the best dropped group
      clear = clear && gap_ok(last, bv);
    } else {
      gsel |= 1u << bg;
      last = bv;
    }
  }
  cut = last;
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    if (e < E && ((gsel >> (e / gs)) & 1u)) avail |= 1u << i;
  }
  // the K best experts of the kept groups in order, then the best one left
  const int ncand = topk_group * gs;
  my_id = 0;
  last = NEG;
  for (int k = 0; k <= K && k < ncand; ++k) {
    KT bv = NEG;
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
      const KT ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if (k > 0) clear = clear && gap_ok(last, bv);
    if (be != 0x7fffffff && bv < cut) cut = bv;
    if (k == K) break;
    last = bv;
    if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
    if (lane == k) my_id = be;
  }
}

template <int PER>
__global__ void __launch_bounds__(256) route_grouped_kernel(const float* __restrict__ logits,
                                                            const float* __restrict__ bias, int T, int E, int K,
                                                            int n_group, int topk_group, int renorm, float scale,
                                                            int32_t* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  const int gs = E / n_group;
  int my_id = 0;
  bool clear = false;
  float key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = -INFINITY;
    if (e < E) key[i] = __fdividef(1.0f, 1.0f + __expf(-__ldg(l + e))) + (bias ? __ldg(bias + e) : 0.0f);
  }
  float cut;
  grouped_choice<PER, float>(key, lane, E, gs, n_group, topk_group, K, my_id, clear, cut);
  if (!clear) {
    // A near-tie: choose on the fp64 keys.  Only keys at or above the lowest key a decision
    // touched (less the fp32 error) can change a decision, so only those are evaluated in
    // fp64; the choice then runs on their order images (integer compares, no fp64 pipe).
    const float lim = cut - 0x1p-18f * (1.0f + fabsf(cut));
    uint64_t k64[PER];
#pragma unroll 1
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      k64[i] = (e < E && key[i] >= lim) ? order_image(key_fp64(l, bias, e)) : 0;
    }
    uint64_t cut64;
    grouped_choice<PER, uint64_t>(k64, lane, E, gs, n_group, topk_group, K, my_id, clear, cut64);
  }
  const float my_sc = (lane < K) ? 1.0f / (1.0f + expf(-__ldg(l + my_id))) : 0.0f;
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, my_sc, k);  // fixed order
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_id;
    w[(size_t)t * K + lane] = (renorm ? my_sc / sum : my_sc) * scale;
  }
}

template <int PER>
void launch_grouped_per(const moe_problem& p, const float* logits, const float* bias, int n_group, int topk_group,
                        int renorm, float scale, int32_t* ids, float* w, cudaStream_t st) {
  const int threads = 256;
  const int blocks = (int)(((int64_t)p.T * 32 + threads - 1) / threads);
  route_grouped_kernel<PER><<<blocks, threads, 0, st>>>(logits, bias, p.T, p.E, p.K, n_group, topk_group, renorm,
                                                        scale, ids, w);
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

// Step 2: counts, offsets, row maps and the dispatch of activations into the
// expert-grouped buffer.
//
// "Inference INFRA methodology (5)", section "DeepGEMM": a static
// [slots, M_max, H] buffer plus a device-resident masked_m (decode), or a
// contiguous expert-grouped layout with per-expert offsets (prefill).
// "vLLM EPLB", section 1.2: physical_to_logical_map and its inverse.
// "MoonEP", "Why dynamic routing is hard": counts sum to the routed records;
// "Zero-copy and static buffer": rows past a slot's count are padding.
//
// Deterministic, without atomics on order: each (slot, token) pair is one bit
// of a [P][ceil(T/32)] mask (a token names an expert at most once, and a
// logical expert maps to one replica per token).  A row's rank inside its
// slot is the popcount of the bits of lower tokens, so rows of a slot are in
// ascending token order.
//
//   [eplb_tables]  map -> logical_to_physical / replica counts (maps only)
//   mark           ids -> slot of each record, mask bits
//   scan           mask -> per-word rank prefix, masked_m, offsets
//   scatter        one CTA per token: row_of, src_of, x -> xg (e4m3: 1x128 quantisation)
//
// Decode batches take shorter paths with the same results (a rank is the number of lower
// tokens in the slot): up to 256 records without a replica map, one launch in which each
// token's CTA derives the counts and its own ranks from all T*K ids in shared memory; up to
// 4096 records, the whole layout in one CTA (replica tables included), then the copy.
#include <algorithm>

#include "common.cuh"
#include "route_select.cuh"

namespace moe {
namespace {

struct PermuteWs {
  uint32_t* bits;   // [P][W], then one int32 counter (cleared with the bits)
  int32_t* prefix;  // [P][W] rank of the first token of each 32-token word
  int32_t* slot_of; // [T*K]
  int32_t* list;    // [P] logical_to_physical_map, compact: the slots of expert 0, then of 1, ...
  int32_t* start;   // [E] first entry of each expert in list
  int32_t* rc;      // [E] logical_replica_count
};

inline int words_of(int T) { return (T + 31) / 32; }
inline int max_replicas(const moe_problem& p) { return p.P - p.E + 1; }

PermuteWs carve(const moe_problem& p, void* ws, size_t* total) {
  const size_t W = words_of(p.T);
  size_t off = 0;
  PermuteWs w{};
  char* base = static_cast<char*>(ws);
  auto take = [&](size_t bytes) {
    char* ptr = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return ptr;
  };
  w.bits = (uint32_t*)take((size_t)p.P * W * 4 + 4);
  w.prefix = (int32_t*)take((size_t)p.P * W * 4);
  w.slot_of = (int32_t*)take((size_t)p.T * p.K * 4);
  w.list = (int32_t*)take((size_t)p.P * 4);
  w.start = (int32_t*)take((size_t)p.E * 4);
  w.rc = (int32_t*)take((size_t)p.E * 4);
  if (total) *total = off;
  return w;
}

// logical_to_physical_map in compact form: list holds the slots of expert 0 (ascending),
// then those of expert 1, ...; start[e] is where expert e's slots begin and rc[e]
// (logical_replica_count) how many there are.  One CTA, a thread per slot and per expert:
// a slot's place among its expert's slots is the number of lower slots holding the same
// expert (the map is staged in shared memory; P, E <= 1024).
__global__ void __launch_bounds__(1024) eplb_tables_kernel(const int32_t* __restrict__ p2l, int P, int E, int R,
                                                           int32_t* __restrict__ list, int32_t* __restrict__ start,
                                                           int32_t* __restrict__ rc, int32_t* err) {
  __shared__ __align__(16) int32_t map[1024];
  __shared__ int32_t cnt[1024];
  __shared__ int32_t first[1024];
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = threadIdx.x; s < 1024; s += blockDim.x) map[s] = (s < P) ? p2l[s] : -1;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < P; s += blockDim.x) {
    const int e = map[s];
    if (e < 0 || e >= E) {
      atomicOr(err, MOE_FLAG_BAD_MAP);
      map[s] = -1;  // this thread's own entry: later counts skip it
    } else {
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  // first[e] = exclusive prefix sum of cnt (one expert per thread, E <= 1024 = blockDim.x)
  {
    const int e = threadIdx.x;
    const int c = (e < E) ? cnt[e] : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (e < E) {
      first[e] = before + inc - c;
      start[e] = before + inc - c;
      rc[e] = c;
      if (c > R) atomicOr(err, MOE_FLAG_BAD_MAP);  // only possible when another expert has no slot
    }
  }
  __syncthreads();
  for (int s = threadIdx.x; s < P; s += blockDim.x) {
    const int e = map[s];
    if (e < 0) continue;
    int r = 0;
    const int4* m4 = reinterpret_cast<const int4*>(map);
    for (int q = 0; q < (s >> 2); ++q) {
      const int4 v = m4[q];
      r += (v.x == e) + (v.y == e) + (v.z == e) + (v.w == e);
    }
    for (int q = s & ~3; q < s; ++q) r += (map[q] == e);
    list[first[e] + r] = s;
  }
}

// Slot of record i = (t, k) of logical expert ids[i]: -1 (and a flag bit) for an id outside
// [0, E), for a token naming the same expert again (the record with the larger k is the one
// not placed), or for an expert whose replica count is 0 or above R; else the (t mod c)-th
// slot holding the expert, c its replica count.  `tok_ids` are the K ids of token t.
__device__ __forceinline__ int slot_of_record(const int32_t* tok_ids, int t, int k, int E, int use_map,
                                              const int32_t* list, const int32_t* start, const int32_t* rc, int R,
                                              int& flags) {
  const int e = tok_ids[k];
  if (e < 0 || e >= E) {
    flags |= MOE_FLAG_BAD_EXPERT;
    return -1;
  }
  for (int j = 0; j < k; ++j) {
    if (tok_ids[j] == e) {
      flags |= MOE_FLAG_BAD_EXPERT;
      return -1;
    }
  }
  if (!use_map) return e;
  const int c = rc[e];
  if (c <= 0 || c > R) {
    flags |= MOE_FLAG_BAD_MAP;
    return -1;
  }
  return list[start[e] + (t % c)];
}

__global__ void mark_kernel(const int32_t* __restrict__ ids, int T, int K, int E, int use_map,
                            const int32_t* __restrict__ list, const int32_t* __restrict__ start,
                            const int32_t* __restrict__ rc, int R, uint32_t* bits,
                            int W, int32_t* __restrict__ slot_of, int32_t* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * K) return;
  const int t = i / K;
  int flags = 0;
  const int s = slot_of_record(ids + (size_t)t * K, t, i - t * K, E, use_map, list, start, rc, R, flags);
  if (flags) atomicOr(err, flags);
  if (s >= 0) atomicOr(bits + (size_t)s * W + (t >> 5), 1u << (t & 31));
  slot_of[i] = s;
}

// One CTA of 1024 threads: per-slot word prefixes (a warp per slot), then an
// exclusive scan of the counts into offsets.
__global__ void __launch_bounds__(1024) scan_kernel(const uint32_t* __restrict__ bits, int W, int P, int S, int T,
                                                    int masked, int M_max, int32_t* __restrict__ prefix,
                                                    int32_t* __restrict__ masked_m, int32_t* __restrict__ offsets,
                                                    int32_t* err) {
  __shared__ int32_t counts[2048];
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int NS = P + S;
  for (int s = warp; s < P; s += nwarps) {
    int base = 0;
    for (int w0 = 0; w0 < W; w0 += 32) {
      const int w = w0 + lane;
      const int c = (w < W) ? __popc(bits[(size_t)s * W + w]) : 0;
      int inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += n;
      }
      if (w < W) prefix[(size_t)s * W + w] = base + inc - c;
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) counts[s] = base;
  }
  if (S && threadIdx.x == 0) counts[P] = T;
  __syncthreads();
  for (int s = threadIdx.x; s < NS; s += blockDim.x) {
    masked_m[s] = counts[s];
    if (masked && counts[s] > M_max) atomicOr(err, MOE_FLAG_OVERFLOW);
  }
  // exclusive scan of counts[0..NS) -> offsets[0..NS]; NS <= 2048, two per thread
  const int i0 = 2 * threadIdx.x;
  const int a = (i0 < NS) ? counts[i0] : 0;
  const int b = (i0 + 1 < NS) ? counts[i0 + 1] : 0;
  int inc = a + b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int v = (lane < nwarps) ? warp_tot[lane] : 0;
    int vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += n;
    }
    warp_tot[lane] = vi - v;
  }
  __syncthreads();
  const int excl = warp_tot[warp] + inc - (a + b);
  if (i0 < NS) offsets[i0] = excl;
  if (i0 + 1 < NS) offsets[i0 + 1] = excl + a;
  if (threadIdx.x == blockDim.x - 1) offsets[NS] = excl + a + b;  // the total
}

// The same outputs for large bitmasks, spread over the GPU: a warp per slot (8 slots per
// CTA) writes the slot's word prefixes and its count; the last CTA to finish (a counter in
// the workspace, cleared with the bits) turns the counts into offsets.
__global__ void __launch_bounds__(256) slot_scan_kernel(const uint32_t* __restrict__ bits, int W, int P, int S, int T,
                                                        int masked, int M_max, int32_t* __restrict__ prefix,
                                                        int32_t* masked_m, int32_t* __restrict__ offsets,
                                                        int32_t* err, int* done) {
  __shared__ int32_t warp_tot[8];
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int s = blockIdx.x * 8 + warp;
  if (s < P) {
    int base = 0;
    for (int w0 = 0; w0 < W; w0 += 32) {
      const int w = w0 + lane;
      const int c = (w < W) ? __popc(bits[(size_t)s * W + w]) : 0;
      int inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += n;
      }
      if (w < W) prefix[(size_t)s * W + w] = base + inc - c;
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      masked_m[s] = base;
      if (masked && base > M_max) atomicOr(err, MOE_FLAG_OVERFLOW);
    }
  }
  __threadfence();  // this CTA's counts are visible before it is counted as done
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(done, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  // exclusive scan of the counts (the shared slot holds T) into offsets, 256 threads in order
  const int NS = P + S;
  const int per = (NS + 255) / 256;
  const int lo = threadIdx.x * per, hi = min(lo + per, NS);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += (i < P) ? __ldcg(masked_m + i) : T;
  int inc = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  int run = before + inc - sum;
  for (int i = lo; i < hi; ++i) {
    offsets[i] = run;
    run += (i < P) ? __ldcg(masked_m + i) : T;
  }
  if (threadIdx.x == 255) offsets[NS] = before + inc;
  if (S && threadIdx.x == 0) {
    masked_m[P] = T;
    if (masked && T > M_max) atomicOr(err, MOE_FLAG_OVERFLOW);
  }
}

// Part of x[t] to its rows of the grouped buffer (`rows`: the token's K+S rows, -1 = not
// placed): the 16-byte vectors [v_lo, v_hi) of the token's row; e4m3: quantised per 1x128
// group on the way (16 vectors per group; v_lo and v_hi are multiples of 16).  Each thread
// requests up to four vectors (two when quantising) before it stores any.  All threads of the
// CTA take part.
template <typename TX, bool QUANT>
__device__ __forceinline__ void copy_token(const TX* __restrict__ x, int t, int H, int KS, const int* rows,
                                           void* __restrict__ xg, float* __restrict__ xg_scales, int v_lo,
                                           int v_hi) {
  constexpr int B = QUANT ? 2 : 4;
  const TX* xr = x + (size_t)t * H;
  if constexpr (QUANT) {
    // 16 threads per 128-element group, 8 bf16 elements (16 bytes) each.
    const int G = H / 128;
    const int g_lo = v_lo / 16, g_hi = v_hi / 16;
    const int per = (int)(blockDim.x >> 4);  // groups per pass
    const int sub = threadIdx.x & 15;
    uint8_t* q = static_cast<uint8_t*>(xg);
    for (int g0 = g_lo; g0 < g_hi; g0 += B * per) {  // same trip count for every thread
      uint4 raw[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int g = g0 + j * per + (int)(threadIdx.x >> 4);
        if (g < g_hi) raw[j] = __ldg(reinterpret_cast<const uint4*>(xr + g * 128 + sub * 8));
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int g = g0 + j * per + (int)(threadIdx.x >> 4);
        const bool live = g < g_hi;
        float f[8];
        float amax = 0.0f;
        if (live) {
          const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 v = __bfloat1622float2(hv[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (!live) continue;
        const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        uint32_t packed[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(f[4 * i], sc), __fdiv_rn(f[4 * i + 1], sc)), __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(f[4 * i + 2], sc), __fdiv_rn(f[4 * i + 3], sc)), __NV_SATFINITE, __NV_E4M3);
          packed[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        const uint2 pv = make_uint2(packed[0], packed[1]);
        for (int k = 0; k < KS; ++k) {
          const int r = rows[k];
          if (r < 0) continue;
          *reinterpret_cast<uint2*>(q + (size_t)r * H + g * 128 + sub * 8) = pv;
          if (sub == 0) xg_scales[(size_t)r * G + g] = sc;
        }
      }
    }
  } else {
    // plain copy in 16-byte vectors
    constexpr int V = 16 / sizeof(TX);
    TX* dst = static_cast<TX*>(xg);
    for (int c0 = v_lo + (int)threadIdx.x; c0 < v_hi; c0 += B * (int)blockDim.x) {
      uint4 raw[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int c = c0 + j * (int)blockDim.x;
        if (c < v_hi) raw[j] = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)c * V));
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int c = c0 + j * (int)blockDim.x;
        if (c >= v_hi) break;
        for (int k = 0; k < KS; ++k) {
          const int r = rows[k];
          if (r < 0) continue;
          *reinterpret_cast<uint4*>(dst + (size_t)r * H + (size_t)c * V) = raw[j];
        }
      }
    }
  }
}

// The part of a token's row that CTA blockIdx.y of gridDim.y copies, in 16-byte vectors
// (whole 128-element groups: a multiple of 16 vectors).
__device__ __forceinline__ void copy_range(int H, int esz, int& v_lo, int& v_hi) {
  const int nv = H * esz / 16;
  const int chunk = ((nv + (int)gridDim.y - 1) / (int)gridDim.y + 15) & ~15;
  v_lo = min(nv, (int)blockIdx.y * chunk);
  v_hi = min(nv, v_lo + chunk);
}

// One CTA per token.
template <typename TX, bool QUANT>
__global__ void __launch_bounds__(256) scatter_kernel(const TX* __restrict__ x, int H, int T, int K, int P, int S,
                                                      int masked, int M_max, const uint32_t* __restrict__ bits,
                                                      const int32_t* __restrict__ prefix, int W,
                                                      const int32_t* __restrict__ slot_of,
                                                      const int32_t* __restrict__ offsets, int32_t* __restrict__ row_of,
                                                      int32_t* __restrict__ src_of, void* __restrict__ xg,
                                                      float* __restrict__ xg_scales) {
  const int t = blockIdx.x;
  const int KS = K + S;
  __shared__ int rows[64];
  if (threadIdx.x < KS) {  // every CTA of the token derives its rows; the first writes the maps
    const int k = threadIdx.x;
    int row = -1;
    if (k < K) {
      const int s = slot_of[(size_t)t * K + k];
      if (s >= 0) {
        const int wd = t >> 5;
        const int rank = prefix[(size_t)s * W + wd] + __popc(bits[(size_t)s * W + wd] & ((1u << (t & 31)) - 1u));
        if (masked)
          row = (rank < M_max) ? s * M_max + rank : -1;
        else
          row = offsets[s] + rank;
      }
    } else {
      row = masked ? P * M_max + t : offsets[P] + t;
    }
    rows[k] = row;
    if (blockIdx.y == 0) {
      row_of[(size_t)t * KS + k] = row;
      if (row >= 0) src_of[row] = t;
    }
  }
  __syncthreads();
  int v_lo, v_hi;
  copy_range(H, (int)sizeof(TX), v_lo, v_hi);
  copy_token<TX, QUANT>(x, t, H, KS, rows, xg, xg_scales, v_lo, v_hi);
}

// Decode batches of at most 256 records without a replica map, in one launch: every CTA
// stages all T*K ids in shared memory and derives the whole layout itself -- the slot of
// every record, the rows per slot, their exclusive prefix sum, and for its own token the rows
// from lower tokens in each of its slots -- then copies its part of the token.  The results
// are those of mark + scan + scatter (rows of a slot in ascending token order); CTA (0, 0)
// writes masked_m, offsets and the flags.
// RPER > 0 (route + dispatch in one launch, E <= 32 * RPER): the ids are not read but chosen
// in the CTA from the logits, one warp per token, by the router's own per-token code (the
// same ids and weights as the router kernel); the CTAs of column split 0 write their token's
// ids and weights.
constexpr int kOneLaunchRecords = 256;  // T*K
constexpr int kSlotsMax = 1024;         // P+S
constexpr int kSmallThreads = 256;

template <typename TX, bool QUANT, int RPER = 0>
__global__ void __launch_bounds__(kSmallThreads) permute_small_kernel(
    const int32_t* __restrict__ ids, const TX* __restrict__ x, int H, int T, int K, int E, int P, int S, int masked,
    int M_max, int32_t* __restrict__ masked_m, int32_t* __restrict__ offsets, int32_t* __restrict__ row_of,
    int32_t* __restrict__ src_of, void* __restrict__ xg, float* __restrict__ xg_scales, int32_t* err,
    const float* __restrict__ logits = nullptr, int32_t* __restrict__ ids_out = nullptr,
    float* __restrict__ w_out = nullptr) {
  __shared__ int32_t rec[kOneLaunchRecords];  // the ids
  __shared__ int32_t cnt[kSlotsMax];          // rows per slot
  __shared__ int32_t below[kSlotsMax];        // rows per slot from tokens before this CTA's token
  __shared__ int32_t off[kSlotsMax + 1];      // exclusive prefix sum of cnt
  __shared__ int32_t warp_tot[kSmallThreads / 32];
  __shared__ int rows[64];
  const int t = blockIdx.x;
  const int n = T * K, NS = P + S, KS = K + S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = threadIdx.x; s < NS; s += kSmallThreads) {
    cnt[s] = (s == P) ? T : 0;  // slot P (when present) is the shared expert: one row per token
    below[s] = (s == P) ? t : 0;
  }
  if constexpr (RPER > 0) {
    // the next token's logits are requested before this token's selection
    float v[RPER], vn[RPER];
    uint32_t avail = 0, availn = 0;
    if (warp < T) avail = route_load<RPER>(logits + (size_t)warp * E, E, lane, v);
    for (int tt = warp; tt < T; tt += kSmallThreads / 32) {
      const int tn = tt + kSmallThreads / 32;
      if (tn < T) availn = route_load<RPER>(logits + (size_t)tn * E, E, lane, vn);
      int id;
      float val;
      route_select<RPER>(v, avail, K, lane, id, val);
      const float wt = route_weight(val, K, lane);
      if (lane < K) {
        rec[tt * K + lane] = id;
        if (tt == t && blockIdx.y == 0) {
          ids_out[(size_t)tt * K + lane] = id;
          w_out[(size_t)tt * K + lane] = wt;
        }
      }
#pragma unroll
      for (int i = 0; i < RPER; ++i) v[i] = vn[i];
      avail = availn;
    }
  } else {
    if ((int)threadIdx.x < n) rec[threadIdx.x] = ids[threadIdx.x];
  }
  __syncthreads();
  int flags = 0;
  int sl = -1;
  if ((int)threadIdx.x < n) {
    const int i = threadIdx.x, ti = i / K;
    sl = slot_of_record(rec + (size_t)ti * K, ti, i - ti * K, E, 0, nullptr, nullptr, nullptr, 1, flags);
    if (sl >= 0) {
      atomicAdd(&cnt[sl], 1);  // integer counts: the order of the adds does not matter
      if (ti < t) atomicAdd(&below[sl], 1);
    }
  }
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;
  if (lead && flags) atomicOr(err, flags);
  __syncthreads();  // every id is read: rec now takes the slots
  if ((int)threadIdx.x < n) rec[threadIdx.x] = sl;
  // exclusive prefix sum of cnt[0..NS): four consecutive slots per thread
  {
    const int i0 = threadIdx.x * 4;
    int a[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a[j] = (i0 + j < NS) ? cnt[i0 + j] : 0;
      sum += a[j];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    int run = before + inc - sum;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i0 + j < NS) off[i0 + j] = run;
      run += a[j];
    }
    if (threadIdx.x == kSmallThreads - 1) off[NS] = before + inc;
  }
  __syncthreads();
  if (lead) {
    for (int s = threadIdx.x; s <= NS; s += kSmallThreads) {
      offsets[s] = off[s];
      if (s < NS) {
        masked_m[s] = cnt[s];
        if (masked && cnt[s] > M_max) atomicOr(err, MOE_FLAG_OVERFLOW);
      }
    }
  }
  if (threadIdx.x < KS) {
    const int k = threadIdx.x;
    int row = -1;
    if (k < K) {
      const int s = rec[(size_t)t * K + k];
      if (s >= 0) {
        const int rank = below[s];
        if (masked)
          row = (rank < M_max) ? s * M_max + rank : -1;
        else
          row = off[s] + rank;
      }
    } else {
      row = masked ? P * M_max + t : off[P] + t;
    }
    rows[k] = row;
    if (blockIdx.y == 0) {
      row_of[(size_t)t * KS + k] = row;
      if (row >= 0) src_of[row] = t;
    }
  }
  __syncthreads();
  int v_lo, v_hi;
  copy_range(H, (int)sizeof(TX), v_lo, v_hi);
  copy_token<TX, QUANT>(x, t, H, KS, rows, xg, xg_scales, v_lo, v_hi);
}

// Decode batches of at most 4096 records (any map) whose slot bitmask fits in shared memory:
// the whole layout in one CTA of 1024 threads, then a copy kernel.  The replica tables are
// built in shared memory as eplb_tables_kernel builds them; the ranks come from the bitmask
// as in mark + scan (a record's rank is the popcount of its slot's bits of lower tokens).
// Writes masked_m, offsets, row_of, src_of and the flags.
constexpr int kLayoutRecords = 4096;
constexpr int kLayoutWords = 4096;  // P * ceil(T/32)
constexpr int kLayoutThreads = 1024;

__global__ void __launch_bounds__(kLayoutThreads) layout_small_kernel(
    const int32_t* __restrict__ ids, int T, int K, int E, int P, int S, int masked, int M_max,
    const int32_t* __restrict__ p2l, int R, int32_t* __restrict__ masked_m, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_of, int32_t* __restrict__ src_of, int32_t* err) {
  __shared__ int16_t rec[kLayoutRecords];   // ids, then slots (-1: not placed); ids and slots are < 1024
  __shared__ uint32_t bits[kLayoutWords];   // [P][W]: bit t of slot s
  __shared__ int32_t cnt[kSlotsMax];        // replica counts while the tables are built, then rows per slot
  __shared__ __align__(16) int32_t off[kSlotsMax + 1];  // the staged map while the tables are built
  __shared__ int32_t m_list[kSlotsMax], m_start[kSlotsMax];
  __shared__ int32_t warp_tot[32];
  const int n = T * K, NS = P + S, KS = K + S, W = (T + 31) >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool use_map = p2l != nullptr;
  int flags = 0;
  // block-wide exclusive prefix sum of one value per thread (1024 threads); total of all
  auto scan = [&](int v, int& total) {
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int before = 0;
    total = 0;
    for (int w = 0; w < 32; ++w) {
      before += (w < warp) ? warp_tot[w] : 0;
      total += warp_tot[w];
    }
    __syncthreads();  // warp_tot may be reused
    return before + inc - v;
  };
  for (int i = tid; i < n; i += kLayoutThreads) {
    const int e = ids[i];
    rec[i] = (e < 0 || e >= E) ? (int16_t)-1 : (int16_t)e;  // out of range: flagged below
  }
  for (int i = tid; i < P * W; i += kLayoutThreads) bits[i] = 0u;
  int32_t* map = off;  // the map is staged where the offsets go later
  if (use_map) {
    map[tid] = (tid < P) ? p2l[tid] : -1;
    cnt[tid] = 0;
  }
  __syncthreads();
  if (use_map) {  // logical_to_physical_map, compact (as eplb_tables_kernel)
    const int e = map[tid];
    if (tid < P && (e < 0 || e >= E)) {
      flags |= MOE_FLAG_BAD_MAP;
      map[tid] = -1;  // this thread's own entry
    } else if (tid < P) {
      atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    int total;
    const int c = (tid < E) ? cnt[tid] : 0;
    const int first = scan(c, total);
    if (tid < E) {
      m_start[tid] = first;
      if (c > R) flags |= MOE_FLAG_BAD_MAP;  // only possible when another expert has no slot
    }
    __syncthreads();
    const int me = map[tid];
    if (me >= 0) {
      int r = 0;
      const int4* m4 = reinterpret_cast<const int4*>(map);
      for (int q = 0; q < (tid >> 2); ++q) {
        const int4 v = m4[q];
        r += (v.x == me) + (v.y == me) + (v.z == me) + (v.w == me);
      }
      for (int q = tid & ~3; q < tid; ++q) r += (map[q] == me);
      m_list[m_start[me] + r] = tid;
    }
    __syncthreads();
  }
  // slot of every record (at most four per thread); mark its bit
  int sl[kLayoutRecords / kLayoutThreads];
#pragma unroll
  for (int j = 0; j < kLayoutRecords / kLayoutThreads; ++j) {
    const int i = tid + j * kLayoutThreads;
    sl[j] = -1;
    if (i < n) {
      const int ti = i / K, k = i - ti * K;
      const int16_t* tok = rec + (size_t)ti * K;
      const int e = tok[k];
      if (e < 0) {
        flags |= MOE_FLAG_BAD_EXPERT;
      } else {
        bool dup = false;
        for (int q = 0; q < k; ++q) dup |= (tok[q] == e);
        if (dup) {
          flags |= MOE_FLAG_BAD_EXPERT;
        } else if (!use_map) {
          sl[j] = e;
        } else {
          const int c = cnt[e];
          if (c <= 0 || c > R)
            flags |= MOE_FLAG_BAD_MAP;
          else
            sl[j] = m_list[m_start[e] + ti % c];
        }
      }
    }
  }
  __syncthreads();  // every id and replica count is read
#pragma unroll
  for (int j = 0; j < kLayoutRecords / kLayoutThreads; ++j) {
    const int i = tid + j * kLayoutThreads;
    if (i < n) {
      rec[i] = (int16_t)sl[j];
      if (sl[j] >= 0) {
        const int ti = i / K;
        atomicOr(&bits[sl[j] * W + (ti >> 5)], 1u << (ti & 31));
      }
    }
  }
  __syncthreads();
  // rows per slot, their prefix sum
  int c = 0;
  if (tid < P)
    for (int w = 0; w < W; ++w) c += __popc(bits[tid * W + w]);
  else if (tid == P && S)
    c = T;
  cnt[tid] = c;
  int total;
  const int o = scan(tid < NS ? c : 0, total);
  if (tid < NS) off[tid] = o;
  if (tid == 0) off[NS] = total;
  __syncthreads();
  if (flags) atomicOr(err, flags);
  if (tid < NS) {
    offsets[tid] = off[tid];
    masked_m[tid] = cnt[tid];
    if (masked && cnt[tid] > M_max) atomicOr(err, MOE_FLAG_OVERFLOW);
  }
  if (tid == 0) offsets[NS] = off[NS];
  for (int i = tid; i < n; i += kLayoutThreads) {
    const int s = rec[i];
    const int t = i / K, k = i - t * K;
    int row = -1;
    if (s >= 0) {
      const uint32_t* b = bits + s * W;
      int rank = __popc(b[t >> 5] & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < (t >> 5); ++w) rank += __popc(b[w]);
      if (masked)
        row = (rank < M_max) ? s * M_max + rank : -1;
      else
        row = off[s] + rank;
    }
    row_of[(size_t)t * KS + k] = row;
    if (row >= 0) src_of[row] = t;
  }
  if (S) {
    for (int t = tid; t < T; t += kLayoutThreads) {
      const int row = masked ? P * M_max + t : off[P] + t;
      row_of[(size_t)t * KS + K] = row;
      src_of[row] = t;
    }
  }
}

// The copy of each token to its rows (row_of written by layout_small_kernel).
template <typename TX, bool QUANT>
__global__ void __launch_bounds__(256) copy_rows_kernel(const TX* __restrict__ x, int H, int KS,
                                                        const int32_t* __restrict__ row_of, void* __restrict__ xg,
                                                        float* __restrict__ xg_scales) {
  __shared__ int rows[64];
  const int t = blockIdx.x;
  if ((int)threadIdx.x < KS) rows[threadIdx.x] = row_of[(size_t)t * KS + threadIdx.x];
  __syncthreads();
  int v_lo, v_hi;
  copy_range(H, (int)sizeof(TX), v_lo, v_hi);
  copy_token<TX, QUANT>(x, t, H, KS, rows, xg, xg_scales, v_lo, v_hi);
}

// CTAs per token for the copy: about two CTAs per SM in all, at least 128 vectors (2 KB of
// the source row) each.
int copy_splits(const moe_problem& p, int esz) {
  const int nv = p.H * esz / 16;
  const int want = (2 * device_info().sm_count + p.T - 1) / p.T;
  return std::max(1, std::min(want, nv / 128));
}

template <typename TX, bool QUANT>
void launch_small(const moe_problem& p, const int32_t* ids, const void* x, const int32_t* p2l, int32_t* masked_m,
                  int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg, float* xg_scales, int32_t* err,
                  cudaStream_t st) {
  const int masked = p.layout == MOE_LAYOUT_MASKED;
  const dim3 grid(p.T, copy_splits(p, (int)sizeof(TX)));
  if ((int64_t)p.T * p.K <= kOneLaunchRecords && !p2l) {  // else P * ceil(T/32) <= kLayoutWords
    permute_small_kernel<TX, QUANT><<<grid, kSmallThreads, 0, st>>>(
        ids, static_cast<const TX*>(x), p.H, p.T, p.K, p.E, p.P, p.has_shared, masked, p.M_max, masked_m, offsets,
        row_of, src_of, xg, xg_scales, err);
  } else {
    layout_small_kernel<<<1, kLayoutThreads, 0, st>>>(ids, p.T, p.K, p.E, p.P, p.has_shared, masked, p.M_max, p2l,
                                                      max_replicas(p), masked_m, offsets, row_of, src_of, err);
    copy_rows_kernel<TX, QUANT><<<grid, 256, 0, st>>>(static_cast<const TX*>(x), p.H, p.K + p.has_shared, row_of,
                                                      xg, xg_scales);
  }
}

template <typename TX, bool QUANT, int RPER>
void launch_route_small(const moe_problem& p, const float* logits, const void* x, int32_t* ids, float* w,
                        int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                        float* xg_scales, int32_t* err, cudaStream_t st) {
  const dim3 grid(p.T, copy_splits(p, (int)sizeof(TX)));
  permute_small_kernel<TX, QUANT, RPER><<<grid, kSmallThreads, 0, st>>>(
      nullptr, static_cast<const TX*>(x), p.H, p.T, p.K, p.E, p.P, p.has_shared, p.layout == MOE_LAYOUT_MASKED,
      p.M_max, masked_m, offsets, row_of, src_of, xg, xg_scales, err, logits, ids, w);
}

template <typename TX, bool QUANT>
void launch_route_small_per(const moe_problem& p, const float* logits, const void* x, int32_t* ids, float* w,
                            int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                            float* xg_scales, int32_t* err, cudaStream_t st) {
  const int per = (p.E + 31) / 32;
  if (per <= 1)
    launch_route_small<TX, QUANT, 1>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
  else if (per <= 2)
    launch_route_small<TX, QUANT, 2>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
  else if (per <= 4)
    launch_route_small<TX, QUANT, 4>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
  else
    launch_route_small<TX, QUANT, 8>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
}

}  // namespace

bool route_permute_one_launch(const moe_problem& p, const int32_t* p2l) {
  return p.T > 0 && (int64_t)p.T * p.K <= kOneLaunchRecords && !p2l && p.E <= 256;
}

int launch_route_permute_small(const moe_problem& p, const float* logits, const void* x, int32_t* ids, float* w,
                               int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                               float* xg_scales, int32_t* err, cudaStream_t st) {
  if (fp8_acts(p))
    launch_route_small_per<__nv_bfloat16, true>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg,
                                                xg_scales, err, st);
  else if (p.wt == MOE_BF16)
    launch_route_small_per<__nv_bfloat16, false>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg,
                                                 xg_scales, err, st);
  else
    launch_route_small_per<float, false>(p, logits, x, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales,
                                         err, st);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t permute_workspace_bytes(const moe_problem& p) {
  size_t total = 0;
  carve(p, nullptr, &total);
  return total;
}

int launch_permute(const moe_problem& p, const int32_t* ids, const void* x, const int32_t* p2l, int32_t* masked_m,
                   int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg, float* xg_scales, int32_t* err,
                   void* ws, cudaStream_t st) {
  const PermuteWs w = carve(p, ws, nullptr);
  const int W = words_of(p.T);
  const int masked = p.layout == MOE_LAYOUT_MASKED;
  const int R = max_replicas(p);
  const int64_t n = (int64_t)p.T * p.K;
  if (p.T > 0 && ((n <= kOneLaunchRecords && !p2l) || (n <= kLayoutRecords && (int64_t)p.P * W <= kLayoutWords))) {
    // decode: one launch, or a one-CTA layout and the copy; no workspace
    if (fp8_acts(p))
      launch_small<__nv_bfloat16, true>(p, ids, x, p2l, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
    else if (p.wt == MOE_BF16)
      launch_small<__nv_bfloat16, false>(p, ids, x, p2l, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
    else
      launch_small<float, false>(p, ids, x, p2l, masked_m, offsets, row_of, src_of, xg, xg_scales, err, st);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (p.P > 0 && W > 0) {
    if (cudaMemsetAsync(w.bits, 0, (size_t)p.P * W * 4 + 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (p2l) eplb_tables_kernel<<<1, 1024, 0, st>>>(p2l, p.P, p.E, R, w.list, w.start, w.rc, err);
  if (p.T > 0) {
    mark_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(ids, p.T, p.K, p.E, p2l != nullptr, w.list, w.start, w.rc, R, w.bits, W,
                                                 w.slot_of, err);
  }
  if ((size_t)p.P * W >= 8192) {  // large bitmask (prefill): a warp per slot across the GPU
    slot_scan_kernel<<<(p.P + 7) / 8, 256, 0, st>>>(w.bits, W, p.P, p.has_shared, p.T, masked, p.M_max, w.prefix,
                                                    masked_m, offsets, err, reinterpret_cast<int*>(w.bits + (size_t)p.P * W));
  } else {
    scan_kernel<<<1, 1024, 0, st>>>(w.bits, W, p.P, p.has_shared, p.T, masked, p.M_max, w.prefix, masked_m, offsets,
                                    err);
  }
  if (p.T > 0) {
    if (fp8_acts(p)) {
      const dim3 grid(p.T, copy_splits(p, 2));
      scatter_kernel<__nv_bfloat16, true><<<grid, 256, 0, st>>>(
          (const __nv_bfloat16*)x, p.H, p.T, p.K, p.P, p.has_shared, masked, p.M_max, w.bits, w.prefix, W,
          w.slot_of, offsets, row_of, src_of, xg, xg_scales);
    } else if (p.wt == MOE_BF16) {
      const dim3 grid(p.T, copy_splits(p, 2));
      scatter_kernel<__nv_bfloat16, false><<<grid, 256, 0, st>>>(
          (const __nv_bfloat16*)x, p.H, p.T, p.K, p.P, p.has_shared, masked, p.M_max, w.bits, w.prefix, W,
          w.slot_of, offsets, row_of, src_of, xg, nullptr);
    } else {
      const dim3 grid(p.T, copy_splits(p, 4));
      scatter_kernel<float, false><<<grid, 256, 0, st>>>((const float*)x, p.H, p.T, p.K, p.P, p.has_shared, masked,
                                                         p.M_max, w.bits, w.prefix, W, w.slot_of, offsets, row_of,
                                                         src_of, xg, nullptr);
    }
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

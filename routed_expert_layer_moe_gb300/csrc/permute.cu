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
#include "common.cuh"

namespace moe {
namespace {

struct PermuteWs {
  uint32_t* bits;   // [P][W], then one int32 counter (cleared with the bits)
  int32_t* prefix;  // [P][W] rank of the first token of each 32-token word
  int32_t* slot_of; // [T*K]
  int32_t* l2p;     // [E][R]
  int32_t* rc;      // [E]
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
  w.l2p = (int32_t*)take((size_t)p.E * max_replicas(p) * 4);
  w.rc = (int32_t*)take((size_t)p.E * 4);
  if (total) *total = off;
  return w;
}

// logical_to_physical_map: for each logical expert the slots holding it in
// ascending slot order; logical_replica_count.  One CTA.
__global__ void eplb_tables_kernel(const int32_t* __restrict__ p2l, int P, int E, int R, int32_t* __restrict__ l2p,
                                   int32_t* __restrict__ rc, int32_t* err) {
  for (int s = threadIdx.x; s < P; s += blockDim.x) {
    const int e = p2l[s];
    if (e < 0 || e >= E) atomicOr(err, MOE_FLAG_BAD_MAP);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int s = 0; s < P; ++s) {
      if (p2l[s] == e) {
        if (c < R) l2p[(size_t)e * R + c] = s;
        ++c;
      }
    }
    rc[e] = c;
  }
}

__global__ void mark_kernel(const int32_t* __restrict__ ids, int T, int K, int E, int use_map,
                            const int32_t* __restrict__ l2p, const int32_t* __restrict__ rc, int R, uint32_t* bits,
                            int W, int32_t* __restrict__ slot_of, int32_t* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * K) return;
  const int t = i / K;
  const int e = ids[i];
  int s = -1;
  if (e < 0 || e >= E) {
    atomicOr(err, MOE_FLAG_BAD_EXPERT);
  } else if (use_map) {
    const int c = rc[e];
    if (c <= 0) {
      atomicOr(err, MOE_FLAG_BAD_MAP);
    } else {
      s = l2p[(size_t)e * R + (t % c)];
    }
  } else {
    s = e;
  }
  if (s >= 0) {
    const uint32_t bit = 1u << (t & 31);
    const uint32_t old = atomicOr(bits + (size_t)s * W + (t >> 5), bit);
    if (old & bit) {  // the same expert twice in one token
      atomicOr(err, MOE_FLAG_BAD_EXPERT);
      s = -1;
    }
  }
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
  if (threadIdx.x < KS) {
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
    row_of[(size_t)t * KS + k] = row;
    if (row >= 0) src_of[row] = t;
  }
  __syncthreads();
  const TX* xr = x + (size_t)t * H;
  if constexpr (QUANT) {
    // 16 threads per 128-element group, 8 bf16 elements (16 bytes) each.
    const int G = H / 128;
    const int sub = threadIdx.x & 15;
    uint8_t* q = static_cast<uint8_t*>(xg);
    for (int g0 = 0; g0 < G; g0 += (int)(blockDim.x >> 4)) {  // same trip count for every thread
      const int g = g0 + (int)(threadIdx.x >> 4);
      const bool live = g < G;
      float f[8];
      float amax = 0.0f;
      if (live) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(xr + g * 128 + sub * 8));
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&raw);
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
  } else {
    // plain copy in 16-byte vectors
    constexpr int V = 16 / sizeof(TX);
    TX* dst = static_cast<TX*>(xg);
    for (int c = threadIdx.x * V; c < H; c += blockDim.x * V) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(xr + c));
      for (int k = 0; k < KS; ++k) {
        const int r = rows[k];
        if (r < 0) continue;
        *reinterpret_cast<uint4*>(dst + (size_t)r * H + c) = raw;
      }
    }
  }
}

}  // namespace

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
  if (p.P > 0 && W > 0) {
    if (cudaMemsetAsync(w.bits, 0, (size_t)p.P * W * 4 + 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (p2l) eplb_tables_kernel<<<1, 1024, 0, st>>>(p2l, p.P, p.E, R, w.l2p, w.rc, err);
  if (p.T > 0) {
    const int n = p.T * p.K;
    mark_kernel<<<(n + 255) / 256, 256, 0, st>>>(ids, p.T, p.K, p.E, p2l != nullptr, w.l2p, w.rc, R, w.bits, W,
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
      scatter_kernel<__nv_bfloat16, true><<<p.T, 256, 0, st>>>(
          (const __nv_bfloat16*)x, p.H, p.T, p.K, p.P, p.has_shared, masked, p.M_max, w.bits, w.prefix, W,
          w.slot_of, offsets, row_of, src_of, xg, xg_scales);
    } else if (p.wt == MOE_BF16) {
      scatter_kernel<__nv_bfloat16, false><<<p.T, 256, 0, st>>>(
          (const __nv_bfloat16*)x, p.H, p.T, p.K, p.P, p.has_shared, masked, p.M_max, w.bits, w.prefix, W,
          w.slot_of, offsets, row_of, src_of, xg, nullptr);
    } else {
      scatter_kernel<float, false><<<p.T, 256, 0, st>>>((const float*)x, p.H, p.T, p.K, p.P, p.has_shared, masked,
                                                        p.M_max, w.bits, w.prefix, W, w.slot_of, offsets, row_of,
                                                        src_of, xg, nullptr);
    }
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

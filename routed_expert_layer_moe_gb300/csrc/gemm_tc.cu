// Steps 3 and 4: grouped per-expert GEMMs on the tcgen05 tensor cores.
//
// "Inference INFRA methodology (5)", section "DeepGEMM": the activations sit
// in a static expert-grouped buffer and the real row count of each expert
// (masked_m) lives in device memory; the kernel reads it at run time, so the
// launch shape is fixed and CUDA-graph capturable, and a tile that would hold
// only padding rows issues no MMA.  FP8 products are accumulated by the tensor
// core over one 128-wide K block and promoted to an FP32 accumulator with the
// weight-block and activation-group scales on the CUDA cores ("two-level
// accumulation").  "MoE inference and expert parallelism", routing section:
// the expert is SwiGLU with W1 = gate, W3 = up, W2 = down.
//
// Design (GB300, one CTA per SM, persistent):
//   * A unit is (slot s, token chunk c, tile pair j, K split q).  A slot's rows
//     are split into chunks of near-equal size (at most 64 rows for FP8 / FP4 on
//     one CTA, 128 for BF16, 256 on SM pairs), so the chunks of one expert take
//     the same time and re-read its weights from L2 together.
//     Gate/up: the pair is the gate tile (rows [128j, 128j+128) of W1) and the
//     up tile (same rows of W3).  Down: two consecutive 128-row tiles of W2.
//     Units exist only for chunks with rows: each CTA builds the unit list from
//     masked_m on the device at kernel start.  A chunk's token box is the
//     smallest of 16 / 32 / 64 / 128 rows that covers it (SM pairs: 128), so a
//     decode expert with a few tokens reads no padding rows.
//   * Two orientations:
//       - token-major (every FP8 problem, and BF16 prefill): the 128 token rows
//         are the MMA's M side and the gate and up tiles together one N = 256
//         MMA; the activation scale is one value per thread, and the SwiGLU, the
//         e4m3 re-quantisation of h and the stores are row-local.  FP8 / FP4 on
//         one CTA: chunks of at most 64 rows and M = 64 MMAs (rows 16q..16q+15
//         in lane quarter q), read with 16x256b loads, so that each thread
//         promotes two token rows and 32 values per tile and K block instead of
//         one row of a 128-row tile that decode fills with padding;
//       - weight-major (BF16 decode): the weight tile is the M = 128 side and the
//         chunk's tokens the N side, rounded up to 16 -- an expert with a few
//         tokens streams its weights at full width and issues N = 16 MMAs.
//   * SM pairs (FP8 / FP4 slots of prefill size, 128 rows or more on average):
//     clusters of two CTAs, 256-row token chunks, one cta_group::2 MMA
//     (M = 256, N = 256) per K block over both CTAs' shared memory; each CTA
//     stages its 128 token rows and one weight tile (32 KB stages, six of them)
//     and keeps its own rows' accumulators (see the kernel's comment).
//   * Warp 0: TMA producer (weights with an evict-first L2 hint).  Warp 1:
//     tensor-memory allocator and the single MMA-issuing thread.  Warps 2-3:
//     FP8 scale loaders (the activation and weight scales of up to 16 K blocks
//     per group into one half of a two-group ring in shared memory, with
//     asynchronous 4-byte copies; the epilogue waits and releases once per
//     group; keeping the scales out of the stages leaves room for four 48 KB
//     stages).  Warps 4-11: epilogue, two warps per tensor-memory lane quarter.
//   * FP8: the MMAs of one 128-K block write one of two tensor-memory buffers;
//     the epilogue reads it, scales it and adds it into fp32 registers while
//     the MMA fills the other (SM pairs: the partial sums read as packed pairs
//     and added with fp32x2 multiply-adds on paired accumulators; one CTA: the
//     16x256b form above).
//     BF16: the whole K range accumulates in tensor memory; the two buffers
//     alternate between units.
//   * MODE_FFN runs gate/up and down in one cooperative launch: the unit list
//     is the gate/up units followed by the down units, and a down unit's token
//     (h) tile and scales are read only after every gate/up unit of its slot
//     has released its rows through a per-slot counter.
//   * Every wait is bounded in time; on expiry the CTA sets an abort flag,
//     drains its copies and MMAs, frees tensor memory, reports
//     MOE_FLAG_TIMEOUT and returns.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace moe {
namespace {

constexpr int MODE_FFN = 2;         // gate/up then down in one launch (units of both phases)
constexpr int STATS_CTAS = 256;     // per-CTA issue counters kept at the start of the workspace
constexpr size_t STATS_BYTES = 2 * STATS_CTAS * 2 * sizeof(int);
constexpr int BM = 128;             // rows of one weight tile
constexpr int BN = 128;             // token rows of one chunk at most
constexpr int ROW_BYTES = 128;      // K bytes per stage row (one 128-byte swizzle span)
constexpr int TILE_A_BYTES = BM * ROW_BYTES;
constexpr int TILE_B_BYTES = BN * ROW_BYTES;
constexpr int STAGE_BYTES = 2 * TILE_A_BYTES + TILE_B_BYTES;  // weight tile 0 | weight tile 1 | token tile
constexpr int NUM_THREADS = 384;    // three warpgroups
constexpr int EPI_THREADS = 256;    // warpgroups 1 and 2
constexpr int EPI_WARP0 = 4;
constexpr int EPI_WARPS = EPI_THREADS / 32;  // epilogue barriers take one arrival per warp
constexpr int LOAD_WARP0 = 2;       // warps 2 and 3 load FP8 scales
constexpr int LOAD_THREADS = 64;
constexpr int RING = 32;            // K blocks of scales staged ahead of the epilogue
constexpr int SG = 16;              // K blocks of scales fetched per loader pass (RING / 2: two groups in flight)
constexpr int DEC_CH = 64;          // FP8 / FP4 on one CTA: token rows of one chunk at most (M = 64 MMAs)
// Register split (setmaxnreg): warpgroup 0 (TMA, MMA, scale loads) gives
// registers to the two epilogue warpgroups, which hold 2 x 64 fp32
// accumulators per thread.  4*32*ctrl + 8*32*epi must not exceed
// 384 * (registers at launch); the launcher checks it before the first launch.
template <bool F8>
struct Regs {
  static constexpr int ctrl = F8 ? 72 : 80;
  static constexpr int epi = F8 ? 216 : 208;
  static constexpr int needed = 4 * 32 * ctrl + 8 * 32 * epi;
};
constexpr uint32_t TMEM_COLS = 512;  // two accumulator buffers of 256 columns
// Bound of every wait: 4e9 SM cycles, about 2 s at the 2.07 GHz maximum clock.
constexpr long long TIMEOUT = 4000000000LL;

// One grouped GEMM of the layer (gate/up + SwiGLU, or down).
struct Phase {
  int mode;          // MODE_SWIGLU or MODE_DOWN
  int kb_total;      // 128-byte K blocks of the reduction
  int kb_per_split;  // K blocks per split
  int ksplit;
  int NA;            // weight rows per slot
  int pairs;         // tile pairs per token chunk
  int pair_stride;   // weight rows between pairs
  int a1_off;        // row of the second tile of a pair relative to the first
  int out_cols;      // columns of the output rows
  int scale_cols;    // K / 128 (e4m3 scales per row of weights and activations)
  const float* a_scales;  // weight block scales [slots * NA/128][K/128]
  const float* b_scales;  // activation group scales [rows][K/128]
  void* out;
  float* out_scales;      // e4m3 gate/up output scales [rows][I/128]
  float* part;            // split-K partial sums [ksplit][rows_total][out_cols] fp32
};

struct TcParams {
  int nslots, masked, M_max;
  uint32_t a_tile_tx;  // bytes one 128-row weight tile adds to its stage's transaction count
  uint32_t w_fmt;      // kind::f8f6f4 format of the weight operand (0 = e4m3, 5 = e2m1)
  int stages;
  int nphase;          // 1, or 2 when gate/up and down run in one launch
  const int32_t* masked_m;
  const int32_t* offsets;
  long rows_total;     // rows of the grouped buffers
  int32_t* err;
  int* ready;          // two-phase launch: gate/up units finished per slot
  int* stats;          // [2 phases][STATS_CTAS][2]: units and token tiles each CTA issued
  Phase ph[2];
  uint32_t sx_off, sw_off, red_off, pre_off, bar_off, misc_off;
};

struct Unit {
  int s, c, j, q;
  int nvalid;           // token rows of the chunk
  int rowB;             // first grouped-buffer row of the chunk
  int rowA0, rowA1;     // first weight row of tile 0 / tile 1
  int kb0, kb1;
  bool a1;              // tile 1 exists
};

__device__ __forceinline__ int slot_rows(const TcParams& p, int s) {
  int m = __ldg(p.masked_m + s);
  if (p.masked) m = min(m, p.M_max);
  return max(m, 0);
}

// srows / sbase: each slot's valid rows and first grouped-buffer row, staged in shared memory
// at kernel start (a unit's decode then needs no global load).
// CH: token rows of one chunk at most (BN, or 2 BN when a CTA pair shares one MMA); with a
// pair, rank 0 takes the first half of the chunk's rows (rounded up) and rank 1 the rest.
template <int CH = BN>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, const Phase& f, int mode, const int* prefix,
                                            const int* srows, const int* sbase, int u, uint32_t rank = 0) {
  int lo = 0, hi = p.nslots;  // prefix[lo] <= u < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  Unit U;
  U.s = lo;
  const int r = u - prefix[lo];
  const int m = srows[lo];
  const int nch = (m + CH - 1) / CH;
  U.q = r % f.ksplit;
  const int rest = r / f.ksplit;
  U.c = rest % nch;
  U.j = rest / nch;
  const int base = m / nch, extra = m - base * nch;  // near-equal chunks
  U.nvalid = base + (U.c < extra ? 1 : 0);
  U.rowB = sbase[lo] + U.c * base + min(U.c, extra);
  if constexpr (CH > BN) {
    const int n0 = (U.nvalid + 1) >> 1;
    if (rank) {
      U.rowB += n0;
      U.nvalid -= n0;
    } else {
      U.nvalid = n0;
    }
  }
  U.rowA0 = lo * f.NA + U.j * f.pair_stride;
  U.rowA1 = U.rowA0 + f.a1_off;
  U.a1 = (mode == MODE_SWIGLU) ? true : (U.j * f.pair_stride + f.a1_off < f.NA);
  U.kb0 = U.q * f.kb_per_split;
  U.kb1 = min(f.kb_total, U.kb0 + f.kb_per_split);
  return U;
}

// FP8 / FP4 on one CTA (64-row chunks, M = 64 MMAs): a[4g], a[4g + 1] += r[4g], r[4g + 1] * sa and
// a[4g + 2], a[4g + 3] += r[4g + 2], r[4g + 3] * sb for the 8 groups of a 16x256b.x8 load (two token
// rows with scales sa and sb), as packed fp32x2 multiply-adds (each element rounded as the scalar
// fmaf would)
__device__ __forceinline__ void promote_rows2(float* a, const uint32_t (&r)[32], float sa, float sb) {
  const float2 va = make_float2(sa, sa), vb = make_float2(sb, sb);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float2 q0 = __ffma2_rn(make_float2(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1])), va,
                                 make_float2(a[4 * g], a[4 * g + 1]));
    const float2 q1 = __ffma2_rn(make_float2(__uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])), vb,
                                 make_float2(a[4 * g + 2], a[4 * g + 3]));
    a[4 * g] = q0.x;
    a[4 * g + 1] = q0.y;
    a[4 * g + 2] = q1.x;
    a[4 * g + 3] = q1.y;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 64 consecutive values of one row as bf16 (128 bytes): 32-byte stores when the row is
// 32-byte aligned (wide), else 16-byte ones.
__device__ __forceinline__ void store_bf16x64(__nv_bfloat16* dst, const float* a, bool wide) {
  auto pk = [&](int v) {
    return make_uint4(pack_bf16x2(a[8 * v + 0], a[8 * v + 1]), pack_bf16x2(a[8 * v + 2], a[8 * v + 3]),
                      pack_bf16x2(a[8 * v + 4], a[8 * v + 5]), pack_bf16x2(a[8 * v + 6], a[8 * v + 7]));
  };
  if (wide) {
#pragma unroll
    for (int v = 0; v < 4; ++v) st_global_v8(dst + 16 * v, pk(2 * v), pk(2 * v + 1));
  } else {
#pragma unroll
    for (int v = 0; v < 8; ++v) reinterpret_cast<uint4*>(dst)[v] = pk(v);
  }
}

// 64 consecutive fp32 values (256 bytes), same store widths.
__device__ __forceinline__ void store_f32x64(float* dst, const float* a, bool wide) {
  auto q = [&](int v) {
    return make_uint4(__float_as_uint(a[4 * v]), __float_as_uint(a[4 * v + 1]), __float_as_uint(a[4 * v + 2]),
                      __float_as_uint(a[4 * v + 3]));
  };
  if (wide) {
#pragma unroll
    for (int v = 0; v < 8; ++v) st_global_v8(dst + 8 * v, q(2 * v), q(2 * v + 1));
  } else {
#pragma unroll
    for (int v = 0; v < 16; ++v) reinterpret_cast<uint4*>(dst)[v] = q(v);
  }
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// PAIR: the CTAs run as clusters of two on an SM pair (prefill-sized slots).  One unit is a
// chunk of up to 256 token rows: each CTA stages its half of the rows (one 128-row box) and
// one weight tile of the pair (rank 0 tile 0 = gate, rank 1 tile 1 = up), and the leader's
// MMA thread issues one cta_group::2 MMA (M = 256 token rows, N = 256 weight rows) over both
// CTAs' shared memory, so each SM stages 32 KB per K block instead of 48 KB for the same
// per-SM tensor work.  Each CTA's tensor memory then holds its own rows' gate and up columns,
// so the epilogue is the one-CTA token-major epilogue.  The MMA's completion is multicast to
// both CTAs' barriers; the peer's copies count on the leader's stage barrier; the peer's
// epilogue hands accumulator buffers back to the leader with cluster-scope arrivals.
template <bool F8, int MODE, bool TM, bool PAIR = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB16,
                           const __grid_constant__ CUtensorMap tmB32, const __grid_constant__ CUtensorMap tmB64,
                           const __grid_constant__ CUtensorMap tmB128, const __grid_constant__ CUtensorMap tmA2,
                           const __grid_constant__ CUtensorMap tmC16, const __grid_constant__ CUtensorMap tmC32,
                           const __grid_constant__ CUtensorMap tmC64, const __grid_constant__ CUtensorMap tmC128,
                           const TcParams p) {
  // tmA / tmB*: weights and token boxes of phase 0; tmA2 / tmC*: those of phase 1 (MODE_FFN)
  static_assert(TM || !F8, "FP8 / FP4 run token-major");
  static_assert(!PAIR || (F8 && TM && MODE != MODE_FFN), "SM pairs: FP8 / FP4 token-major, one GEMM per launch");
  // FP8 / FP4 on one CTA: 64-row chunks, M = 64 MMAs, the 16x256b promotion (see the epilogue)
  constexpr bool DEC = F8 && TM && !PAIR;
  constexpr int CH = PAIR ? 2 * BN : DEC ? DEC_CH : BN;  // token rows of one chunk at most
  constexpr uint32_t SB = PAIR ? TILE_A_BYTES + TILE_B_BYTES : STAGE_BYTES;  // bytes of one pipeline stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float* sx = reinterpret_cast<float*>(smem + p.sx_off);    // [RING][BN] activation scales of one K block
  float* sw = reinterpret_cast<float*>(smem + p.sw_off);    // [RING][2 tiles] weight scales of one K block
  float* red = reinterpret_cast<float*>(smem + p.red_off);  // [2 parities][512] group maxima
  int* prefix = reinterpret_cast<int*>(smem + p.pre_off);   // [nphase][nslots + 1] unit prefix
  int* srows = prefix + p.nphase * (p.nslots + 1);          // [nslots] valid rows per slot
  int* sbase = srows + p.nslots;                            // [nslots] first grouped-buffer row per slot
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* tfull = empty + p.stages;  // [2] accumulator buffer written
  uint64_t* tempty = tfull + 2;        // [2] accumulator buffer read
  uint64_t* gfull = tempty + 2;        // [2] scale group loaded (one per half of the ring)
  uint64_t* gempty = gfull + 2;        // [2] scale group consumed
  uint64_t* drain = gempty + 2;        // [1]
  uint64_t* ebar = drain + 1;          // [1] all epilogue threads
  uint64_t* fin = ebar + 1;            // [1] SM pairs: the peer CTA is done with this CTA's memory
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + p.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // SM pairs: rank 0 (the leader) issues the MMAs; units are dealt per cluster
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int unit0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int ustride = PAIR ? (int)nclusters_x() : (int)gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], PAIR ? 2 * EPI_WARPS : EPI_WARPS);  // pairs: both CTAs' epilogue warps
      mbar_init(&gfull[i], LOAD_THREADS);
      mbar_init(&gempty[i], EPI_WARPS);
    }
    mbar_init(drain, 1);
    mbar_init(ebar, EPI_WARPS);
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(tmem_base_smem, TMEM_COLS);
    tmem_relinquish<PAIR>();
  }
  // unit counts per slot -> prefix (one list per phase; the units of phase 1 follow phase 0's)
  constexpr int NPH = (MODE == MODE_FFN) ? 2 : 1;
  const int pstride = p.nslots + 1;
  for (int s = tid; s < p.nslots; s += NUM_THREADS) {
    const int m = slot_rows(p, s);
    srows[s] = m;
    sbase[s] = p.masked ? s * p.M_max : __ldg(p.offsets + s);
    const int nch = (m + CH - 1) / CH;
#pragma unroll
    for (int h = 0; h < NPH; ++h) prefix[h * pstride + s + 1] = nch * p.ph[h].pairs * p.ph[h].ksplit;
  }
  if (tid == 0) {
#pragma unroll
    for (int h = 0; h < NPH; ++h) prefix[h * pstride] = 0;
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp < NPH) {
    int* pre = prefix + warp * pstride;
    int run = 0;
    for (int base = 1; base <= p.nslots; base += 32) {
      const int i = base + lane;
      int v = (i <= p.nslots) ? pre[i] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
      }
      if (i <= p.nslots) pre[i] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  // SM pairs: both CTAs' barriers are initialised before either CTA touches the other's
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_base_smem;
  const int total0 = prefix[p.nslots];
  const int total = (MODE == MODE_FFN) ? total0 + prefix[pstride + p.nslots] : total0;
  // Two-phase launch: a down unit reads rows of h (and their scales) that gate/up units of
  // other CTAs wrote; wait (bounded) until every gate/up unit of slot s has released them.
  auto wait_ready = [&](int s) -> bool {
    const int m = srows[s];
    const int need = ((m + CH - 1) / CH) * p.ph[0].pairs * p.ph[0].ksplit * EPI_WARPS;  // one release per epilogue warp
    const long long t0 = clock64();
    while (ld_acquire_gpu(p.ready + s) < need) {
      if (*abort_flag) return false;
      if (clock64() - t0 > TIMEOUT) {
        *abort_flag = 1;
        return false;
      }
      __nanosleep(64);
    }
    fence_proxy_async_global();
    return true;
  };
  // unit u -> (phase, its GEMM mode, the unit of that phase)
  auto locate = [&](int u, int& h, int& mode) -> Unit {
    h = (MODE == MODE_FFN && u >= total0) ? 1 : 0;
    mode = (MODE == MODE_FFN) ? p.ph[h].mode : MODE;
    return decode_unit<CH>(p, p.ph[h], mode, prefix + h * pstride, srows, sbase, h ? u - total0 : u, crank);
  };

  if (warp < EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<F8>::ctrl));
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB128);
        if (!PAIR) {
          tma_prefetch_map(&tmB16);
          tma_prefetch_map(&tmB32);
          tma_prefetch_map(&tmB64);
        }
        if (MODE == MODE_FFN) {
          tma_prefetch_map(&tmA2);
          tma_prefetch_map(&tmC128);
        }
        const uint64_t pol = policy_evict_first();
        const int kb_elems = F8 ? ROW_BYTES : ROW_BYTES / 2;
        int stage = 0;
        uint32_t phase = 0;
        long issued = 0;
        bool ok = true;
        // Two-phase launch: a down unit's first stage requests its weight tiles first and its
        // token tile (rows of h) only once the slot's gate/up units have released them.
        for (int u = unit0; ok && u < total; u += ustride) {
          int h, mode;
          const Unit U = locate(u, h, mode);
          const CUtensorMap* ma = h ? &tmA2 : &tmA;
          const CUtensorMap* mb = h ? &tmC128 : &tmB128;
          // token box: the smallest of 16 / 32 / 64 / 128 rows that covers the chunk (SM pairs: 128).
          // Token-major MMAs still read 128 rows; the rows past the box hold stale shared memory
          // and only give accumulator rows past the chunk, which are never used or stored.
          int box = 128;
          if (!PAIR) {
            if (U.nvalid <= 16) {
              mb = h ? &tmC16 : &tmB16;
              box = 16;
            } else if (U.nvalid <= 32) {
              mb = h ? &tmC32 : &tmB32;
              box = 32;
            } else if (U.nvalid <= 64) {
              mb = h ? &tmC64 : &tmB64;
              box = 64;
            }
          }
          bool check_ready = (MODE == MODE_FFN) && h == 1;
          // SM pairs: the leader's stage barrier counts both CTAs' copies (a token box and one
          // weight tile each); the peer's own stage barriers are not used
          const uint32_t bytes = PAIR ? 2u * (p.a_tile_tx + (uint32_t)BN * ROW_BYTES)
                                      : p.a_tile_tx * (U.a1 ? 2u : 1u) + (uint32_t)box * ROW_BYTES;
          for (int kb = U.kb0; kb < U.kb1; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, TIMEOUT)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + (size_t)stage * SB;
            const int x = kb * kb_elems;
            if constexpr (PAIR) {
              // stage = [this CTA's 128 token rows | its weight tile]: rank 0 holds tile 0 and rank 1
              // tile 1, the two halves of the N = 256 pair MMA's B operand
              if (leader) {
                mbar_arrive_expect_tx(&full[stage], bytes);
                tma_load_2d(st, mb, &full[stage], x, U.rowB);
                tma_load_2d_hint(st + TILE_B_BYTES, ma, &full[stage], x, U.rowA0, pol);
              } else {
                const uint32_t lbar = mapa_shared(&full[stage], 0);
                tma_load_2d_pair(st, mb, lbar, x, U.rowB);
                tma_load_2d_pair_hint(st + TILE_B_BYTES, ma, lbar, x, U.rowA1, pol);
              }
              ++issued;
              if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
            tma_load_2d_hint(st, ma, &full[stage], x, U.rowA0, pol);
            if (U.a1) tma_load_2d_hint(st + TILE_A_BYTES, ma, &full[stage], x, U.rowA1, pol);
            if (check_ready) {
              check_ready = false;
              if (!wait_ready(U.s)) ok = false;  // the stage is still completed below, then the loop ends
            }
            tma_load_2d(st + 2 * TILE_A_BYTES, mb, &full[stage], x, U.rowB);
            ++issued;
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
            if (!ok) break;
          }
        }
        if (!ok && PAIR && !leader) {
          // the peer's copies count on the leader's barriers: give those in flight time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000u) {
          }
        } else if (!ok) {
          // let the copies already in flight land before the CTA's shared memory is released
          const long first = issued > p.stages ? issued - p.stages : 0;
          for (long i = first; i < issued; ++i) {
            const int st = (int)(i % p.stages);
            const uint32_t ph = (uint32_t)((i / p.stages) & 1);
            const long long t0 = clock64();
            while (!mbar_try_wait(&full[st], ph) && clock64() - t0 < TIMEOUT) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_it = 0;
        bool ok = true;
        bool any = false;
        int units[2] = {0, 0}, tiles[2] = {0, 0};
        // SM pairs: the leader issues every MMA of the pair; the peer's thread only reports zeros
        for (int u = unit0; ok && leader && u < total; u += ustride) {
          int h, mode;
          const Unit U = locate(u, h, mode);
          ++units[h];
          tiles[h] += (U.j == 0 && U.q == 0);  // one unit per (slot, token chunk) has j = q = 0
          // weight-major: M = 128 weight rows, N = tokens rounded to 16 (one MMA per tile);
          // token-major: M = 128 token rows, N = both weight tiles (one MMA); SM pairs: M = 256
          // token rows over both CTAs, N = 256 (each CTA holds one weight tile)
          // (token-major: the weights are the B operand, of format w_fmt)
          // (token-major FP8 / FP4: the weights are the B operand, of format w_fmt)
          const uint32_t idesc = PAIR ? (mma_idesc<F8>(2 * BM, 2 * BM) | (p.w_fmt << 10))
                                 : TM ? (mma_idesc<F8>(DEC ? DEC_CH : BM, U.a1 ? 2 * BM : BM) |
                                         (F8 ? p.w_fmt << 10 : 0u))
                                      : mma_idesc<F8>(BM, (U.nvalid + 15) & ~15);
          uint32_t b = 0;
          if constexpr (!F8) {
            b = acc_it & 1u;
            if (!mbar_wait(&tempty[b], ((acc_it >> 1) & 1u) ^ 1u, abort_flag, TIMEOUT)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          for (int kb = U.kb0; kb < U.kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, TIMEOUT)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            if constexpr (F8) {
              // FP8 / FP4 (token-major): one N = 256 MMA group per K block (tile 0 = gate or the
              // first down tile in columns 0-127 of buffer b, tile 1 in 128-255), a fresh partial
              // sum per block for the epilogue's promotion
              b = acc_it & 1u;
              if (!mbar_wait(&tempty[b], ((acc_it >> 1) & 1u) ^ 1u, abort_flag, TIMEOUT)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              const uint32_t st = smem_u32(smem + (size_t)stage * SB);
              // one CTA: [tile 0 | tile 1 | tokens]; pairs: [tokens | this CTA's weight tile]
              const uint64_t dtok = smem_desc_sw128(PAIR ? st : st + 2 * TILE_A_BYTES);
              const uint64_t dw = smem_desc_sw128(PAIR ? st + TILE_B_BYTES : st);
              const uint32_t d0 = tmem_base + b * 256u;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                if constexpr (PAIR)
                  tc_mma_pair_f8(d0, dtok + 2 * ks, dw + 2 * ks, idesc, ks > 0);
                else
                  tc_mma<true>(d0, dtok + 2 * ks, dw + 2 * ks, idesc, ks > 0);
              }
              any = true;
              if constexpr (PAIR) {
                tc_commit_pair(&empty[stage], 3);  // both CTAs' stages are free
                tc_commit_pair(&tfull[b], 3);      // both CTAs' accumulators are written
              } else {
                tc_commit(&empty[stage]);
                tc_commit(&tfull[b]);
              }
              ++acc_it;
              if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            const uint32_t st = smem_u32(smem + (size_t)stage * STAGE_BYTES);
            const uint64_t dw0 = smem_desc_sw128(st);
            const uint64_t dw1 = smem_desc_sw128(st + TILE_A_BYTES);
            const uint64_t dtok = smem_desc_sw128(st + 2 * TILE_A_BYTES);
            const uint32_t d0 = tmem_base + b * 256u;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint32_t acc = F8 ? (ks > 0) : (kb > U.kb0 || ks > 0);
              if constexpr (TM) {
                tc_mma<F8>(d0, dtok + 2 * ks, dw0 + 2 * ks, idesc, acc);
              } else {
                tc_mma<F8>(d0, dw0 + 2 * ks, dtok + 2 * ks, idesc, acc);
                if (U.a1) tc_mma<F8>(d0 + 128u, dw1 + 2 * ks, dtok + 2 * ks, idesc, acc);
              }
            }
            any = true;
            tc_commit(&empty[stage]);
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if constexpr (!F8) {
            if (ok) {
              tc_commit(&tfull[b]);
              ++acc_it;
            }
          }
        }
        // issue counters of this launch (no tile exists for padding rows: token tiles per GEMM =
        // sum over slots of ceil(rows / 128)); CTA 0 also clears the entries of absent CTAs
        if (p.stats) {
          for (int h = 0; h < 2; ++h) {
            if (blockIdx.x < STATS_CTAS) {
              p.stats[(h * STATS_CTAS + blockIdx.x) * 2] = units[h];
              p.stats[(h * STATS_CTAS + blockIdx.x) * 2 + 1] = tiles[h];
            }
            if (blockIdx.x == 0)
              for (int c = gridDim.x; c < STATS_CTAS; ++c) {
                p.stats[(h * STATS_CTAS + c) * 2] = 0;
                p.stats[(h * STATS_CTAS + c) * 2 + 1] = 0;
              }
          }
        }
        if (!ok && any) {
          // all MMAs issued by this thread must finish before tensor memory is freed
          if constexpr (PAIR)
            tc_commit_pair(drain, 1);
          else
            tc_commit(drain);
          const long long t0 = clock64();
          while (!mbar_try_wait(drain, 0) && clock64() - t0 < TIMEOUT) {
          }
        }
      }
    } else if (F8) {
      // ------------------------------------------------------------ FP8 scale loaders
      // The activation and weight scales of up to SG K blocks per group go into one half of
      // a two-group ring in shared memory with asynchronous 4-byte copies; the loaders never
      // wait for data, so the ring runs a group ahead of the epilogue.  The group's gfull
      // barrier completes when the copies issued by all loader threads have landed; the
      // epilogue waits on it once per group and releases the half once per group, so the
      // scales cost it no barrier operation per K block.
      const int lt = tid - LOAD_WARP0 * 32;
      uint32_t gi = 0;  // groups staged so far
      bool ok = true;
      for (int u = unit0; ok && u < total; u += ustride) {
        int h, mode;
        const Unit U = locate(u, h, mode);
        const Phase& f = p.ph[h];
        const int ra0 = U.rowA0 / BM, ra1 = U.rowA1 / BM;
        bool check_ready = (MODE == MODE_FFN) && h == 1;  // h scales of a down unit: written by gate/up units
        for (int k0 = U.kb0; ok && k0 < U.kb1; k0 += SG, ++gi) {
          const int nk = min(SG, U.kb1 - k0);
          const uint32_t gh = gi & 1u;  // half of the ring
          if (!mbar_wait(&gempty[gh], ((gi >> 1) & 1u) ^ 1u, abort_flag, TIMEOUT)) {
            ok = false;
            break;
          }
          if (check_ready) {
            check_ready = false;
            if (!wait_ready(U.s)) {
              ok = false;
              break;
            }
          }
          float* sxg = sx + gh * SG * BN;  // [SG][BN]
          float* swg = sw + gh * SG * 2;   // [SG][2 tiles]
          // activation scales of the chunk's rows: element (c, j) = b_scales[rowB + c][k0 + j]
          const int n = U.nvalid * nk;
          for (int idx = lt; idx < n; idx += LOAD_THREADS) {
            const int c = idx / nk, j = idx - c * nk;
            cp_async4(sxg + j * BN + c, f.b_scales + (size_t)(U.rowB + c) * f.scale_cols + k0 + j);
          }
          // weight block scales of the two tiles (a missing second tile's value is never used)
          for (int idx = lt; idx < 2 * nk; idx += LOAD_THREADS) {
            const int j = idx >> 1, t = idx & 1;
            if (t == 0 || U.a1)
              cp_async4(swg + j * 2 + t, f.a_scales + (size_t)(t ? ra1 : ra0) * f.scale_cols + k0 + j);
          }
          cp_async_arrive_noinc(&gfull[gh]);
        }
      }
      cp_async_wait_all();  // no copy may land after the CTA has exited
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Regs<F8>::epi));
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;             // tensor-memory lane quarter this warp may access
    const int half = (warp - EPI_WARP0) >> 2; // column half (warpgroup 1 or 2)
    const int lrow = quarter * 32 + lane;     // tensor-memory lane of this thread
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t acc_it = 0, g_it = 0, u_it = 0;
    uint32_t ephase = 0;
    bool ok = true;
    // one arrival per warp, after the warp's own threads are ordered by __syncwarp
    auto warp_arrive = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    // Two-phase launch: each epilogue warp releases its rows of a finished gate/up unit later,
    // once the stores have long landed (after the next unit's K loop, or before a down unit,
    // which may itself be waiting for them); the down side counts EPI_WARPS releases per unit.
    int pending = -1;
    auto release_pending = [&]() {
      if (MODE == MODE_FFN && pending >= 0) {
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_gpu_add(p.ready + pending, 1);
        pending = -1;
      }
    };
    // bounded barriers among the epilogue threads (a plain bar.sync could not give up)
    auto epi_sync = [&]() {
      warp_arrive(ebar);
      const bool r = mbar_wait(ebar, ephase, abort_flag, TIMEOUT);
      ephase ^= 1u;
      return r;
    };
    for (int u = unit0; ok && u < total; u += ustride, ++u_it) {
      int h, mode;
      const Unit U = locate(u, h, mode);
      const Phase& f = p.ph[h];
      const size_t oc = (size_t)f.out_cols;
      const int nkb = U.kb1 - U.kb0;
      const bool split = f.ksplit > 1;
      // FP8 / FP4 on one CTA: the M = 64 accumulator row r sits in lane 32 (r / 16) + r % 16; each
      // warp reads its quarter's 16 rows with 16x256b loads, so thread t holds token rows
      // mr0 = 16 q + t / 4 and mr1 = mr0 + 8, columns c_lo + 8 g + mc and the next one of every
      // 8-column group g (half the values of a 32x32b read of all 128 lanes, and none from the
      // lanes the M = 64 layout leaves empty)
      const int mr0 = quarter * 16 + (lane >> 2), mr1 = mr0 + 8, mc = 2 * (lane & 3);
      if (h == 1) release_pending();
      // weight-major: this thread owns weight row lrow of each tile and token columns
      // [c_lo, c_lo + ncols); token-major (BF16, SM pairs): token row lrow and weight columns
      // [64*half, +64); FP8 / FP4 on one CTA: rows mr0, mr1 within the same columns
      const int c_lo = half * 64;
      const int ncols = TM ? 64 : max(0, min(64, U.nvalid - c_lo));
      const int npair = (ncols + 31) >> 5;  // 32-column loads
      float acc0[64], acc1[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        acc0[i] = 0.0f;
        acc1[i] = 0.0f;
      }

      if constexpr (F8) {
        // SM pairs: the fp32 accumulators as packed pairs (accp0[i] = columns c_lo + 2i, 2i+1 of
        // tile 0), unpacked into acc0 / acc1 after the K loop
        uint64_t accp0[32], accp1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          accp0[i] = 0;
          accp1[i] = 0;
        }
        for (int k = 0; k < nkb; ++k) {
          const int j = k % SG;  // K block within its scale group (groups restart with each unit)
          const uint32_t gh = g_it & 1u;  // half of the scale ring
          if (j == 0 && !mbar_wait(&gfull[gh], (g_it >> 1) & 1u, abort_flag, TIMEOUT)) {
            ok = false;
            break;
          }
          const uint32_t b = acc_it & 1u;
          if (!mbar_wait(&tfull[b], (acc_it >> 1) & 1u, abort_flag, TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int slot = (int)gh * SG + j;
          if constexpr (PAIR) {
            const float xs = sx[slot * BN + lrow];
            const float s0 = sw[slot * 2] * xs, s1 = sw[slot * 2 + 1] * xs;
            // SM pairs: two steps of 64 columns (tile 0 and tile 1, columns c_lo.. then c_lo+32..),
            // loaded as packed pairs and added with fp32x2 multiply-adds on paired accumulators;
            // the buffer is handed back once the second step is loaded, before its multiply-adds
            const uint64_t p0 = pair_of(s0), p1 = pair_of(s1);
            const uint32_t c0 = t_lane + b * 256u + (uint32_t)c_lo;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              uint64_t v[32];
              tmem_ld32x2_pairs(c0 + (uint32_t)(pr * 32), c0 + 128u + (uint32_t)(pr * 32), v);
              if (pr == 1) {
                tc_fence_before_sync();
                if (!leader) {  // to the leader's MMA thread, which waits on its own barrier
                  __syncwarp();
                  if (lane == 0) mbar_arrive_remote(mapa_shared(&tempty[b], 0));
                } else {
                  warp_arrive(&tempty[b]);
                }
              }
              fma2_pairs<16>(accp0 + pr * 16, v, p0);
              fma2_pairs<16>(accp1 + pr * 16, v + 16, p1);
            }
          } else {
            // one CTA: 64 columns of each tile, 32 values a thread (two token rows); the buffer is
            // handed back once loaded, before the multiply-adds
            uint32_t ra[32], rb[32];
            const uint32_t c0 = t_lane + b * 256u + (uint32_t)c_lo;
            tmem_ld16x256_x8(c0, ra);
            tmem_ld16x256_x8(c0 + 128u, rb);
            tmem_wait_ld32(ra);
            tmem_wait_ld32(rb);
            tc_fence_before_sync();
            warp_arrive(&tempty[b]);
            const float w0 = sw[slot * 2], w1 = sw[slot * 2 + 1];
            const float xa = sx[slot * BN + mr0], xb = sx[slot * BN + mr1];
            promote_rows2(acc0, ra, w0 * xa, w0 * xb);
            promote_rows2(acc1, rb, w1 * xa, w1 * xb);
          }
          if (j == SG - 1 || k == nkb - 1) {  // the group's scales are no longer read
            warp_arrive(&gempty[gh]);
            ++g_it;
          }
          ++acc_it;
        }
        if (!ok) break;
        if constexpr (PAIR) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc0[2 * i] = __uint_as_float((uint32_t)accp0[i]);
          acc0[2 * i + 1] = __uint_as_float((uint32_t)(accp0[i] >> 32));
          acc1[2 * i] = __uint_as_float((uint32_t)accp1[i]);
          acc1[2 * i + 1] = __uint_as_float((uint32_t)(accp1[i] >> 32));
        }
        }
      } else {
        // BF16: the accumulator of the whole K range (or this split of it) is in tensor memory
        const uint32_t b = acc_it & 1u;
        if (!mbar_wait(&tfull[b], (acc_it >> 1) & 1u, abort_flag, TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          if (pr < npair) {
            float v0[32], v1[32];
            const uint32_t col = b * 256u + (uint32_t)(c_lo + pr * 32);
            tmem_ld32x2(t_lane + col, t_lane + col + 128u, v0, v1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              acc0[pr * 32 + i] = v0[i];
              acc1[pr * 32 + i] = v1[i];
            }
          }
        }
        tc_fence_before_sync();
        warp_arrive(&tempty[b]);
        ++acc_it;
      }

      if constexpr (DEC) {
        // acc0 / acc1 [4g], [4g + 1] = row mr0, columns c_lo + 8g + mc (+ 1) of tile 0 / 1;
        // [4g + 2], [4g + 3] = the same columns of row mr1
        {
          const bool v0 = mr0 < U.nvalid, v1 = mr1 < U.nvalid;
          if (split) {
            float* pq = f.part + (size_t)U.q * p.rows_total * oc + (size_t)U.j * f.pair_stride + c_lo + mc;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              if (v0) {
                float* d = pq + (size_t)(U.rowB + mr0) * oc + 8 * g;
                *reinterpret_cast<float2*>(d) = make_float2(acc0[4 * g], acc0[4 * g + 1]);
                if (U.a1) *reinterpret_cast<float2*>(d + BM) = make_float2(acc1[4 * g], acc1[4 * g + 1]);
              }
              if (v1) {
                float* d = pq + (size_t)(U.rowB + mr1) * oc + 8 * g;
                *reinterpret_cast<float2*>(d) = make_float2(acc0[4 * g + 2], acc0[4 * g + 3]);
                if (U.a1) *reinterpret_cast<float2*>(d + BM) = make_float2(acc1[4 * g + 2], acc1[4 * g + 3]);
              }
            }
            continue;
          }
          release_pending();
          if (mode == MODE_SWIGLU) {
            // e4m3 per 1x128 group: a row's 128 columns of tile j sit in the four threads of a quad
            // of both column halves
            float hv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) hv[i] = silu(acc0[i]) * acc1[i];
            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              a0 = fmaxf(a0, fmaxf(fabsf(hv[4 * g]), fabsf(hv[4 * g + 1])));
              a1 = fmaxf(a1, fmaxf(fabsf(hv[4 * g + 2]), fabsf(hv[4 * g + 3])));
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
              a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, off));
              a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, off));
            }
            float* redp = red + (size_t)(u_it & 1u) * 512;  // [2 halves][128 rows]
            if ((lane & 3) == 0) {
              redp[half * 128 + mr0] = a0;
              redp[half * 128 + mr1] = a1;
            }
            if (!epi_sync()) break;
            const float m0 = fmaxf(redp[mr0], redp[128 + mr0]), m1 = fmaxf(redp[mr1], redp[128 + mr1]);
            const float sc0 = (m0 == 0.0f) ? 1.0f : __fdiv_rn(m0, 448.0f);
            const float sc1 = (m1 == 0.0f) ? 1.0f : __fdiv_rn(m1, 448.0f);
            const float i0 = 1.0f / sc0, i1 = 1.0f / sc1;
            uint8_t* o8 = static_cast<uint8_t*>(f.out) + (size_t)U.j * BM + c_lo + mc;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              if (v0)
                *reinterpret_cast<__nv_fp8x2_storage_t*>(o8 + (size_t)(U.rowB + mr0) * oc + 8 * g) =
                    __nv_cvt_float2_to_fp8x2(make_float2(hv[4 * g] * i0, hv[4 * g + 1] * i0), __NV_SATFINITE,
                                             __NV_E4M3);
              if (v1)
                *reinterpret_cast<__nv_fp8x2_storage_t*>(o8 + (size_t)(U.rowB + mr1) * oc + 8 * g) =
                    __nv_cvt_float2_to_fp8x2(make_float2(hv[4 * g + 2] * i1, hv[4 * g + 3] * i1), __NV_SATFINITE,
                                             __NV_E4M3);
            }
            if (half == 0 && (lane & 3) == 0) {
              if (v0) f.out_scales[(size_t)(U.rowB + mr0) * (oc / 128) + U.j] = sc0;
              if (v1) f.out_scales[(size_t)(U.rowB + mr1) * (oc / 128) + U.j] = sc1;
            }
          } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(f.out) + (size_t)U.j * f.pair_stride + c_lo + mc;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              if (v0) {
                __nv_bfloat16* d = o + (size_t)(U.rowB + mr0) * oc + 8 * g;
                *reinterpret_cast<uint32_t*>(d) = pack_bf16x2(acc0[4 * g], acc0[4 * g + 1]);
                if (U.a1) *reinterpret_cast<uint32_t*>(d + BM) = pack_bf16x2(acc1[4 * g], acc1[4 * g + 1]);
              }
              if (v1) {
                __nv_bfloat16* d = o + (size_t)(U.rowB + mr1) * oc + 8 * g;
                *reinterpret_cast<uint32_t*>(d) = pack_bf16x2(acc0[4 * g + 2], acc0[4 * g + 3]);
                if (U.a1) *reinterpret_cast<uint32_t*>(d + BM) = pack_bf16x2(acc1[4 * g + 2], acc1[4 * g + 3]);
              }
            }
          }
          if (MODE == MODE_FFN && mode == MODE_SWIGLU) pending = U.s;  // released later (see release_pending)
          continue;
        }
      } else {
      if (split) {
        // this split's fp32 partial sums go to the dense [split][row][column] workspace; a
        // separate reduction kernel adds the splits in split order (no atomics, no waits)
        float* pq = f.part + (size_t)U.q * p.rows_total * oc;
        if constexpr (TM) {
          if (lrow < U.nvalid) {
            float* prow = pq + (size_t)(U.rowB + lrow) * oc + (size_t)U.j * f.pair_stride + c_lo;
            const bool wide = (reinterpret_cast<uintptr_t>(f.part) & 31u) == 0;  // offsets are 256-byte multiples
            store_f32x64(prow, acc0, wide);
            if (U.a1) store_f32x64(prow + BM, acc1, wide);
          }
        } else {
          const size_t col0 = (size_t)U.j * f.pair_stride + lrow;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (i < ncols) {
              float* prow = pq + (size_t)(U.rowB + c_lo + i) * oc;
              prow[col0] = acc0[i];
              if (U.a1) prow[col0 + BM] = acc1[i];
            }
          }
        }
        continue;
      }

      release_pending();
      // ---- final values of this unit
      float* redp = red + (size_t)(u_it & 1u) * 512;  // maxima, double-buffered by unit parity
      if constexpr (TM) {
        const bool row_ok = lrow < U.nvalid;
        const size_t row = (size_t)(U.rowB + lrow);
        if (mode == MODE_SWIGLU) {
          // rows past the chunk hold other tokens' data: no SwiGLU, no store
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 64; ++i) acc0[i] = silu(acc0[i]) * acc1[i];
          }
          const size_t col = (size_t)U.j * BM + c_lo;
          if constexpr (F8) {
            // e4m3 per 1x128 group: the group is this row's 128 columns of the tile (two halves)
            float a = 0.0f;
            if (row_ok) {
#pragma unroll
              for (int i = 0; i < 64; ++i) a = fmaxf(a, fabsf(acc0[i]));
            }
            redp[half * 128 + lrow] = a;
            if (!epi_sync()) break;
            if (row_ok) {
              const float amax = fmaxf(redp[lrow], redp[128 + lrow]);
              const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
              const float inv = 1.0f / sc;  // one division per group; the codes use h * (1/s)
              uint8_t* dst = static_cast<uint8_t*>(f.out) + row * oc + col;
              auto pk = [&](int v) {
                const float* h = acc0 + 16 * v;
                return make_uint4(pack_e4m3x4(h[0] * inv, h[1] * inv, h[2] * inv, h[3] * inv),
                                  pack_e4m3x4(h[4] * inv, h[5] * inv, h[6] * inv, h[7] * inv),
                                  pack_e4m3x4(h[8] * inv, h[9] * inv, h[10] * inv, h[11] * inv),
                                  pack_e4m3x4(h[12] * inv, h[13] * inv, h[14] * inv, h[15] * inv));
              };
              if ((reinterpret_cast<uintptr_t>(f.out) & 31u) == 0) {  // row and column offsets: 64-byte multiples
                st_global_v8(dst, pk(0), pk(1));
                st_global_v8(dst + 32, pk(2), pk(3));
              } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(dst)[v] = pk(v);
              }
              if (half == 0) f.out_scales[row * (oc / 128) + U.j] = sc;
            }
          } else {
            if (row_ok)
              store_bf16x64(static_cast<__nv_bfloat16*>(f.out) + row * oc + col, acc0,
                            (reinterpret_cast<uintptr_t>(f.out) & 31u) == 0);
          }
        } else {
          if (row_ok) {
            __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(f.out) + row * oc + (size_t)U.j * f.pair_stride + c_lo;
            const bool wide = (reinterpret_cast<uintptr_t>(f.out) & 31u) == 0;  // offsets are 128-byte multiples
            store_bf16x64(yrow, acc0, wide);
            if (U.a1) store_bf16x64(yrow + BM, acc1, wide);
          }
        }
      } else {
        // weight-major: this thread holds output column (weight row) col0 for token columns c_lo + i
        const int col0 = (mode == MODE_SWIGLU) ? U.j * BM + lrow : U.j * f.pair_stride + lrow;
        {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(f.out);
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (i < ncols) {
              const size_t row = (size_t)(U.rowB + c_lo + i);
              if (mode == MODE_SWIGLU) {
                o[row * oc + col0] = __float2bfloat16_rn(silu(acc0[i]) * acc1[i]);
              } else {
                o[row * oc + col0] = __float2bfloat16_rn(acc0[i]);
                if (U.a1) o[row * oc + col0 + BM] = __float2bfloat16_rn(acc1[i]);
              }
            }
          }
        }
      }
      if (MODE == MODE_FFN && mode == MODE_SWIGLU) pending = U.s;  // released later (see release_pending)
      }
    }
    release_pending();
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) {
    // Neither CTA of the pair frees its tensor memory or leaves while the other may still use
    // it: the leader's MMAs read the peer's shared memory and write its tensor memory, the
    // peer's copies and buffer releases land on the leader's barriers.  Each CTA tells the
    // other it is done (all of its roles have finished above) and waits, bounded, for the
    // other's word.
    if (tid == 0) {
      mbar_arrive_remote(mapa_shared(fin, crank ^ 1u));
      const long long t0 = clock64();
      while (!mbar_try_wait<true>(fin, 0)) {
        if (clock64() - t0 > TIMEOUT) {
          *abort_flag = 1;
          break;
        }
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) atomicOr(p.err, MOE_FLAG_TIMEOUT);
}

// Split-K: out[row][col] = bf16(sum over splits q = 0..ksplit-1, in order, of part[q][row][col])
// for every valid grouped row (padding rows are left untouched).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int ksplit, long rows,
                                                            int cols, const int32_t* __restrict__ masked_m,
                                                            const int32_t* __restrict__ offsets, int nslots,
                                                            int masked, int M_max, __nv_bfloat16* __restrict__ out) {
  const long row = blockIdx.x;
  if (masked) {
    const int s = (int)(row / M_max);
    if ((int)(row - (long)s * M_max) >= min(__ldg(masked_m + s), M_max)) return;
  } else if (row >= __ldg(offsets + nslots)) {
    return;
  }
  const int c = (int)(blockIdx.y * blockDim.x + threadIdx.x) * 4;  // one float4 of the row per thread
  if (c >= cols) return;
  // the splits are added in split order; up to eight are requested before the adds
  constexpr int QB = 8;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 < ksplit; q0 += QB) {
    float4 v[QB];
#pragma unroll
    for (int j = 0; j < QB; ++j)
      if (q0 + j < ksplit)
        v[j] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)(q0 + j) * rows + row) * cols + c));
#pragma unroll
    for (int j = 0; j < QB; ++j) {
      if (q0 + j < ksplit) {
        acc.x += v[j].x;
        acc.y += v[j].y;
        acc.z += v[j].z;
        acc.w += v[j].w;
      }
    }
  }
  uint2 o;
  o.x = pack_bf16x2(acc.x, acc.y);
  o.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + (size_t)row * cols + c) = o;
}

// Split-K reduction and combine in one kernel ("MoE inference and expert parallelism",
// routing section: moe_sum weighs each token's K expert outputs by its route weights, plus
// the shared expert with weight 1): for token t and each of its records k in order, the
// record's row of the down GEMM is reduced over the splits exactly as splitk_reduce_kernel
// does (fp32 adds in split order, one rounding to bf16, stored to yg), and that bf16 value
// enters the token's fp32 sum as in combine_kernel (fmaf in k order, one rounding) -- the
// same yg and out as the two kernels.  One CTA per (token, 1024 columns), 8 columns a thread.
__global__ void __launch_bounds__(128) splitk_reduce_combine_kernel(
    const float* __restrict__ part, int ksplit, long rows, int H, const int32_t* __restrict__ row_of,
    const float* __restrict__ w, int K, int KS, __nv_bfloat16* __restrict__ yg, __nv_bfloat16* __restrict__ out) {
  const int t = blockIdx.x;
  const int c = (int)(blockIdx.y * blockDim.x + threadIdx.x) * 8;
  __shared__ int rws[33];
  __shared__ float wts[33];
  if ((int)threadIdx.x < KS) {
    rws[threadIdx.x] = row_of[(size_t)t * KS + threadIdx.x];
    wts[threadIdx.x] = ((int)threadIdx.x < K) ? w[(size_t)t * K + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  if (c >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int k = 0; k < KS; ++k) {
    const int row = rws[k];
    if (row < 0) continue;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    constexpr int QB = 8;
    for (int q0 = 0; q0 < ksplit; q0 += QB) {
      float4 v0[QB], v1[QB];
#pragma unroll
      for (int j = 0; j < QB; ++j) {
        if (q0 + j < ksplit) {
          const float* src = part + ((size_t)(q0 + j) * rows + row) * H + c;
          v0[j] = __ldcg(reinterpret_cast<const float4*>(src));
          v1[j] = __ldcg(reinterpret_cast<const float4*>(src + 4));
        }
      }
#pragma unroll
      for (int j = 0; j < QB; ++j) {
        if (q0 + j < ksplit) {
          a0.x += v0[j].x;
          a0.y += v0[j].y;
          a0.z += v0[j].z;
          a0.w += v0[j].w;
          a1.x += v1[j].x;
          a1.y += v1[j].y;
          a1.z += v1[j].z;
          a1.w += v1[j].w;
        }
      }
    }
    uint4 yv;
    yv.x = pack_bf16x2(a0.x, a0.y);
    yv.y = pack_bf16x2(a0.z, a0.w);
    yv.z = pack_bf16x2(a1.x, a1.y);
    yv.w = pack_bf16x2(a1.z, a1.w);
    *reinterpret_cast<uint4*>(yg + (size_t)row * H + c) = yv;
    const float wk = wts[k];
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&yv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(hv[i]);
      acc[2 * i] = fmaf(wk, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wk, f.y, acc[2 * i + 1]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = o;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct Plan {
  int ksplit, kb_per_split, kb_total, stages, nslots, pairs;
  bool tm;
  bool pair;  // clusters of two CTAs sharing cta_group::2 MMAs over 256-row token chunks
  size_t smem;
  uint32_t sx_off, sw_off, red_off, pre_off, bar_off, misc_off;
  size_t part_bytes;
};

// SM pairs for FP8 / FP4 slots of prefill size (128 rows or more on average): one 256-row
// chunk per slot instead of two 128-row chunks that each stage the slot's weight tiles, and
// 32 KB stages (each SM holds its token rows and one weight tile).  The down GEMM needs
// whole pairs of weight tiles (H a multiple of 256); the one-launch FFN stays on single CTAs.
bool use_pairs(const moe_problem& p, int mode, int nphase) {
  const double rows_per_slot = (double)p.T * p.K / std::max(1, p.P);
  return fp8_acts(p) && nphase == 1 && rows_per_slot >= 128.0 && (mode == MODE_SWIGLU || p.H % 256 == 0);
}

Plan make_plan(const moe_problem& p, int mode, int sm_count, int smem_cap, int nphase = 1) {
  Plan pl{};
  const bool f8 = fp8_acts(p);
  const int esz = f8 ? 1 : 2;
  const int K = (mode == MODE_SWIGLU) ? p.H : p.I;
  const int NA = (mode == MODE_SWIGLU) ? 2 * p.I : p.H;
  pl.kb_total = K * esz / ROW_BYTES;
  pl.nslots = p.P + p.has_shared;
  pl.pairs = (mode == MODE_SWIGLU) ? p.I / BM : (NA + 2 * BM - 1) / (2 * BM);
  // Token-major for FP8 / FP4 always: the activation scale is then one value per thread and
  // the SwiGLU / e4m3 re-quantisation of h are row-local.  A weight-major FP8 variant (tokens
  // as the MMA's N) measured slower even for decode experts with two to eight tokens.  BF16
  // needs no promotion; there weight-major is kept for decode-sized experts.
  const double rows_per_slot = (double)p.T * p.K / std::max(1, p.P);
  pl.tm = f8 || rows_per_slot >= 64.0;
  pl.pair = use_pairs(p, mode, nphase);
  const int ch = pl.pair ? 2 * BN : f8 ? DEC_CH : BN;  // token rows of one chunk at most
  // upper bound of the token chunks over all slots
  long chunks;
  if (p.layout == MOE_LAYOUT_MASKED) {
    chunks = (long)pl.nslots * ((p.M_max + ch - 1) / ch);
  } else {
    const long rows = (long)p.T * p.K + (long)p.has_shared * p.T;
    chunks = std::min<long>((long)pl.nslots * ((p.T + ch - 1) / ch), pl.nslots + rows / ch);
  }
  const long tiles = chunks * pl.pairs;
  pl.ksplit = 1;
  if (mode == MODE_DOWN && !pl.pair && tiles > 0 && tiles < 3L * sm_count) {
    // split K so the unit count fills whole waves; keep >= 4 K blocks per split
    double best = 0.0;
    for (int ks = 1; ks <= 16 && pl.kb_total / ks >= 4; ++ks) {
      const double waves = (double)(tiles * ks) / sm_count;
      const double eff = waves / std::ceil(waves);
      if (eff > best + 0.02) {
        best = eff;
        pl.ksplit = ks;
      }
      if (waves >= 2.0 && eff >= 0.9) {
        pl.ksplit = ks;
        break;
      }
    }
  }
  pl.kb_per_split = (pl.kb_total + pl.ksplit - 1) / pl.ksplit;
  pl.ksplit = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  // the partial sums live in a dense [split][row][column] fp32 workspace; keep it modest
  const size_t out_cols = (mode == MODE_SWIGLU) ? p.I : p.H;
  if (pl.ksplit > 1 && (size_t)pl.ksplit * grouped_rows(p) * out_cols * 4 > (size_t(1) << 30)) {
    pl.ksplit = 1;
    pl.kb_per_split = pl.kb_total;
  }
  // shared memory carve (offsets relative to the 1024-aligned base)
  size_t extra = 0;
  auto carve = [&](size_t bytes, size_t align) {
    extra = align_up(extra, align);
    const size_t off = extra;
    extra += bytes;
    return off;
  };
  const size_t sx_b = f8 ? (size_t)RING * BN * 4 : 0;
  const size_t sw_b = f8 ? (size_t)RING * 2 * 4 : 0;
  const size_t red_b = (size_t)2 * 512 * 4;
  const size_t pre_b = ((size_t)nphase * (pl.nslots + 1) + 2 * (size_t)pl.nslots) * 4;  // prefix, rows, bases
  pl.stages = 0;
  const size_t stage_bytes = pl.pair ? (size_t)(TILE_A_BYTES + TILE_B_BYTES) : (size_t)STAGE_BYTES;
  for (int st = 8; st >= 2; --st) {
    extra = (size_t)st * stage_bytes;
    pl.sx_off = (uint32_t)carve(sx_b, 16);
    pl.sw_off = (uint32_t)carve(sw_b, 16);
    pl.red_off = (uint32_t)carve(red_b, 16);
    pl.pre_off = (uint32_t)carve(pre_b, 16);
    pl.bar_off = (uint32_t)carve((size_t)(2 * st + 16) * 8, 8);
    pl.misc_off = (uint32_t)carve(16, 16);
    const size_t total = extra + 1024;
    if ((int)total <= smem_cap) {
      pl.stages = st;
      pl.smem = total;
      break;
    }
  }
  pl.part_bytes = pl.ksplit > 1 ? (size_t)pl.ksplit * grouped_rows(p) * out_cols * 4 : 0;
  return pl;
}

// Register split and shared-memory limit of one kernel instantiation, checked once per device
// (the flags are per instantiation: all of them share one function type).
template <bool F8, int MODE, bool TM, bool PAIR = false>
int prepare_kernel() {
  auto kern = grouped_gemm_tc_kernel<F8, MODE, TM, PAIR>;
  const int needed_regs = Regs<F8>::needed;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && attr_set[dev]) return MOE_OK;
  // the register split must fit in what the launch provides, or setmaxnreg.inc would wait forever
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return MOE_ERR_CUDA;
  if (fa.numRegs * NUM_THREADS < needed_regs) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_info().max_smem_optin) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (dev < 64) attr_set[dev] = true;
  return MOE_OK;
}

// Tensor maps of one GEMM: the weights (tA) and the grouped activations in 16/32/64/128-row boxes.
int make_maps(const moe_problem& p, int mode, const void* act, const void* w, CUtensorMap& tA, CUtensorMap* tB) {
  const bool f8 = fp8_acts(p);
  const int esz = f8 ? 1 : 2;
  const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int K = (mode == MODE_SWIGLU) ? p.H : p.I;
  const int NA = (mode == MODE_SWIGLU) ? 2 * p.I : p.H;
  const uint64_t rowsA = (uint64_t)(p.P + p.has_shared) * NA;
  const uint64_t rowsB = (uint64_t)grouped_rows(p);
  const uint32_t box_k = ROW_BYTES / esz;
  // e2m1 weights: packed 4-bit rows of K/2 bytes; TMA spreads each 8 bytes of codes over
  // 16 bytes of shared memory (the layout kind::f8f6f4 reads) and counts the 8 bytes read
  const bool w4 = p.wt == MOE_E2M1;
  if (encode_tensor_map(&tA, w4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : dt, K, rowsA,
                        w4 ? (uint64_t)K / 2 : (uint64_t)K * esz, box_k, BM, w) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;
  const int boxes[4] = {16, 32, 64, 128};
  for (int i = 0; i < 4; ++i)
    if (encode_tensor_map(&tB[i], dt, K, rowsB, (uint64_t)K * esz, box_k, boxes[i], act) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  return MOE_OK;
}

Phase make_phase(const moe_problem& p, int mode, const Plan& pl, const float* act_scales, const float* w_scales,
                 void* out, float* out_scales, float* part) {
  Phase f{};
  const int K = (mode == MODE_SWIGLU) ? p.H : p.I;
  f.mode = mode;
  f.kb_total = pl.kb_total;
  f.kb_per_split = pl.kb_per_split;
  f.ksplit = pl.ksplit;
  f.NA = (mode == MODE_SWIGLU) ? 2 * p.I : p.H;
  f.pairs = pl.pairs;
  f.pair_stride = (mode == MODE_SWIGLU) ? BM : 2 * BM;
  f.a1_off = (mode == MODE_SWIGLU) ? p.I : BM;
  f.out_cols = (mode == MODE_SWIGLU) ? p.I : p.H;
  f.scale_cols = K / 128;
  f.a_scales = w_scales;
  f.b_scales = act_scales;
  f.out = out;
  f.out_scales = out_scales;
  f.part = pl.ksplit > 1 ? part : nullptr;
  return f;
}

TcParams make_params(const moe_problem& p, const Plan& pl, const int32_t* masked_m, const int32_t* offsets,
                     int32_t* err) {
  TcParams prm{};
  prm.nslots = pl.nslots;
  prm.masked = p.layout == MOE_LAYOUT_MASKED;
  prm.M_max = p.M_max;
  const bool w4 = p.wt == MOE_E2M1;
  prm.a_tile_tx = w4 ? TILE_A_BYTES / 2 : TILE_A_BYTES;
  prm.w_fmt = w4 ? 5u : 0u;
  prm.stages = pl.stages;
  prm.nphase = 1;
  prm.masked_m = masked_m;
  prm.offsets = offsets;
  prm.rows_total = (long)grouped_rows(p);
  prm.err = err;
  prm.sx_off = pl.sx_off;
  prm.sw_off = pl.sw_off;
  prm.red_off = pl.red_off;
  prm.pre_off = pl.pre_off;
  prm.bar_off = pl.bar_off;
  prm.misc_off = pl.misc_off;
  return prm;
}

// After the down GEMM: the split-K reduction (when the GEMM was split), and the combine when
// comb is given -- fused into the reduction, or on its own after an unsplit GEMM.
int launch_reduce(const moe_problem& p, const Plan& pl, const Phase& f, const int32_t* masked_m,
                  const int32_t* offsets, cudaStream_t st, const CombineArgs* comb = nullptr) {
  if (comb && pl.ksplit > 1) {
    if (p.T == 0) return MOE_OK;
    const dim3 grid((unsigned)p.T, (unsigned)((p.H / 8 + 127) / 128));
    splitk_reduce_combine_kernel<<<grid, 128, 0, st>>>(f.part, pl.ksplit, (long)grouped_rows(p), p.H, comb->row_of,
                                                       comb->w, p.K, p.K + p.has_shared,
                                                       static_cast<__nv_bfloat16*>(f.out),
                                                       static_cast<__nv_bfloat16*>(comb->out));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (comb) return launch_combine(p, f.out, comb->row_of, comb->w, comb->out, st);
  if (pl.ksplit <= 1) return MOE_OK;
  const long rows = (long)grouped_rows(p);
  const dim3 grid((unsigned)rows, (unsigned)((f.out_cols / 4 + 255) / 256));
  splitk_reduce_kernel<<<grid, 256, 0, st>>>(f.part, pl.ksplit, rows, f.out_cols, masked_m, offsets, pl.nslots,
                                             p.layout == MOE_LAYOUT_MASKED, p.M_max,
                                             static_cast<__nv_bfloat16*>(f.out));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Clusters of two that the device keeps resident at once for the SM-pair kernel (its shared
// memory allows one CTA per SM), queried once per device and instantiation.
template <bool F8, int MODE>
int pair_clusters(size_t smem) {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && n[dev] > 0) return n[dev];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * (device_info().sm_count / 2));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int c = 0;
  if (cudaOccupancyMaxActiveClusters(&c, grouped_gemm_tc_kernel<F8, MODE, true, true>, &cfg) != cudaSuccess ||
      c <= 0)
    return 0;
  c = std::min(c, device_info().sm_count / 2);
  if (dev < 64) n[dev] = c;
  return c;
}

template <bool F8, int MODE, bool TM, bool PAIR = false>
int launch_tc(const moe_problem& p, const Plan& pl, const void* act, const float* act_scales, const void* w,
              const float* w_scales, const int32_t* masked_m, const int32_t* offsets, void* out, float* out_scales,
              int32_t* err, void* ws, cudaStream_t st, const CombineArgs* comb) {
  auto kern = grouped_gemm_tc_kernel<F8, MODE, TM, PAIR>;
  int r = prepare_kernel<F8, MODE, TM, PAIR>();
  if (r) return r;
  CUtensorMap tA, tB[4];
  r = make_maps(p, MODE, act, w, tA, tB);
  if (r) return r;
  TcParams prm = make_params(p, pl, masked_m, offsets, err);
  prm.stats = static_cast<int*>(ws);
  prm.ph[0] = make_phase(p, MODE, pl, act_scales, w_scales, out, out_scales,
                         reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + STATS_BYTES));
  prm.ph[1] = prm.ph[0];
  if constexpr (PAIR) {
    const int nc = pair_clusters<F8, MODE>(pl.smem);
    if (nc <= 0) return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * nc);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tA, tB[0], tB[1], tB[2], tB[3], tA, tB[0], tB[1], tB[2], tB[3], prm) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    kern<<<device_info().sm_count, NUM_THREADS, pl.smem, st>>>(tA, tB[0], tB[1], tB[2], tB[3], tA, tB[0], tB[1],
                                                               tB[2], tB[3], prm);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return launch_reduce(p, pl, prm.ph[0], masked_m, offsets, st, comb);
}

// Gate/up and down in one cooperative launch: every CTA works through the gate/up units and
// then the down units; a down unit waits (bounded) until all gate/up units of its slot have
// written their rows of h, so the down GEMM starts while the last gate/up units finish.
template <bool F8, bool TM>
int launch_ffn(const moe_problem& p, const Plan& pl0, const Plan& pl1, const void* xg, const float* xg_scales,
               const void* w13, const float* w13_scales, const void* w2, const float* w2_scales,
               const int32_t* masked_m, const int32_t* offsets, void* hg, float* hg_scales, void* yg, int32_t* err,
               void* ws, cudaStream_t st, const CombineArgs* comb) {
  auto kern = grouped_gemm_tc_kernel<F8, MODE_FFN, TM>;
  int r = prepare_kernel<F8, MODE_FFN, TM>();
  if (r) return r;
  CUtensorMap tA, tB[4], tA2, tC[4];
  if ((r = make_maps(p, MODE_SWIGLU, xg, w13, tA, tB))) return r;
  if ((r = make_maps(p, MODE_DOWN, hg, w2, tA2, tC))) return r;
  TcParams prm = make_params(p, pl0, masked_m, offsets, err);
  prm.nphase = 2;
  prm.stats = static_cast<int*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + STATS_BYTES);
  prm.ph[0] = make_phase(p, MODE_SWIGLU, pl0, xg_scales, w13_scales, hg, hg_scales, nullptr);
  prm.ph[1] = make_phase(p, MODE_DOWN, pl1, hg_scales, w2_scales, yg, nullptr, part);
  prm.ready = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + STATS_BYTES + align_up(pl1.part_bytes, 256));
  if (cudaMemsetAsync(prm.ready, 0, sizeof(int) * pl0.nslots, st) != cudaSuccess) return MOE_ERR_CUDA;
  // all CTAs must be resident at once (a down unit may wait for another CTA's gate/up unit)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(device_info().sm_count);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = pl0.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tA, tB[0], tB[1], tB[2], tB[3], tA2, tC[0], tC[1], tC[2], tC[3], prm) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_reduce(p, pl1, prm.ph[1], masked_m, offsets, st, comb);
}

// ---------------------------------------------------------------------------
// fp32 path on the CUDA cores (small fp32 problems; the tensor-core path
// covers bf16 and e4m3).  One warp per output column, lanes across K.
// ---------------------------------------------------------------------------

template <int MODE>
__global__ void __launch_bounds__(256) grouped_gemm_f32_kernel(const float* __restrict__ act,
                                                               const float* __restrict__ w,
                                                               const int32_t* __restrict__ masked_m,
                                                               const int32_t* __restrict__ offsets, float* __restrict__ out,
                                                               int nslots, int masked, int M_max, long rows_total,
                                                               int K, int NA, int out_cols, int I) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;  // output column
  if (n >= out_cols) return;
  const long r0 = (long)blockIdx.y * 8;
  for (long R = r0; R < r0 + 8 && R < rows_total; ++R) {
    int s;
    if (masked) {
      s = (int)(R / M_max);
      const int r = (int)(R - (long)s * M_max);
      if (r >= min(masked_m[s], M_max)) continue;  // padding row: nothing to compute
    } else {
      if (R >= offsets[nslots]) continue;
      int lo = 0, hi = nslots;  // offsets[lo] <= R < offsets[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= R)
          lo = mid;
        else
          hi = mid;
      }
      s = lo;
    }
    const float* x = act + R * K;
    const float* w0 = w + ((size_t)s * NA + n) * K;
    float a0 = 0.0f, a1 = 0.0f;
    if (MODE == MODE_SWIGLU) {
      const float* w1 = w0 + (size_t)I * K;
      for (int k = lane; k < K; k += 32) {
        a0 = fmaf(w0[k], x[k], a0);
        a1 = fmaf(w1[k], x[k], a1);
      }
    } else {
      for (int k = lane; k < K; k += 32) a0 = fmaf(w0[k], x[k], a0);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, off);
      a1 += __shfl_xor_sync(0xffffffffu, a1, off);
    }
    if (lane == 0) out[R * out_cols + n] = (MODE == MODE_SWIGLU) ? a0 / (1.0f + expf(-a0)) * a1 : a0;
  }
}

}  // namespace

int gemm_tile_rows(const moe_problem& p, int mode) {
  if (p.wt == MOE_F32) return 0;
  return use_pairs(p, mode, 1) ? 2 * BN : fp8_acts(p) ? DEC_CH : BN;
}

size_t gemm_workspace_bytes(const moe_problem& p) {
  if (p.wt == MOE_F32) return 0;
  // Split-K state depends on the SM count; size it for the largest plausible GPU (up to 256 SMs).
  size_t best = 0;
  for (int mode = 0; mode < 2; ++mode) {
    for (int sms : {132, 148, 152, 160, 170, 188, 256}) {
      const Plan pl = make_plan(p, mode, sms, 232448);
      best = std::max(best, pl.part_bytes);
    }
  }
  // issue counters first, then the split-K partial sums, then (two-phase launch) one counter per slot
  return STATS_BYTES + align_up(best, 256) + align_up(sizeof(int) * (size_t)(p.P + p.has_shared), 256);
}

int launch_gemm(const moe_problem& p, int mode, const void* act, const float* act_scales, const void* w,
                const float* w_scales, const int32_t* masked_m, const int32_t* offsets, void* out, float* out_scales,
                int32_t* err, void* ws, cudaStream_t st, const CombineArgs* comb) {
  const int nslots = p.P + p.has_shared;
  if (p.wt == MOE_F32) {
    const int K = (mode == MODE_SWIGLU) ? p.H : p.I;
    const int NA = (mode == MODE_SWIGLU) ? 2 * p.I : p.H;
    const int out_cols = (mode == MODE_SWIGLU) ? p.I : p.H;
    const long rows = (long)grouped_rows(p);
    if (rows == 0) return MOE_OK;
    const dim3 grid((out_cols + 7) / 8, (unsigned)((rows + 7) / 8));
    if (mode == MODE_SWIGLU)
      grouped_gemm_f32_kernel<MODE_SWIGLU><<<grid, 256, 0, st>>>(
          (const float*)act, (const float*)w, masked_m, offsets, (float*)out, nslots,
          p.layout == MOE_LAYOUT_MASKED, p.M_max, rows, K, NA, out_cols, p.I);
    else
      grouped_gemm_f32_kernel<MODE_DOWN><<<grid, 256, 0, st>>>(
          (const float*)act, (const float*)w, masked_m, offsets, (float*)out, nslots,
          p.layout == MOE_LAYOUT_MASKED, p.M_max, rows, K, NA, out_cols, p.I);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return comb ? launch_combine(p, out, comb->row_of, comb->w, comb->out, st) : MOE_OK;
  }
  const DeviceInfo& di = device_info();
  const Plan pl = make_plan(p, mode, di.sm_count, di.max_smem_optin);
  if (pl.stages == 0) return MOE_ERR_UNSUPPORTED;
  const bool f8 = fp8_acts(p);
#define MOE_LAUNCH(F8_, MODE_, TM_)                                                                              \
  return launch_tc<F8_, MODE_, TM_>(p, pl, act, act_scales, w, w_scales, masked_m, offsets, out, out_scales, err, \
                                    ws, st, comb)
  if (f8) {
    if (pl.pair) {
      if (mode == MODE_SWIGLU)
        return launch_tc<true, MODE_SWIGLU, true, true>(p, pl, act, act_scales, w, w_scales, masked_m, offsets, out,
                                                        out_scales, err, ws, st, comb);
      return launch_tc<true, MODE_DOWN, true, true>(p, pl, act, act_scales, w, w_scales, masked_m, offsets, out,
                                                    out_scales, err, ws, st, comb);
    }
    if (mode == MODE_SWIGLU) MOE_LAUNCH(true, MODE_SWIGLU, true);
    MOE_LAUNCH(true, MODE_DOWN, true);
  }
  if (mode == MODE_SWIGLU) {
    if (pl.tm) MOE_LAUNCH(false, MODE_SWIGLU, true);
    MOE_LAUNCH(false, MODE_SWIGLU, false);
  }
  if (pl.tm) MOE_LAUNCH(false, MODE_DOWN, true);
  MOE_LAUNCH(false, MODE_DOWN, false);
#undef MOE_LAUNCH
}

int launch_grouped_ffn(const moe_problem& p, const void* xg, const float* xg_scales, const void* w13,
                       const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                       const int32_t* offsets, void* hg, float* hg_scales, void* yg, int32_t* err, void* ws,
                       cudaStream_t st, const CombineArgs* comb) {
  if (p.wt == MOE_F32) {  // CUDA-core path: the two GEMMs one after the other
    int r = launch_gemm(p, MODE_SWIGLU, xg, nullptr, w13, nullptr, masked_m, offsets, hg, nullptr, err, ws, st);
    if (r) return r;
    return launch_gemm(p, MODE_DOWN, hg, nullptr, w2, nullptr, masked_m, offsets, yg, nullptr, err, ws, st, comb);
  }
  const DeviceInfo& di = device_info();
  const Plan pl0 = make_plan(p, MODE_SWIGLU, di.sm_count, di.max_smem_optin, 2);
  const Plan pl1 = make_plan(p, MODE_DOWN, di.sm_count, di.max_smem_optin, 2);
  if (pl0.stages == 0 || pl1.stages != pl0.stages || pl1.smem != pl0.smem) return MOE_ERR_UNSUPPORTED;
  if (fp8_acts(p))
    return launch_ffn<true, true>(p, pl0, pl1, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, hg,
                                  hg_scales, yg, err, ws, st, comb);
  if (pl0.tm)
    return launch_ffn<false, true>(p, pl0, pl1, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets,
                                   hg, hg_scales, yg, err, ws, st, comb);
  return launch_ffn<false, false>(p, pl0, pl1, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, hg,
                                  hg_scales, yg, err, ws, st, comb);
}

}  // namespace moe

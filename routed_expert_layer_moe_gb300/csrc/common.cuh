// Internal helpers of the MoE layer library: launch plumbing, and inline-PTX
// wrappers for mbarriers, TMA bulk-tensor copies and the tcgen05 tensor-core
// instructions of sm_100-family GPUs (GB300 = sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Host-side launch helpers (defined in api.cu)
// ---------------------------------------------------------------------------

struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
};
const DeviceInfo& device_info();  // of the current device, cached

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry point.
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint64_t inner, uint64_t outer,
                           uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, const void* base);

// The combine's arguments, when a GEMM call also runs step 5 (fused into its split-K reduction,
// or after it).
struct CombineArgs {
  const int32_t* row_of;
  const float* w;
  void* out;
};

// Per-call launchers (each returns a moe_status).
int launch_route(const moe_problem& p, const float* logits, int32_t* ids, float* w, cudaStream_t st);
int launch_route_grouped(const moe_problem& p, const float* logits, const float* bias, int n_group, int topk_group,
                         int renorm, float scale, int32_t* ids, float* w, cudaStream_t st);
int launch_permute(const moe_problem& p, const int32_t* ids, const void* x, const int32_t* p2l, int32_t* masked_m,
                   int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg, float* xg_scales, int32_t* err,
                   void* ws, cudaStream_t st);
size_t permute_workspace_bytes(const moe_problem& p);
// Route + dispatch in one launch (batches of at most 256 records, no replica map, E <= 256).
bool route_permute_one_launch(const moe_problem& p, const int32_t* p2l);
int launch_route_permute_small(const moe_problem& p, const float* logits, const void* x, int32_t* ids, float* w,
                               int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                               float* xg_scales, int32_t* err, cudaStream_t st);
int launch_gemm(const moe_problem& p, int mode, const void* a_act, const float* a_act_scales, const void* w,
                const float* w_scales, const int32_t* masked_m, const int32_t* offsets, void* out,
                float* out_scales, int32_t* err, void* ws, cudaStream_t st, const CombineArgs* comb = nullptr);
size_t gemm_workspace_bytes(const moe_problem& p);
int gemm_tile_rows(const moe_problem& p, int mode);  // token rows of one MMA tile (0: CUDA-core GEMM)
int launch_grouped_ffn(const moe_problem& p, const void* xg, const float* xg_scales, const void* w13,
                       const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                       const int32_t* offsets, void* hg, float* hg_scales, void* yg, int32_t* err, void* ws,
                       cudaStream_t st, const CombineArgs* comb = nullptr);
int launch_eplb_record(const moe_problem& p, const int32_t* masked_m, int64_t pass, int window, int32_t* load_window,
                       cudaStream_t st);
int launch_eplb_rebalance(const moe_problem& p, const int32_t* load_window, int window, const int32_t* p2l,
                          int64_t* logical_load, int32_t* new_p2l, int32_t* err, cudaStream_t st);
int launch_bounded_wait_selftest(long long cycles, int32_t* err, cudaStream_t st);
int launch_combine(const moe_problem& p, const void* yg, const int32_t* row_of, const float* w, void* out,
                   cudaStream_t st);

enum { MODE_SWIGLU = 0, MODE_DOWN = 1 };

inline int64_t grouped_rows(const moe_problem& p) {
  return p.layout == MOE_LAYOUT_MASKED ? (int64_t)(p.P + p.has_shared) * p.M_max
                                       : (int64_t)p.T * p.K + (int64_t)p.has_shared * p.T;
}

// Grouped activations (Xg, Hg) are e4m3 with 1x128 scales for FP8 and FP4 experts.
inline bool fp8_acts(const moe_problem& p) { return p.wt == MOE_E4M3 || p.wt == MOE_E2M1; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ----

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// CL: acquire at cluster scope (the barrier also takes arrivals from the peer CTA of a pair).
template <bool CL = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CL) {
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort is set by another role of the CTA, or after
// `timeout_cycles` SM clock cycles, in which case it sets *abort itself.
// The clock is read only every 64 polls, so a wait that ends quickly costs
// nothing beyond the polls themselves.
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          long long timeout_cycles) {
  if (mbar_try_wait<CL>(bar, parity)) return true;
  long long t0 = 0;
  uint32_t n = 0;
  while (!mbar_try_wait<CL>(bar, parity)) {
    if ((++n & 63u) == 0) {
      if (*abort) return false;
      const long long now = clock64();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_cycles) {
        *abort = 1;
        return false;
      }
    }
  }
  return true;
}

// ---- thread-block clusters (a CTA pair sharing one tcgen05 MMA) ----

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Shared::cluster address of the variable at `bar` in the CTA of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* bar, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(bar)), "r"(rank));
  return r;
}

// One arrival on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
// The waiter orders only tensor-memory accesses after it (tcgen05 fences on both sides), so the
// default CTA-scope release is enough.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of every CTA of the cluster (used once, after the mbarriers are initialised,
// while all CTAs of the cluster are known to be running).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}

// ---- packed fp32 arithmetic ----

// ---- wide stores ----

// One 32-byte store (a full L2 sector); dst must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, uint4 a, uint4 b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// ---- flags between CTAs ----

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's later async-proxy (TMA) reads of global memory after what it has acquired.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- cp.async (asynchronous global -> shared copies) ----

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued before has landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- TMA ----

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Pair form: the copy lands in this CTA's shared memory and its bytes are counted on the
// mbarrier at `bar_cluster` (a shared::cluster address, here the leader CTA's barrier).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint "
      "[%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 2-D tiled bulk-tensor load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Same, with an L2 cache-policy hint (a createpolicy value).
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory) ----

// PAIR: .cta_group::2, performed together by one warp of each CTA of the pair.
template <bool PAIR = false>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

template <bool PAIR = false>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (PAIR)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <bool PAIR = false>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction, issued by one thread.
template <bool F8>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  if constexpr (F8) {
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Pair form (issued by the leader CTA of a pair): D[256 rows, two TMEMs] (+)= A * B^T, A's rows
// 0-127 and B's rows 0..N/2-1 in the leader's shared memory, the other halves at the same
// offsets in the peer's; D rows 0-127 land in the leader's tensor memory, 128-255 in the peer's.
__device__ __forceinline__ void tc_mma_pair_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask` when every pair
// (cta_group::2) tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Two 32-lane x 32-column fp32 loads from tensor memory, waited for in the same asm statement.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[32 + i]);
  }
}

// One 16-lane load of 8 groups of 8 columns (tcgen05.ld 16x256b.x8) from the 16 lanes at ta, not
// waited for (tmem_wait_ld32 on r): thread t gets lanes t/4 and t/4 + 8 of them, columns 2 (t % 4)
// and 2 (t % 4) + 1 of each group, as r[4g] = (lane t/4, column 8g + 2 (t % 4)), r[4g + 1] = the
// next column, r[4g + 2], r[4g + 3] = the same columns of lane t/4 + 8 (checked on a GB300 by
// storing lane * 1000 + column with 32x32b stores and reading it back).
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t ta, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta)
      : "memory");
}

// Wait for this thread's tensor-memory loads; r is the array the last load wrote.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;\n"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// Two 32-lane x 32-column fp32 loads from tensor memory (32 columns at ta, 32 at tb), waited for
// in the same statement, as 32 packed pairs (r[i] = columns 2i, 2i+1 of ta for i < 16, of tb for
// i >= 16; the lower column in the low word): operands of fma.rn.f32x2 that need no moves.
__device__ __forceinline__ void tmem_ld32x2_pairs(uint32_t ta, uint32_t tb, uint64_t (&r)[32]) {
  asm volatile(
      "{\n"
      "  .reg .b32 t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31, t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63;\n"
      "  tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%32];\n"
      "  tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%33];\n"
      "  tcgen05.wait::ld.sync.aligned;\n"
      "  mov.b64 %0, {t0, t1};\n"
      "  mov.b64 %1, {t2, t3};\n"
      "  mov.b64 %2, {t4, t5};\n"
      "  mov.b64 %3, {t6, t7};\n"
      "  mov.b64 %4, {t8, t9};\n"
      "  mov.b64 %5, {t10, t11};\n"
      "  mov.b64 %6, {t12, t13};\n"
      "  mov.b64 %7, {t14, t15};\n"
      "  mov.b64 %8, {t16, t17};\n"
      "  mov.b64 %9, {t18, t19};\n"
      "  mov.b64 %10, {t20, t21};\n"
      "  mov.b64 %11, {t22, t23};\n"
      "  mov.b64 %12, {t24, t25};\n"
      "  mov.b64 %13, {t26, t27};\n"
      "  mov.b64 %14, {t28, t29};\n"
      "  mov.b64 %15, {t30, t31};\n"
      "  mov.b64 %16, {t32, t33};\n"
      "  mov.b64 %17, {t34, t35};\n"
      "  mov.b64 %18, {t36, t37};\n"
      "  mov.b64 %19, {t38, t39};\n"
      "  mov.b64 %20, {t40, t41};\n"
      "  mov.b64 %21, {t42, t43};\n"
      "  mov.b64 %22, {t44, t45};\n"
      "  mov.b64 %23, {t46, t47};\n"
      "  mov.b64 %24, {t48, t49};\n"
      "  mov.b64 %25, {t50, t51};\n"
      "  mov.b64 %26, {t52, t53};\n"
      "  mov.b64 %27, {t54, t55};\n"
      "  mov.b64 %28, {t56, t57};\n"
      "  mov.b64 %29, {t58, t59};\n"
      "  mov.b64 %30, {t60, t61};\n"
      "  mov.b64 %31, {t62, t63};\n"
      "}\n"
      : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15]), "=l"(r[16]), "=l"(r[17]), "=l"(r[18]), "=l"(r[19]), "=l"(r[20]), "=l"(r[21]), "=l"(r[22]), "=l"(r[23]), "=l"(r[24]), "=l"(r[25]), "=l"(r[26]), "=l"(r[27]), "=l"(r[28]), "=l"(r[29]), "=l"(r[30]), "=l"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

// a[i] += r[i] * (s, s) for n packed pairs (two fmaf roundings each).
template <int N>
__device__ __forceinline__ void fma2_pairs(uint64_t* a, const uint64_t* r, uint64_t s2) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a[i]) : "l"(r[i]), "l"(s2));
}

// (s, s) as one packed pair.
__device__ __forceinline__ uint64_t pair_of(float s) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address (16-byte units)
  d |= (uint64_t)1 << 16;                    // leading byte offset: unused for swizzled K-major
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version of the tcgen05 family
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulate, A and B K-major, M x N.
template <bool F8>
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N) {
  return (1u << 4)                        // D format: f32
         | ((F8 ? 0u : 1u) << 7)          // A format: e4m3 (kind::f8f6f4) or bf16 (kind::f16)
         | ((F8 ? 0u : 1u) << 10)         // B format
         | ((uint32_t)(N >> 3) << 17)     // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// SiLU with the fast division: for g -> -inf the denominator overflows to inf and
// the quotient to 0, which is the limit of g * sigmoid(g).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace moe

/*
 * moe.h -- C ABI of the single-GPU forward pass of one routed
 * Mixture-of-Experts layer (GB300, sm_103a).
 *
 * The forward pass is five calls, made in this order on one stream:
 *
 *   moe_route_topk          softmax top-K routing of the router logits
 *   moe_permute             counts, offsets, row maps; dispatch of the
 *                           activations into the expert-grouped buffer
 *   moe_grouped_swiglu_gemm per-expert gate/up GEMM with SiLU(gate) * up
 *   moe_grouped_down_gemm   per-expert down GEMM
 *   moe_combine             weighted sum of each token's expert outputs
 *
 * Sources, by page title and section:
 *   "MoE inference and expert parallelism" (blog.vllbc.top): the routing
 *     section and Table 3-1 (softmax top-K with renormalisation, SwiGLU experts
 *     with W1/W3 = gate/up and W2 = down, moe_sum, DeepSeek-V3 shared expert,
 *     Eq. 12) and the forward-pass section (fused_topk -> moe_align_block_size
 *     -> W1/W3 GEMM -> activation -> W2 GEMM -> moe_sum).
 *   "Inference INFRA methodology (5): MoE inference -- Batch, DeepEP, DeepGEMM
 *     and load balancing" (yfxerp.com): section "DeepGEMM" (static
 *     [E_loc, M_max, K] buffer with a device-resident masked_m read at run
 *     time, no MMA for tiles that hold only padding, FP8 with the 128-wide K
 *     promotion to FP32, contiguous layout for prefill).
 *   "vLLM EPLB" (pnsm.cn): section 1.2 (physical_to_logical_map,
 *     logical_to_physical_map, logical_replica_count).
 *   "MoonEP: dynamic redundant experts" (wineandchord.com): sections "Why
 *     dynamic routing is hard" (counts sum to the routed records) and
 *     "Zero-copy and static buffer" (offsets / cu_seqlens, padding described
 *     by the plan).
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers unless a comment says otherwise.
 *     The caller allocates and owns every buffer, including the workspace.
 *     The library never allocates, frees or synchronises; every call only
 *     enqueues kernels (and memsets) on `stream`, so a sequence of calls can be
 *     captured in a CUDA graph once the first call on the device has been made
 *     outside of capture (it caches device attributes).
 *   - Return status: checked on the host from the arguments and from the
 *     launch; nothing is enqueued when a call returns MOE_ERR_INVALID or
 *     MOE_ERR_UNSUPPORTED.  Data-dependent problems found on the device set
 *     bits of the caller's int32 `err_flag` (MOE_FLAG_*); tokens are never
 *     dropped silently.
 *   - Layouts are row-major.  Counts: T tokens, H hidden, I expert
 *     intermediate, E logical routed experts, K experts per token, P physical
 *     slots (P == E without a replica map), S = has_shared (0/1).  The shared
 *     expert, when present, is slot P.
 *   - Dtypes: bf16 is IEEE binary32's upper half, e4m3 is OCP FP8 E4M3,
 *     e2m1 is OCP FP4 E2M1 (weights only; the FP4 experts of "Inference INFRA
 *     methodology (5)", shape-evolution table, DS-V4-Pro row).
 *     Supported combinations (act / wt / out): F32/F32/F32, BF16/BF16/BF16,
 *     BF16/E4M3/BF16, BF16/E2M1/BF16.  `wt` is the type of the expert
 *     weights; the grouped activations Xg and Hg are of type wt, except that
 *     they are E4M3 when wt is E2M1.  Yg is F32 when wt is F32, else BF16.
 *   - e4m3 and e2m1 scales are fp32: weights one per 128x128 block
 *     ([slots][N/128][K/128]), grouped activations one per 1x128 group
 *     ([rows][cols/128]).  Quantised value = code * scale.
 *   - e2m1 weights are packed two codes per byte along the reduced
 *     dimension: byte j of a row holds column 2j in bits 0-3 and column 2j+1
 *     in bits 4-7 (a row of K codes is K/2 bytes).  Their base address must
 *     be 32-byte aligned.
 *   - Weights are stored transposed with the reduced dimension contiguous:
 *     W13 [P+S][2I][H] (rows 0..I-1 = gate W1^T, rows I..2I-1 = up W3^T),
 *     W2 [P+S][H][I].  Slot s holds the weights of the logical expert
 *     physical_to_logical[s] (a replica is a copy).
 *   - Grouped buffers have `rows` rows: (P+S)*M_max (masked layout, row of
 *     slot s rank r = s*M_max + r) or T*K + S*T (contiguous layout, row =
 *     offsets[s] + r).  Rows of a slot hold its tokens in ascending token
 *     order.  Rows at or past masked_m[s] are padding: no call writes them.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,     /* a null pointer, a size out of range, an inconsistent problem */
  MOE_ERR_UNSUPPORTED = -2, /* a valid problem this build does not run (dtype combination, alignment) */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime error at launch */
  MOE_ERR_WORKSPACE = -4    /* workspace smaller than moe_workspace_bytes() */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2, MOE_E2M1 = 3 } moe_dtype;

typedef enum moe_layout { MOE_LAYOUT_MASKED = 0, MOE_LAYOUT_CONTIG = 1 } moe_layout;

/* Bits of the device error flag. */
#define MOE_FLAG_OVERFLOW 1   /* a slot received more than M_max rows (masked layout); extra rows not written, their row_of is -1 */
/* an expert id outside [0,E), or one token naming an expert twice (the record
 * with the larger k is the one not placed) */
#define MOE_FLAG_BAD_EXPERT 2
/* a physical_to_logical entry outside [0,E), or a routed expert held by no
 * slot or by more than P-E+1 slots (its records are not placed) */
#define MOE_FLAG_BAD_MAP 4
#define MOE_FLAG_TIMEOUT 8    /* a pipeline wait inside a GEMM kernel gave up; its outputs are incomplete */

/* CUDA stream, ABI-compatible with cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

typedef struct moe_problem {
  int32_t T;          /* tokens, >= 0 */
  int32_t H;          /* hidden size */
  int32_t I;          /* expert intermediate size */
  int32_t E;          /* logical routed experts, 1..1024 */
  int32_t K;          /* experts per token, 1..min(E, 32) */
  int32_t P;          /* physical slots, >= E (== E without a replica map) */
  int32_t M_max;      /* rows per slot of the masked layout; >= T when has_shared; unused for contiguous */
  int32_t has_shared; /* 1 = one always-on shared expert in slot P, weight 1 */
  int32_t act;        /* moe_dtype of x */
  int32_t wt;         /* moe_dtype of the expert weights, Xg and Hg */
  int32_t out;        /* moe_dtype of the layer output */
  int32_t layout;     /* moe_layout of the grouped buffers */
} moe_problem;

/* Library version, (major << 16) | minor. */
int32_t moe_version(void);

/* A static string naming a status code. */
const char* moe_status_string(int32_t status);

/* Rows of the grouped buffers for this problem (see the conventions above). */
int64_t moe_grouped_rows(const moe_problem* p);

/* Workspace bytes one call sequence needs (the maximum over all calls).
 * One workspace may serve every call of a layer as long as the calls are
 * ordered on one stream.  Returns 0 for an invalid problem. */
size_t moe_workspace_bytes(const moe_problem* p);

/* Issue counters ("Inference INFRA methodology (5)", section "DeepGEMM": a tile
 * whose first row is at or past masked_m issues no MMA).  After a tensor-core
 * moe_grouped_swiglu_gemm, moe_grouped_down_gemm or moe_grouped_ffn call, the
 * first MOE_STATS_BYTES of the workspace hold int32 counters
 * [2 phases][MOE_STATS_CTAS][2]: for each CTA, the units it issued (token
 * chunk x weight-tile pair x K split) and the token tiles among them (one per
 * slot and chunk of at most BM rows, BM = moe_gemm_tile_rows; a GEMM that runs
 * on SM pairs counts each pair's units once, in its first CTA).  Summed over
 * CTAs, the token tiles of a GEMM equal the sum over slots of
 * ceil(masked_m[s] / BM).  Phase 1 is the down GEMM of moe_grouped_ffn and
 * zero otherwise.  The counters stay valid until the next call that uses the
 * workspace. */
#define MOE_STATS_CTAS 256
#define MOE_STATS_BYTES (2 * MOE_STATS_CTAS * 2 * 4)

/* Token rows BM of one tile of the tensor-core GEMM of step 3 (step = 3) or
 * step 4 (step = 4) for this problem ("Inference INFRA methodology (5)",
 * section "DeepGEMM": the tile height BM of the padding-waste ratio
 * ceil(M_e / BM) * BM / M_e).  For bf16 experts 128.  For FP8 / FP4 experts
 * 256 with at least 128 rows per slot on average (and, for step 4, H a multiple
 * of 256): those GEMMs run on pairs of SMs (thread-block clusters of two), each
 * SM holding 128 of the tile's token rows and one of its two 128-row weight
 * tiles, with one cta_group::2 MMA over both; else 64: one CTA per SM with
 * M = 64 MMAs.  moe_grouped_ffn runs on single CTAs: 64-row tiles for FP8 /
 * FP4 experts, 128 for bf16.
 * 0 for an invalid problem or one whose GEMMs run on the CUDA cores (F32).
 * Host only; touches no GPU. */
int32_t moe_gemm_tile_rows(const moe_problem* p, int32_t step);

/* Check a problem without touching the GPU: MOE_OK, MOE_ERR_INVALID or
 * MOE_ERR_UNSUPPORTED. */
moe_status moe_check_problem(const moe_problem* p);

/* Step 1 (routing; "MoE inference and expert parallelism", routing section,
 * Table 3-1).  For each token t: the K largest of the E logits, in descending
 * order, ties to the lower expert index; weights
 * w[t,k] = exp(l_k - l_max) / sum_j exp(l_j - l_max) over the chosen K
 * (= softmax over all E renormalised over the K; fp32).
 *   logits [T][E] fp32 (device, read), ids [T][K] int32 and w [T][K] fp32
 *   (device, written).  One warp per token. */
moe_status moe_route_topk(const moe_problem* p, const float* logits, int32_t* ids, float* w, moe_stream_t stream);

/* Step 1, DeepSeek-V3 variant ("MoE inference and expert parallelism", routing
 * section, Table 3-1: sigmoid scoring with e_score_correction_bias, grouped
 * top-k; the bias decides which experts are chosen, the weights use the
 * unbiased scores).  Per token: s_e = sigmoid(l_e), key_e = s_e + bias_e;
 * the E experts form n_group contiguous groups of E/n_group, a group scored by
 * its largest key; the topk_group best groups are kept, then the K largest
 * keys among their experts (all ties to the lower index; keys compared in
 * fp64).  w[t,k] = s_{e_k} (divided by the sum over the K when renormalize),
 * times scale.
 *   logits [T][E] fp32, bias [E] fp32 or NULL (device, read); ids [T][K] int32,
 *   w [T][K] fp32 (device, written).  Requires 1 <= n_group <= 32, E % n_group
 *   == 0, 1 <= topk_group <= n_group, K <= topk_group * E / n_group. */
moe_status moe_route_grouped_topk(const moe_problem* p, const float* logits, const float* bias, int32_t n_group,
                                  int32_t topk_group, int32_t renormalize, float scale, int32_t* ids, float* w,
                                  moe_stream_t stream);

/* Step 2 (dispatch; "Inference INFRA methodology (5)", section "DeepGEMM";
 * "vLLM EPLB", section 1.2; "MoonEP", sections "Why dynamic routing is hard"
 * and "Zero-copy and static buffer").
 *   ids [T][K] int32: logical expert ids (from moe_route_topk).
 *   x [T][H]: activations, dtype p->act.
 *   phys_to_log [P] int32 or NULL: physical_to_logical_map.  With a map, a
 *     record (t, k) of logical expert e goes to the (t mod c)-th slot holding
 *     e, slots taken in ascending index, c = logical_replica_count[e]
 *     (round-robin by token index).  Without one, slot = e and P must be E.
 * Writes:
 *   masked_m [P+S] int32: rows per slot (the shared slot holds T).
 *   offsets [P+S+1] int32: exclusive prefix sum of masked_m.
 *   row_of [T][K+S] int32: grouped row of record (t,k); column K is the
 *     shared expert's row.  -1 for a record that was not placed (see err_flag).
 *   src_of [rows] int32: token of each written row (padding rows untouched).
 *   xg [rows][H], dtype p->wt (e4m3 for E2M1 weights): x[t] copied to its
 *     rows; for e4m3 each row is
 *     quantised per 1x128 group: s = amax/448 (fp32 IEEE division, s = 1 for an
 *     all-zero group), code = e4m3(x / s) nearest-even, saturating.
 *   xg_scales [rows][H/128] fp32: the group scales (e4m3 only, else NULL).
 *   err_flag: device int32, MOE_FLAG_* bits are OR-ed in (never cleared).
 *   workspace: device scratch of moe_workspace_bytes(p) bytes. */
moe_status moe_permute(const moe_problem* p, const int32_t* ids, const void* x, const int32_t* phys_to_log,
                       int32_t* masked_m, int32_t* offsets, int32_t* row_of, int32_t* src_of, void* xg,
                       float* xg_scales, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/* moe_permute for callers that cannot allocate device memory.  The pages
 * describe no such variant; it is an addition of this library.
 * Some callers cannot call cudaMalloc where they run the layer: an inference
 * engine plugin whose enqueue step must not allocate, code running while its
 * stream is being captured into a CUDA graph, a framework whose device memory
 * all belongs to its own pool.  This call takes the same arguments and writes
 * the same outputs as moe_permute, but needs no workspace: its scratch is a
 * fixed 4 MiB array inside the library, which every GPU that loads the library
 * keeps until the process exits.
 *   - A problem whose scratch exceeds 4 MiB is rejected with MOE_ERR_WORKSPACE
 *     before anything is enqueued (the scratch is (4*P*ceil(T/32) + 4) +
 *     4*P*ceil(T/32) + 4*T*K + 4*P + 4*E + 4*E bytes, each term rounded up
 *     to 256; the prefill workload T=8192, E=P=512, K=10 needs about 1.3 MiB).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it; make that first call outside of any
 *     stream capture.  The kept address is valid for the life of the device's
 *     primary context: do not call this entry point again after
 *     cudaDeviceReset on that device.
 *   - All calls share the one array, which keeps the previous call's contents
 *     (the call clears what must start at zero itself).  Calls that overlap on
 *     the GPU -- on different streams, or from different threads, without
 *     ordering between them -- race on it and give wrong results. */
moe_status moe_permute_no_workspace(const moe_problem* p, const int32_t* ids, const void* x,
                                    const int32_t* phys_to_log, int32_t* masked_m, int32_t* offsets,
                                    int32_t* row_of, int32_t* src_of, void* xg, float* xg_scales, int32_t* err_flag,
                                    moe_stream_t stream);

/* Step 3 (expert gate/up; "MoE inference and expert parallelism", routing
 * section: SwiGLU with W1 = gate, W3 = up; "Inference INFRA methodology (5)",
 * section "DeepGEMM": masked_m read on the device, no MMA for padding tiles,
 * FP8 accumulated in FP32 once per 128-wide K block).
 * For every slot s and row r < masked_m[s] (row index per the layout):
 *   g = W1[s] . xg[row], u = W3[s] . xg[row], h = SiLU(g) * u
 *   hg[row][0..I) = h, stored as p->wt (e4m3 for E2M1 weights; e4m3: 1x128
 *   groups as in moe_permute, scales in hg_scales [rows][I/128]; bf16:
 *   nearest-even; f32: as is).
 *   xg_scales / w13_scales / hg_scales: e4m3 / e2m1 weights only, else NULL.
 *   masked_m [P+S], offsets [P+S+1]: as written by moe_permute (device).
 * bf16 / e4m3 / e2m1 run on the tcgen05 tensor cores and need H, I multiples
 * of 128 (e2m1: e4m3 x e2m1 products, kind::f8f6f4). */
moe_status moe_grouped_swiglu_gemm(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                                   const float* w13_scales, const int32_t* masked_m, const int32_t* offsets,
                                   void* hg, float* hg_scales, int32_t* err_flag, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream);

/* Step 4 (expert down): yg[row][0..H) = W2[s] . hg[row] for every valid row,
 * stored as fp32 (wt = F32) or bf16.  Same skipping and promotion as step 3. */
moe_status moe_grouped_down_gemm(const moe_problem* p, const void* hg, const float* hg_scales, const void* w2,
                                 const float* w2_scales, const int32_t* masked_m, const int32_t* offsets,
                                 void* yg, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream);

/* Steps 3 and 4 in one launch (the fused path of "MoE inference and expert
 * parallelism", routing section: "fused MoE" runs the grouped gate/up, the
 * activation and the grouped down GEMM as one unit of work).  Same arguments,
 * outputs and numerics as moe_grouped_swiglu_gemm followed by
 * moe_grouped_down_gemm (hg/hg_scales are still written; yg is bit-identical
 * to the two separate calls).  On the tensor cores it is one persistent
 * cooperative launch in which a CTA moves on to down tiles as soon as every
 * gate/up tile of that slot has released its rows of h, so the down GEMM's
 * weight streaming overlaps the end of gate/up (plus the split-K reduction
 * kernel when the down GEMM is split); fp32 problems run the two CUDA-core
 * GEMMs one after the other.  All CTAs must be resident at once: the launch
 * fails (MOE_ERR_CUDA) if the device cannot co-schedule them.  workspace:
 * moe_workspace_bytes(p) bytes (it holds the per-slot ready counters, cleared
 * by this call). */
moe_status moe_grouped_ffn(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                           const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                           const int32_t* offsets, void* hg, float* hg_scales, void* yg, int32_t* err_flag,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Step 5 (combine; "MoE inference and expert parallelism", routing section:
 * moe_sum / TopKWeightAndReduce, DeepSeek-V3 Eq. 12 for the shared expert):
 *   out[t] = sum_{k<K} w[t,k] * yg[row_of[t,k]]  (+ yg[row_of[t,K]] if S),
 * summed in fp32 in k order, then rounded once to p->out.  Records with
 * row_of = -1 are skipped.  yg [rows][H] (F32 or BF16 per p->wt), row_of
 * [T][K+S], w [T][K] fp32, out [T][H] (p->out). */
moe_status moe_combine(const moe_problem* p, const void* yg, const int32_t* row_of, const float* w, void* out,
                       moe_stream_t stream);

/* Steps 1 and 2 in one call ("MoE inference and expert parallelism", routing
 * section and forward-pass section: fused_topk followed by the dispatch).
 * Same arguments, outputs and numerics as moe_route_topk followed by
 * moe_permute (ids and w are written and bit-identical to moe_route_topk's).
 * Batches of at most 256 records (T*K <= 256) without a replica map and with
 * E <= 256 run as one launch: every CTA chooses the experts of all tokens
 * (one warp per token, the router's own per-token code) and derives the layout
 * from them in shared memory; other batches run the two calls' kernels back
 * to back.  workspace: moe_workspace_bytes(p) bytes. */
moe_status moe_route_permute(const moe_problem* p, const float* logits, const void* x, const int32_t* phys_to_log,
                             int32_t* ids, float* w, int32_t* masked_m, int32_t* offsets, int32_t* row_of,
                             int32_t* src_of, void* xg, float* xg_scales, int32_t* err_flag, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream);

/* Steps 3, 4 and 5 in one call ("MoE inference and expert parallelism",
 * routing section: fused MoE runs the grouped GEMMs, the activation and
 * moe_sum as one unit of work).  Same arguments and numerics as
 * moe_grouped_swiglu_gemm, moe_grouped_down_gemm and moe_combine in that order
 * (row_of and w as written by moe_permute and the router; hg, hg_scales and
 * yg are written as by those calls; out is bit-identical to moe_combine's).
 * bf16 experts run both GEMMs in one launch (as moe_grouped_ffn); FP8 / FP4
 * experts in two.  When the down GEMM is split along K (decode-sized slots),
 * the combine runs inside the split-K reduction: each record's row is
 * reduced over the splits and enters its token's k-order sum in the same
 * kernel; otherwise the combine kernel follows the down GEMM.
 * workspace: moe_workspace_bytes(p) bytes. */
moe_status moe_ffn_combine(const moe_problem* p, const void* xg, const float* xg_scales, const void* w13,
                           const float* w13_scales, const void* w2, const float* w2_scales, const int32_t* masked_m,
                           const int32_t* offsets, const int32_t* row_of, const float* w, void* hg, float* hg_scales,
                           void* yg, void* out, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream);

/* EPLB load statistics ("vLLM EPLB", section 1.2: expert_load_pass and
 * expert_load_window).  Copies this pass's per-slot row counts masked_m[0..P)
 * (as written by moe_permute; the shared slot is not recorded) into row
 * (pass mod window) of load_window [window][P] int32 (device). */
moe_status moe_eplb_record(const moe_problem* p, const int32_t* masked_m, int64_t pass, int32_t window,
                           int32_t* load_window, moe_stream_t stream);

/* Rebalance from a load window ("vLLM EPLB", section 1.2: the window's physical
 * loads are summed per logical expert through physical_to_logical_map, then
 * replicas are re-assigned).  logical_load [E] int64 = sum over the window and
 * over the slots holding each expert; new_phys_to_log [P]: slots 0..E-1 hold
 * experts 0..E-1, slots E..P-1 hold the P-E experts with the largest load in
 * descending order (ties to the lower index) -- the single-GPU policy of this
 * library (the page's node / GPU packing is a multi-node control plane).
 * phys_to_log [P] is the map the window was recorded with (NULL when P == E).
 * Requires P - E <= E.  A map entry outside [0,E) sets MOE_FLAG_BAD_MAP.  One
 * CTA; all pointers device. */
moe_status moe_eplb_rebalance(const moe_problem* p, const int32_t* load_window, int32_t window,
                              const int32_t* phys_to_log, int64_t* logical_load, int32_t* new_phys_to_log,
                              int32_t* err_flag, moe_stream_t stream);

/* Diagnostic, an addition of this library (the pages describe none): runs the
 * bounded wait that every kernel here uses on an mbarrier that nothing
 * completes, with a limit of `cycles` SM cycles (1 .. 4e9), so that the expiry
 * path can be checked without a fault: the kernel ORs MOE_FLAG_TIMEOUT into
 * *err_flag (device int32) and returns; the context stays usable. */
moe_status moe_selftest_bounded_wait(int64_t cycles, int32_t* err_flag, moe_stream_t stream);

/* Host helper ("vLLM EPLB", section 1.2): invert a physical_to_logical map.
 * All pointers are HOST pointers.  p2l [P] in, l2p [E][R] out (slots of each
 * logical expert in ascending order, padded with -1), rc [E] out.  Returns
 * the largest replica count, or MOE_ERR_INVALID for an entry outside [0,E) or
 * an expert with more than R replicas. */
int32_t moe_eplb_invert(int32_t P, int32_t E, const int32_t* p2l, int32_t R, int32_t* l2p, int32_t* rc);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

/*
 * CPU oracle for the forward pass of one routed Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file.  The product path (the CUDA library and
 * its Python binding) never links, imports or calls it, and it shares no code,
 * header or table with that path.
 *
 * Plain, slow, obviously correct: per-token and per-row loops in fp64 that
 * write out the definition of each step.  Sources, cited by page and section:
 *   [MoE-EP]   "MoE inference and expert parallelism" (blog.vllbc.top,
 *              visual-reading/moe-inference-expert-parallel): routing section
 *              (Table 3-1), the forward-pass section (fused_topk ->
 *              moe_align_block_size -> W1/W3 GEMM -> activation -> W2 GEMM ->
 *              moe_sum), the shared expert (DeepSeek-V3 Eq. 12).
 *   [INFRA-5]  "Inference INFRA methodology (5): MoE inference - Batch, DeepEP,
 *              DeepGEMM and load balancing" (yfxerp.com): section "DeepGEMM"
 *              (masked [E_loc, M_max, K] layout with masked_m, FP8 with two-level
 *              accumulation), section "Batch" (coverage C(B)).
 *   [EPLB]     "vLLM EPLB" (pnsm.cn): section 1.2 "Basic concepts"
 *              (physical_to_logical_map, logical_to_physical_map,
 *              logical_replica_count and their worked example).
 *   [MoonEP]   "MoonEP: dynamic redundant experts" (wineandchord.com): sections
 *              "Why dynamic routing is hard" (sum_e T_e = R S K), "Perfect
 *              balance" (replicas leave the model function unchanged), "Zero-copy
 *              and static buffer" (padding described by the plan), "Correctness".
 * Codecs follow the OCP 8-bit floating point specification (E4M3) and IEEE 754
 * round-to-nearest-even for bf16.
 *
 * Readings of points the pages leave open are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Codecs                                                                    */
/* ------------------------------------------------------------------------ */

/* E4M3 (OCP 8-bit FP): sign, 4 exponent bits with bias 7, 3 mantissa bits.
 * E = 0 is subnormal: (M/8) * 2^-6.  S.1111.111 is NaN; there is no infinity,
 * so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t code) {
  const int s = code >> 7, E = (code >> 3) & 15, M = code & 7;
  if (E == 15 && M == 7) return NAN;
  const double v = (E == 0) ? ldexp((double)M, -9) : ldexp((double)(8 + M), E - 10);
  return s ? -v : v;
}

/* Round a float to E4M3: the nearest finite code, ties to the code with an
 * even mantissa, magnitudes above 448 saturate to 448 ("satfinite").
 * Found by brute force over the 127 non-negative finite codes. */
uint8_t orc_e4m3_encode(float v) {
  if (v != v) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (a > 448.0) return sign | 0x7E;
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      bestd = d;
      best = c;
    }
  }
  return sign | (uint8_t)best;
}

/* E2M1 (OCP Microscaling FP4): sign bit 3, exponent bits 2-1 with bias 1,
 * mantissa bit 0.  E = 0 is subnormal: (M/2) * 2^0; otherwise
 * (1 + M/2) * 2^(E-1).  No infinity or NaN: magnitudes 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6.  Used for the FP4 experts ("Inference INFRA methodology (5)",
 * shape-evolution table, DS-V4-Pro row: native FP4). */
double orc_e2m1_decode(uint8_t code) {
  const int s = (code >> 3) & 1, E = (code >> 1) & 3, M = code & 1;
  const double v = (E == 0) ? 0.5 * M : ldexp(1.0 + 0.5 * M, E - 1);
  return s ? -v : v;
}

/* The 256 decoded E4M3 values, tabulated from orc_e4m3_decode at load time. */
static double e4m3_table[256];

__attribute__((constructor)) static void build_e4m3_table(void) {
  for (int c = 0; c < 256; ++c) e4m3_table[c] = orc_e4m3_decode((uint8_t)c);
}

void orc_e4m3_decode_array(int64_t n, const uint8_t* codes, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(codes[i]);
}

void orc_e4m3_encode_array(int64_t n, const float* v, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

/* bf16 = the upper 16 bits of an IEEE binary32. */
double orc_bf16_decode(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a real value to the nearest bf16 (8 significant bits, exponent range
 * of binary32), ties to even, overflow to infinity. */
uint16_t orc_bf16_encode(double v) {
  if (v != v) return 0x7FC0;
  const double a = fabs(v);
  double r;
  if (a < ldexp(1.0, -126)) {
    r = nearbyint(ldexp(a, 133)) * ldexp(1.0, -133); /* subnormal quantum 2^-133 */
  } else {
    int e;
    frexp(a, &e);                        /* a in [2^(e-1), 2^e) */
    const double m = ldexp(a, 8 - e);    /* in [128, 256) */
    r = ldexp(nearbyint(m), e - 8);      /* nearbyint: ties to even */
  }
  const double maxf = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  float f = (r > maxf) ? INFINITY : (float)r;
  if (signbit(v)) f = -f;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

void orc_bf16_encode_array(int64_t n, const double* v, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_encode(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Matrix views over the storage formats                                     */
/* ------------------------------------------------------------------------ */

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_E2M1 = 3 };

/* rows x cols, row-major.  E2M1 data is packed two codes per byte along a
 * row (column 2j in bits 0-3 of byte j, column 2j+1 in bits 4-7), so a row
 * is cols/2 bytes.  E4M3 and E2M1 data carry fp32 scales, one per
 * (scale_rows x 128) block: [rows/scale_rows][cols/128].  scale_rows is 128
 * for expert weights (128x128 blocks) and 1 for activations (1x128 groups). */
typedef struct {
  int32_t dtype;
  int32_t scale_rows;
  const void* data;
  const float* scales;
  int64_t rows, cols;
} orc_mat;

static double mat_at(const orc_mat* m, int64_t r, int64_t c) {
  const int64_t i = r * m->cols + c;
  switch (m->dtype) {
    case ORC_F32:
      return (double)((const float*)m->data)[i];
    case ORC_BF16:
      return orc_bf16_decode(((const uint16_t*)m->data)[i]);
    case ORC_E2M1: {
      const uint8_t byte = ((const uint8_t*)m->data)[r * (m->cols / 2) + c / 2];
      const double s = (double)m->scales[(r / m->scale_rows) * (m->cols / 128) + c / 128];
      return orc_e2m1_decode((c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15)) * s;
    }
    default: {
      const double s = (double)m->scales[(r / m->scale_rows) * (m->cols / 128) + c / 128];
      return e4m3_table[((const uint8_t*)m->data)[i]] * s;
    }
  }
}

static void mat_row(const orc_mat* m, int64_t r, double* out) {
  for (int64_t c = 0; c < m->cols; ++c) out[c] = mat_at(m, r, c);
}

/* ------------------------------------------------------------------------ */
/* a1: routing                                                               */
/* ------------------------------------------------------------------------ */

/* [MoE-EP] routing section, Table 3-1: softmax scoring, top-K, renormalize.
 * p_e = exp(l_e) / sum_j exp(l_j) over all E experts; the K experts with the
 * largest p are chosen (ties: lower expert index first; ids are listed in
 * that order); weights are p renormalised over the chosen K.  Mixtral's
 * "top-2 then softmax" gives the same weights. */
void orc_route(int T, int E, int K, const float* logits, int32_t* ids, double* w) {
#pragma omp parallel
  {
    double* p = (double*)malloc((size_t)E * sizeof(double));
    char* taken = (char*)malloc((size_t)E);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      const float* l = logits + (int64_t)t * E;
      double lmax = -INFINITY;
      for (int e = 0; e < E; ++e)
        if ((double)l[e] > lmax) lmax = (double)l[e];
      double z = 0.0;
      for (int e = 0; e < E; ++e) {
        p[e] = exp((double)l[e] - lmax);
        z += p[e];
      }
      for (int e = 0; e < E; ++e) {
        p[e] /= z;
        taken[e] = 0;
      }
      double sum = 0.0;
      for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
        taken[best] = 1;
        ids[(int64_t)t * K + k] = best;
        sum += p[best];
      }
      for (int k = 0; k < K; ++k) w[(int64_t)t * K + k] = p[ids[(int64_t)t * K + k]] / sum;
    }
    free(p);
    free(taken);
  }
}

/* [MoE-EP] routing section, Table 3-1, DeepSeek-V3 row: sigmoid scoring with
 * e_score_correction_bias, grouped top-k ("first the top groups, then the
 * experts inside them"); the bias only decides which experts are chosen, the
 * weights use the unbiased sigmoid score.
 * Readings: s_e = 1/(1+exp(-l_e)); selection key c_e = s_e + bias_e (bias 0 when
 * absent); experts form n_group contiguous groups of E/n_group; a group's score
 * is the largest key in it; the topk_group best groups are kept (ties: lower
 * group index), then the K best keys among their experts (ties: lower expert
 * index), listed in that order; w_k = s_{e_k}, divided by their sum when
 * renormalize, then multiplied by scale.  All in fp64. */
void orc_route_grouped(int T, int E, int K, const float* logits, const float* bias, int n_group, int topk_group,
                       int renormalize, double scale, int32_t* ids, double* w) {
  const int gs = E / n_group;
#pragma omp parallel
  {
    double* sc = (double*)malloc((size_t)E * sizeof(double));
    double* key = (double*)malloc((size_t)E * sizeof(double));
    double* gsc = (double*)malloc((size_t)n_group * sizeof(double));
    char* gsel = (char*)malloc((size_t)n_group);
    char* taken = (char*)malloc((size_t)E);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      for (int e = 0; e < E; ++e) {
        sc[e] = 1.0 / (1.0 + exp(-(double)logits[(int64_t)t * E + e]));
        key[e] = sc[e] + (bias ? (double)bias[e] : 0.0);
        taken[e] = 0;
      }
      for (int g = 0; g < n_group; ++g) {
        gsc[g] = -INFINITY;
        for (int e = g * gs; e < (g + 1) * gs; ++e)
          if (key[e] > gsc[g]) gsc[g] = key[e];
        gsel[g] = 0;
      }
      for (int r = 0; r < topk_group; ++r) {
        int best = -1;
        for (int g = 0; g < n_group; ++g)
          if (!gsel[g] && (best < 0 || gsc[g] > gsc[best])) best = g;
        gsel[best] = 1;
      }
      double sum = 0.0;
      for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (gsel[e / gs] && !taken[e] && (best < 0 || key[e] > key[best])) best = e;
        taken[best] = 1;
        ids[(int64_t)t * K + k] = best;
        sum += sc[best];
      }
      for (int k = 0; k < K; ++k) {
        const double v = sc[ids[(int64_t)t * K + k]];
        w[(int64_t)t * K + k] = (renormalize ? v / sum : v) * scale;
      }
    }
    free(sc);
    free(key);
    free(gsc);
    free(gsel);
    free(taken);
  }
}

/* ------------------------------------------------------------------------ */
/* EPLB maps                                                                 */
/* ------------------------------------------------------------------------ */

/* [EPLB] section 1.2: physical_to_logical_map [P] names the logical expert in
 * each physical slot; logical_to_physical_map [E][R] lists, for each logical
 * expert, the slots holding it (ascending slot index), padded with -1;
 * logical_replica_count [E] counts them.
 * Returns the largest replica count, -1 for an out-of-range entry, -2 when a
 * logical expert has more than R replicas. */
int orc_eplb_invert(int P, int E, const int32_t* p2l, int R, int32_t* l2p, int32_t* rc) {
  for (int e = 0; e < E; ++e) {
    rc[e] = 0;
    for (int j = 0; j < R; ++j) l2p[e * R + j] = -1;
  }
  int maxr = 0;
  for (int s = 0; s < P; ++s) {
    const int e = p2l[s];
    if (e < 0 || e >= E) return -1;
    if (rc[e] >= R) return -2;
    l2p[e * R + rc[e]] = s;
    rc[e] += 1;
    if (rc[e] > maxr) maxr = rc[e];
  }
  return maxr;
}

/* [EPLB] section 1.2: expert_load_pass holds each physical slot's token count
 * for one forward pass (the per-slot row counts, masked_m); the passes of a
 * window are kept in expert_load_window [W][P]; at a rebalance the window's
 * physical loads are summed per logical expert through physical_to_logical_map
 * and replicas are re-assigned.
 * Reading of the policy (the page's hierarchical / global packing is a
 * multi-node control plane): slots 0..E-1 keep experts 0..E-1 and the P-E
 * extra slots hold the P-E experts with the largest load, in descending load
 * (ties: lower expert index).  window may be NULL for W = 0.  Returns -1 for a
 * map entry outside [0,E) or sizes with E < 1, P < E or P - E > E, 0
 * otherwise. */
int orc_eplb_rebalance(int P, int E, int W, const int32_t* window, const int32_t* p2l, int64_t* logical_load,
                       int32_t* new_p2l) {
  if (E <= 0 || P < E || P - E > E) return -1;
  for (int e = 0; e < E; ++e) logical_load[e] = 0;
  for (int s = 0; s < P; ++s) {
    const int e = p2l ? p2l[s] : s;
    if (e < 0 || e >= E) return -1;
    for (int w = 0; w < W; ++w) logical_load[e] += window[(int64_t)w * P + s];
  }
  for (int e = 0; e < E; ++e) new_p2l[e] = e;
  char* used = (char*)calloc((size_t)E, 1);
  for (int r = 0; r < P - E; ++r) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!used[e] && (best < 0 || logical_load[e] > logical_load[best])) best = e;
    used[best] = 1;
    new_p2l[E + r] = best;
  }
  free(used);
  return 0;
}

/* [INFRA-5] "DeepGEMM", the padding-waste example: an expert with M_e rows
 * occupies ceil(M_e / BM) token tiles of BM rows, so the MMA work is
 * ceil(M_e / BM) * BM / M_e times the useful work.  orc_token_tiles sums the
 * tiles over the slots (a slot with no rows has none); orc_pad_waste is the
 * ratio for one expert. */
int64_t orc_token_tiles(int nslots, const int32_t* masked_m, int BM) {
  int64_t n = 0;
  for (int s = 0; s < nslots; ++s)
    if (masked_m[s] > 0) n += (masked_m[s] + BM - 1) / BM;
  return n;
}

double orc_pad_waste(int M_e, int BM) { return (double)((M_e + BM - 1) / BM) * BM / (double)M_e; }

/* ------------------------------------------------------------------------ */
/* a2: dispatch layout                                                       */
/* ------------------------------------------------------------------------ */

/* [INFRA-5] "DeepGEMM": the masked layout is a static buffer [E_loc, M_max, H]
 * plus a per-slot row count masked_m; prefill uses a contiguous
 * expert-grouped layout with per-expert offsets.  [MoonEP] "Why dynamic
 * routing is hard": the per-expert counts T_e sum to the number of routed
 * records.  [EPLB] section 1.2 gives the replica maps.
 *
 * Readings: record (t,k) of logical expert e goes to slot e without a map, or
 * to replica l2p[e][t mod rc[e]] with one (round-robin by token index).  Rows
 * of a slot are in ascending token order.  With a shared expert (S = 1) slot P
 * holds every token, row t.  masked: row = s*M_max + rank; contiguous:
 * row = offsets[s] + rank, offsets the exclusive prefix sum of masked_m.
 * src_of[row] = t for every written row (others untouched).
 *
 * Outputs: slot_of [T*K], masked_m [P+S], offsets [P+S+1], row_of [T*(K+S)],
 * src_of [rows].  Returns 0, -1 for a bad expert id or map entry, -2 for a
 * slot whose count exceeds M_max (masked layout; rows >= M_max not written),
 * -3 for an expert chosen twice by one token, -4 for a logical expert that
 * is routed to but has no slot. */
int orc_layout(int T, int K, int E, int P, int S, int masked, int M_max, const int32_t* ids,
               const int32_t* p2l, int32_t* slot_of, int32_t* masked_m, int32_t* offsets, int32_t* row_of,
               int32_t* src_of) {
  int status = 0;
  int32_t* rc = NULL;
  int32_t* l2p = NULL;
  if (p2l) {
    rc = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    l2p = (int32_t*)malloc((size_t)E * (size_t)P * sizeof(int32_t));
    if (orc_eplb_invert(P, E, p2l, P, l2p, rc) < 0) {
      free(rc);
      free(l2p);
      return -1;
    }
  }
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      const int e = ids[t * K + k];
      int s = -1;
      if (e < 0 || e >= E) {
        status = -1;
      } else if (p2l) {
        if (rc[e] == 0)
          status = -4;
        else
          s = l2p[e * P + (t % rc[e])];
      } else {
        s = e;
      }
      for (int j = 0; j < k; ++j)
        if (ids[t * K + j] == e) status = -3;
      slot_of[t * K + k] = s;
    }
  }
  if (status) {
    free(rc);
    free(l2p);
    return status;
  }
  for (int s = 0; s < P + S; ++s) masked_m[s] = 0;
  for (int i = 0; i < T * K; ++i) masked_m[slot_of[i]] += 1;
  if (S) masked_m[P] = T;
  offsets[0] = 0;
  for (int s = 0; s < P + S; ++s) offsets[s + 1] = offsets[s] + masked_m[s];
  for (int s = 0; s < P + S; ++s)
    if (masked && masked_m[s] > M_max) status = -2;

  /* ranks: one pass over tokens in ascending order, a running count per slot */
  int32_t* next = (int32_t*)calloc((size_t)(P + S), sizeof(int32_t));
  const int KS = K + S;
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < KS; ++k) {
      const int s = (k < K) ? slot_of[t * K + k] : P;
      const int rank = next[s]++;
      const int row = masked ? s * M_max + rank : offsets[s] + rank;
      row_of[t * KS + k] = row;
      if (!masked || rank < M_max) src_of[row] = t;
    }
  }
  free(next);
  free(rc);
  free(l2p);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Quantisation of activations                                               */
/* ------------------------------------------------------------------------ */

/* [INFRA-5] "DeepGEMM" / "DeepEP": activations travel in FP8 with 1x128 group
 * scales.  Reading: per row and group of 128, amax = max|x| in fp32,
 * s = amax / 448 (IEEE fp32 division; s = 1 when amax = 0),
 * q = e4m3(x / s) (fp32 division, nearest-even, satfinite).
 * x [n][H] fp32 -> q [n][H], s [n][H/128]. */
void orc_quant_rows_e4m3(int64_t n, int H, const float* x, uint8_t* q, float* s) {
  const int G = H / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int g = 0; g < G; ++g) {
      const float* xs = x + r * H + g * 128;
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i)
        if (fabsf(xs[i]) > amax) amax = fabsf(xs[i]);
      volatile float sc = amax / 448.0f;
      if (amax == 0.0f) sc = 1.0f;
      s[r * G + g] = sc;
      for (int i = 0; i < 128; ++i) {
        volatile float v = xs[i] / sc;
        q[r * H + g * 128 + i] = orc_e4m3_encode(v);
      }
    }
  }
}

/* Round a row of real values to the storage type of an intermediate and back.
 * dtype f32 / bf16: nearest-even.  e4m3: the 1x128 group rule above applied to
 * the fp32 value of each element; the result is q * s. */
static void round_row(int dtype, int n, double* v) {
  if (dtype == ORC_F32) {
    for (int i = 0; i < n; ++i) v[i] = (double)(float)v[i];
  } else if (dtype == ORC_BF16) {
    for (int i = 0; i < n; ++i) v[i] = orc_bf16_decode(orc_bf16_encode(v[i]));
  } else {
    float xs[128];
    uint8_t q[128];
    float sc;
    for (int g = 0; g < n / 128; ++g) {
      for (int i = 0; i < 128; ++i) xs[i] = (float)v[g * 128 + i];
      orc_quant_rows_e4m3(1, 128, xs, q, &sc);
      for (int i = 0; i < 128; ++i) v[g * 128 + i] = e4m3_table[q[i]] * (double)sc;
    }
  }
}

/* Store a row of real values in a storage type (scales for e4m3). */
static void store_row(int dtype, int n, const double* v, void* dst, int64_t row, float* scales) {
  if (dtype == ORC_F32) {
    for (int i = 0; i < n; ++i) ((float*)dst)[row * n + i] = (float)v[i];
  } else if (dtype == ORC_BF16) {
    for (int i = 0; i < n; ++i) ((uint16_t*)dst)[row * n + i] = orc_bf16_encode(v[i]);
  } else {
    float xs[128];
    for (int g = 0; g < n / 128; ++g) {
      for (int i = 0; i < 128; ++i) xs[i] = (float)v[g * 128 + i];
      orc_quant_rows_e4m3(1, 128, xs, (uint8_t*)dst + row * n + g * 128, scales + row * (n / 128) + g);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* a3 / a4: one SwiGLU expert                                                */
/* ------------------------------------------------------------------------ */

/* [MoE-EP] routing section: each chosen expert is a SwiGLU FFN; W1 / W3 are
 * gate / up, W2 is down:  h = silu(W1 x) * (W3 x),  y = W2 h,
 * silu(z) = z / (1 + exp(-z)).
 * Storage (math weights kept transposed, rows contiguous along the reduced
 * dimension): W13 rows [slot*2I, slot*2I + I) are W1 (gate), the next I rows
 * are W3 (up), each of length H; W2 rows [slot*H, slot*H + H), length I. */
static void gate_up(const orc_mat* w13, int64_t slot, int H, int I, const double* x, double* h, double* wrow) {
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    mat_row(w13, slot * 2 * I + n, wrow);
    for (int k = 0; k < H; ++k) g += wrow[k] * x[k];
    mat_row(w13, slot * 2 * I + I + n, wrow);
    for (int k = 0; k < H; ++k) u += wrow[k] * x[k];
    h[n] = g / (1.0 + exp(-g)) * u;
  }
}

static void down(const orc_mat* w2, int64_t slot, int H, int I, const double* h, double* y, double* wrow) {
  for (int n = 0; n < H; ++n) {
    double acc = 0.0;
    mat_row(w2, slot * H + n, wrow);
    for (int k = 0; k < I; ++k) acc += wrow[k] * h[k];
    y[n] = acc;
  }
}

/* ------------------------------------------------------------------------ */
/* Per-call oracles over the grouped layout                                  */
/* ------------------------------------------------------------------------ */

static int64_t group_row(int masked, int M_max, const int32_t* offsets, int s, int r) {
  return masked ? (int64_t)s * M_max + r : (int64_t)offsets[s] + r;
}

/* a3 [INFRA-5] "DeepGEMM": for every slot s and valid row r < masked_m[s]
 * (rows past masked_m are padding and are not computed),
 * Hg[row] = store(h_dtype, silu(W1[s] xg[row]) * (W3[s] xg[row])). */
void orc_grouped_swiglu(int nslots, int H, int I, int masked, int M_max, const orc_mat* xg, const orc_mat* w13,
                        const int32_t* masked_m, const int32_t* offsets, int h_dtype, void* hg, float* hg_scales) {
  int64_t total = 0;
  for (int s = 0; s < nslots; ++s) total += masked_m[s];
  int32_t* rs = (int32_t*)malloc((size_t)(total + 1) * 2 * sizeof(int32_t));
  int64_t c = 0;
  for (int s = 0; s < nslots; ++s)
    for (int r = 0; r < masked_m[s]; ++r) {
      rs[2 * c] = s;
      rs[2 * c + 1] = r;
      ++c;
    }
#pragma omp parallel
  {
    double* x = (double*)malloc((size_t)H * sizeof(double));
    double* h = (double*)malloc((size_t)I * sizeof(double));
    double* wrow = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < total; ++i) {
      const int s = rs[2 * i], r = rs[2 * i + 1];
      const int64_t row = group_row(masked, M_max, offsets, s, r);
      mat_row(xg, row, x);
      gate_up(w13, s, H, I, x, h, wrow);
      store_row(h_dtype, I, h, hg, row, hg_scales);
    }
    free(x);
    free(h);
    free(wrow);
  }
  free(rs);
}

/* a4: Yg[row] = store(y_dtype, W2[s] hg[row]) for every valid row. */
void orc_grouped_down(int nslots, int H, int I, int masked, int M_max, const orc_mat* hg, const orc_mat* w2,
                      const int32_t* masked_m, const int32_t* offsets, int y_dtype, void* yg) {
  int64_t total = 0;
  for (int s = 0; s < nslots; ++s) total += masked_m[s];
  int32_t* rs = (int32_t*)malloc((size_t)(total + 1) * 2 * sizeof(int32_t));
  int64_t c = 0;
  for (int s = 0; s < nslots; ++s)
    for (int r = 0; r < masked_m[s]; ++r) {
      rs[2 * c] = s;
      rs[2 * c + 1] = r;
      ++c;
    }
#pragma omp parallel
  {
    double* h = (double*)malloc((size_t)I * sizeof(double));
    double* y = (double*)malloc((size_t)H * sizeof(double));
    double* wrow = (double*)malloc((size_t)I * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < total; ++i) {
      const int s = rs[2 * i], r = rs[2 * i + 1];
      const int64_t row = group_row(masked, M_max, offsets, s, r);
      mat_row(hg, row, h);
      down(w2, s, H, I, h, y, wrow);
      store_row(y_dtype, H, y, yg, row, NULL);
    }
    free(h);
    free(y);
    free(wrow);
  }
  free(rs);
}

/* a5 [MoE-EP] routing section (moe_sum / TopKWeightAndReduce) and the shared
 * expert of DeepSeek-V3 Eq. 12:
 *   out[t] = sum_k w[t,k] * Yg[row_of[t,k]]  (+ Yg[row_of[t,K]] with weight 1),
 * then rounded once to the output type.  out_exact receives the unrounded sum. */
void orc_combine(int T, int H, int K, int S, const orc_mat* yg, const int32_t* row_of, const float* w,
                 int out_dtype, void* out, double* out_exact) {
#pragma omp parallel
  {
    double* y = (double*)malloc((size_t)H * sizeof(double));
    double* acc = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      for (int i = 0; i < H; ++i) acc[i] = 0.0;
      for (int k = 0; k < K + S; ++k) {
        const double wk = (k < K) ? (double)w[t * K + k] : 1.0;
        mat_row(yg, row_of[t * (K + S) + k], y);
        for (int i = 0; i < H; ++i) acc[i] += wk * y[i];
      }
      if (out_exact)
        for (int i = 0; i < H; ++i) out_exact[(int64_t)t * H + i] = acc[i];
      store_row(out_dtype, H, acc, out, t, NULL);
    }
    free(y);
    free(acc);
  }
}

/* ------------------------------------------------------------------------ */
/* The whole layer, token by token                                           */
/* ------------------------------------------------------------------------ */

/* out[t] = (S ? FFN_shared(xq[t]) : 0) + sum_k w[t,k] * FFN_{ids[t,k]}(xq[t])
 * [MoE-EP] routing section (Mixtral: weighted sum of the top-2 SwiGLU experts;
 * DeepSeek-V3 Eq. 12: shared + routed, the residual u_t excluded as it is
 * added outside the layer).  Replicas from an EPLB map hold the same weights
 * and so do not change the result ([MoonEP] "Perfect balance"); the oracle
 * reads the logical experts directly.
 * Readings of the storage roundings the GPU path also performs:
 *   xq  = x, or for e4m3 activations the 1x128 group quantisation of x;
 *   h   rounded to h_dtype; y rounded to y_dtype; out rounded to out_dtype.
 * w13 / w2 are the logical experts [E+S] (shared last).  Computes the tokens
 * listed in toks (n_toks of them), writing out row i for toks[i]; the fp64
 * unrounded result goes to out_exact[i] when given. */
void orc_layer_tokens(int T, int H, int I, int E, int K, int S, const float* logits, const orc_mat* x,
                      int act_dtype, const orc_mat* w13, const orc_mat* w2, int h_dtype, int y_dtype,
                      int out_dtype, int n_toks, const int32_t* toks, void* out, double* out_exact) {
  (void)T;
#pragma omp parallel
  {
    double* xr = (double*)malloc((size_t)H * sizeof(double));
    double* h = (double*)malloc((size_t)I * sizeof(double));
    double* y = (double*)malloc((size_t)H * sizeof(double));
    double* acc = (double*)malloc((size_t)H * sizeof(double));
    double* wrow = (double*)malloc((size_t)(H > I ? H : I) * sizeof(double));
    double* wk = (double*)malloc((size_t)(K + 1) * sizeof(double));
    int32_t* ek = (int32_t*)malloc((size_t)(K + 1) * sizeof(int32_t));
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_toks; ++i) {
      const int t = toks[i];
      orc_route(1, E, K, logits + (int64_t)t * E, ek, wk);
      mat_row(x, t, xr);
      if (act_dtype == ORC_E4M3) round_row(ORC_E4M3, H, xr);
      for (int c = 0; c < H; ++c) acc[c] = 0.0;
      for (int k = 0; k < K + S; ++k) {
        const int e = (k < K) ? ek[k] : E;
        const double g = (k < K) ? wk[k] : 1.0;
        gate_up(w13, e, H, I, xr, h, wrow);
        round_row(h_dtype, I, h);
        down(w2, e, H, I, h, y, wrow);
        round_row(y_dtype, H, y);
        for (int c = 0; c < H; ++c) acc[c] += g * y[c];
      }
      if (out_exact)
        for (int c = 0; c < H; ++c) out_exact[(int64_t)i * H + c] = acc[c];
      store_row(out_dtype, H, acc, out, i, NULL);
    }
    free(xr);
    free(h);
    free(y);
    free(acc);
    free(wrow);
    free(wk);
    free(ek);
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

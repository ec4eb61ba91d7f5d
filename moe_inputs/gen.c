/*
 * Seeded synthetic inputs for the routed-expert MoE layer.
 *
 * This file draws random numbers and packs them into the storage formats the
 * layer consumes (fp32, bf16, e4m3 with 128x128 block scales).  It holds none
 * of the layer's own arithmetic: no routing, no dispatch, no expert FFN, no
 * combine.  Both the CPU oracle and the CUDA path read what it writes.
 *
 * Generator (counter based, so any slice can be regenerated on its own):
 *   mix(z)        = the splitmix64 finaliser
 *                   z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(seed, s)  = mix(mix(seed) + s)                   one key per tensor stream s
 *   bits(key, i)  = mix(key + (i+1) * 0x9E3779B97F4A7C15) i-th raw draw
 *   uniform(i)    = (bits >> 11) * 2^-53                  in [0, 1)
 *   normal(i)     = Box-Muller on the pair j = i/2:
 *                   r = sqrt(-2 ln(1 - uniform(2j))), a = 2 pi uniform(2j+1)
 *                   normal(2j) = r cos a, normal(2j+1) = r sin a
 *
 * Results are identical from run to run on one machine.  libm's log/sin/cos
 * may differ in the last bit between CPU architectures, so no test compares
 * generated values across machines; every reference is computed in-process
 * from the same arrays the GPU receives.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

uint64_t mg_stream_key(uint64_t seed, uint64_t stream) { return mix64(mix64(seed) + stream); }

static inline uint64_t draw_bits(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static inline double draw_uniform(uint64_t key, uint64_t i) {
  return (double)(draw_bits(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

static inline void draw_normal_pair(uint64_t key, uint64_t j, double* n0, double* n1) {
  const double u1 = draw_uniform(key, 2 * j);
  const double u2 = draw_uniform(key, 2 * j + 1);
  const double r = sqrt(-2.0 * log(1.0 - u1));
  const double a = 6.283185307179586476925286766559 * u2;
  *n0 = r * cos(a);
  *n1 = r * sin(a);
}

static inline double draw_normal(uint64_t key, uint64_t i) {
  double n0, n1;
  draw_normal_pair(key, i >> 1, &n0, &n1);
  return (i & 1) ? n1 : n0;
}

/* out[i] = mean + std * normal(offset + i) for i < n, two draws per Box-Muller pair. */
static void fill_normal(uint64_t key, uint64_t offset, int64_t n, double mean, double std, double* out) {
  int64_t i = 0;
  if (n > 0 && (offset & 1)) {
    out[0] = mean + std * draw_normal(key, offset);
    i = 1;
  }
  for (; i + 1 < n; i += 2) {
    double n0, n1;
    draw_normal_pair(key, (offset + (uint64_t)i) >> 1, &n0, &n1);
    out[i] = mean + std * n0;
    out[i + 1] = mean + std * n1;
  }
  if (i < n) out[i] = mean + std * draw_normal(key, offset + (uint64_t)i);
}

#define CHUNK 4096

/* ---- storage codecs used to pack inputs (input preparation only) ---- */

/* Round a double to the nearest bf16 value (ties to even); returns the bits. */
static uint16_t pack_bf16(double v) {
  float f;
  if (v != v) return 0x7FC0;
  /* Round to 8 significant bits at the binade of v, or to the subnormal quantum. */
  double a = fabs(v);
  double r;
  if (a == 0.0) {
    r = 0.0;
  } else {
    int e;
    frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8; /* quantum exponent: 8 significant bits */
    if (q < -133) q = -133;
    r = ldexp(nearbyint(ldexp(a, -q)), q);
  }
  if (r > 3.38953138925153547590470800371487866880e+38) r = INFINITY;
  f = (float)(v < 0 ? -r : r); /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Encode a double as e4m3 (bias 7, 3 mantissa bits, max 448, no inf),
 * round to nearest even, saturating to +-448. */
static uint8_t pack_e4m3(double v) {
  uint8_t sign = (v < 0) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a != a) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  int e;
  if (a == 0.0) return sign;
  frexp(a, &e);
  int ex = e - 1; /* a in [2^ex, 2^(ex+1)) */
  if (ex < -6) ex = -6;
  double r = ldexp(nearbyint(ldexp(a, 3 - ex)), ex - 3); /* quantum 2^(ex-3) */
  if (r >= 448.0) return sign | 0x7E;
  if (r == 0.0) return sign;
  if (r < 0.015625) { /* subnormal: r = m * 2^-9, m in 1..7 */
    return sign | (uint8_t)nearbyint(ldexp(r, 9));
  }
  frexp(r, &e);
  ex = e - 1;
  int man = (int)nearbyint(ldexp(r, 3 - ex)) - 8;
  return sign | (uint8_t)(((ex + 7) << 3) | man);
}

/* Encode a double as OCP FP4 E2M1 (sign, 2 exponent bits with bias 1, 1
 * mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6): the nearest
 * magnitude, ties to the code with mantissa bit 0, saturating to +-6. */
static uint8_t pack_e2m1(double v) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = (v < 0) ? 0x8 : 0x0;
  const double a = fabs(v);
  if (a != a) return 0;
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double d = fabs(mag[c] - a), bd = fabs(mag[best] - a);
    if (d < bd || (d == bd && (c & 1) == 0)) best = c;
  }
  return sign | (uint8_t)best;
}

/* ---- public entry points ---- */

void mg_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double lo, double hi,
                    double* out) {
  const uint64_t key = mg_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = lo + (hi - lo) * draw_uniform(key, offset + (uint64_t)i);
}

void mg_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean, double std,
             double* out) {
  const uint64_t key = mg_stream_key(seed, stream);
  const int64_t nchunks = (n + CHUNK - 1) / CHUNK;
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < nchunks; ++c) {
    double buf[CHUNK];
    const int64_t i0 = c * CHUNK;
    const int64_t m = (n - i0 < CHUNK) ? n - i0 : CHUNK;
    fill_normal(key, offset + (uint64_t)i0, m, mean, std, buf);
    for (int64_t i = 0; i < m; ++i) out[i0 + i] = buf[i];
  }
}

void mg_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean, double std,
             float* out) {
  const uint64_t key = mg_stream_key(seed, stream);
  const int64_t nchunks = (n + CHUNK - 1) / CHUNK;
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < nchunks; ++c) {
    double buf[CHUNK];
    const int64_t i0 = c * CHUNK;
    const int64_t m = (n - i0 < CHUNK) ? n - i0 : CHUNK;
    fill_normal(key, offset + (uint64_t)i0, m, mean, std, buf);
    for (int64_t i = 0; i < m; ++i) out[i0 + i] = (float)buf[i];
  }
}

void mg_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean, double std,
              uint16_t* out) {
  const uint64_t key = mg_stream_key(seed, stream);
  const int64_t nchunks = (n + CHUNK - 1) / CHUNK;
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < nchunks; ++c) {
    double buf[CHUNK];
    const int64_t i0 = c * CHUNK;
    const int64_t m = (n - i0 < CHUNK) ? n - i0 : CHUNK;
    fill_normal(key, offset + (uint64_t)i0, m, mean, std, buf);
    for (int64_t i = 0; i < m; ++i) out[i0 + i] = pack_bf16(buf[i]);
  }
}

/* Expert weights in e4m3 with one fp32 scale per 128x128 block.
 * The logical tensor is [n_exp, N, K] (row-major, K contiguous); this fills
 * experts [e0, e0+ne).  Element (e,n,k) uses draw index (e*N+n)*K+k of the
 * normal stream; block (e,nb,kb) uses draw index (e*(N/128)+nb)*(K/128)+kb of
 * the uniform stream u ~ U[0.5, 2].  Per block: s = fp32(u * max|w| / 448),
 * q = e4m3(w / s) rounded to nearest even and saturated to +-448.
 * q is [ne, N, K] bytes, s is [ne, N/128, K/128] floats.  N, K % 128 == 0. */
void mg_weights_e4m3(uint64_t seed, uint64_t w_stream, uint64_t s_stream, int64_t e0, int64_t ne, int64_t N,
                     int64_t K, double std, uint8_t* q, float* s) {
  const uint64_t wkey = mg_stream_key(seed, w_stream);
  const uint64_t skey = mg_stream_key(seed, s_stream);
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t nblocks = ne * NB * KB;
#pragma omp parallel
  {
    double* buf = (double*)malloc(128 * 128 * sizeof(double));
#pragma omp for schedule(dynamic, 4)
    for (int64_t b = 0; b < nblocks; ++b) {
      const int64_t el = b / (NB * KB);
      const int64_t nb = (b / KB) % NB;
      const int64_t kb = b % KB;
      const int64_t e = e0 + el;
      double amax = 0.0;
      for (int64_t i = 0; i < 128; ++i) {
        const uint64_t base = (uint64_t)((e * N + nb * 128 + i) * K + kb * 128);
        fill_normal(wkey, base, 128, 0.0, std, buf + i * 128);
        for (int64_t j = 0; j < 128; ++j)
          if (fabs(buf[i * 128 + j]) > amax) amax = fabs(buf[i * 128 + j]);
      }
      const double u = 0.5 + 1.5 * draw_uniform(skey, (uint64_t)((e * NB + nb) * KB + kb));
      float sc = (float)(u * amax / 448.0);
      if (sc == 0.0f) sc = 1.0f;
      s[(el * NB + nb) * KB + kb] = sc;
      for (int64_t i = 0; i < 128; ++i) {
        uint8_t* dst = q + (el * N + nb * 128 + i) * K + kb * 128;
        for (int64_t j = 0; j < 128; ++j) dst[j] = pack_e4m3(buf[i * 128 + j] / (double)sc);
      }
    }
    free(buf);
  }
}

/* Expert weights in FP4 E2M1 with one fp32 scale per 128x128 block: the
 * e4m3 recipe above with the E2M1 maximum, s = fp32(u * max|w| / 6) and
 * q = e2m1(w / s) nearest (ties to an even mantissa), saturated to +-6.
 * Same draw indices as mg_weights_e4m3.  q is [ne, N, K/2] bytes, two codes
 * per byte along K: column 2j in bits 0-3, column 2j+1 in bits 4-7. */
void mg_weights_e2m1(uint64_t seed, uint64_t w_stream, uint64_t s_stream, int64_t e0, int64_t ne, int64_t N,
                     int64_t K, double std, uint8_t* q, float* s) {
  const uint64_t wkey = mg_stream_key(seed, w_stream);
  const uint64_t skey = mg_stream_key(seed, s_stream);
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t nblocks = ne * NB * KB;
#pragma omp parallel
  {
    double* buf = (double*)malloc(128 * 128 * sizeof(double));
#pragma omp for schedule(dynamic, 4)
    for (int64_t b = 0; b < nblocks; ++b) {
      const int64_t el = b / (NB * KB);
      const int64_t nb = (b / KB) % NB;
      const int64_t kb = b % KB;
      const int64_t e = e0 + el;
      double amax = 0.0;
      for (int64_t i = 0; i < 128; ++i) {
        const uint64_t base = (uint64_t)((e * N + nb * 128 + i) * K + kb * 128);
        fill_normal(wkey, base, 128, 0.0, std, buf + i * 128);
        for (int64_t j = 0; j < 128; ++j)
          if (fabs(buf[i * 128 + j]) > amax) amax = fabs(buf[i * 128 + j]);
      }
      const double u = 0.5 + 1.5 * draw_uniform(skey, (uint64_t)((e * NB + nb) * KB + kb));
      float sc = (float)(u * amax / 6.0);
      if (sc == 0.0f) sc = 1.0f;
      s[(el * NB + nb) * KB + kb] = sc;
      for (int64_t i = 0; i < 128; ++i) {
        uint8_t* dst = q + ((el * N + nb * 128 + i) * K + kb * 128) / 2;
        for (int64_t j = 0; j < 128; j += 2)
          dst[j / 2] = (uint8_t)(pack_e2m1(buf[i * 128 + j] / (double)sc) |
                                 (pack_e2m1(buf[i * 128 + j + 1] / (double)sc) << 4));
      }
    }
    free(buf);
  }
}

/* Expert weights in bf16: logical tensor [n_exp, N, K], experts [e0, e0+ne). */
void mg_weights_bf16(uint64_t seed, uint64_t w_stream, int64_t e0, int64_t ne, int64_t N, int64_t K, double std,
                     uint16_t* out) {
  const uint64_t wkey = mg_stream_key(seed, w_stream);
  const int64_t rows = ne * N;
#pragma omp parallel
  {
    double* buf = (double*)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      fill_normal(wkey, (uint64_t)((e0 * N + r) * K), K, 0.0, std, buf);
      for (int64_t k = 0; k < K; ++k) out[r * K + k] = pack_bf16(buf[k]);
    }
    free(buf);
  }
}

/* Expert weights in fp32: logical tensor [n_exp, N, K], experts [e0, e0+ne). */
void mg_weights_f32(uint64_t seed, uint64_t w_stream, int64_t e0, int64_t ne, int64_t N, int64_t K, double std,
                    float* out) {
  const uint64_t wkey = mg_stream_key(seed, w_stream);
  const int64_t rows = ne * N;
#pragma omp parallel
  {
    double* buf = (double*)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      fill_normal(wkey, (uint64_t)((e0 * N + r) * K), K, 0.0, std, buf);
      for (int64_t k = 0; k < K; ++k) out[r * K + k] = (float)buf[k];
    }
    free(buf);
  }
}

int mg_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

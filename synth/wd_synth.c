/*
 * wd_synth.c - seeded synthetic inputs for the MoE decode layer.
 *
 * This module generates the inputs that BOTH sides consume: the CPU oracle and
 * the CUDA path.  It holds none of the layer's arithmetic (no dequantisation,
 * no dot products, no SiLU, no combine); it only draws numbers and encodes the
 * weights the way a producer of MXFP8 checkpoints would.
 *
 * Workload recipe (Qwen-3-style shapes from the warp-decode blog, Cursor,
 * "用 warp decode 实现更好的 MoE 模型推理", section 传统的 MoE 路径: 8 of 128
 * experts per token):
 *   - activations x ~ N(0,1), rounded to BF16 (round to nearest even);
 *   - router logits ~ N(0,1) over E experts, softmax, top-K with ties broken
 *     toward the lower expert id, K weights renormalised to sum to 1 (FP32);
 *   - expert weights W ~ N(0, std = 1/sqrt(fan_in)) in FP32, quantised to MXFP8:
 *     E4M3 elements and one E8M0 scale per 32 contiguous elements along the
 *     reduction dimension, scale = 2^(floor(log2(amax)) - 8), elements rounded to
 *     nearest even and saturated to +-448.
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC 2011), keyed by the 64-bit seed.  Every value
 * has its own counter (layer, kind, expert, row, column/4), so any slice of any
 * tensor can be regenerated on its own, in any order, on any number of threads.
 * Normals come from the Box-Muller transform of two uniforms in (0,1).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WD_SYNTH_API __attribute__((visibility("default")))

/* Counter "kind" field: which tensor a draw belongs to. */
enum { KIND_X = 1, KIND_LOGITS = 2, KIND_GATE_UP = 3, KIND_DOWN = 4, KIND_PERM = 5 };

/* ---------------------------------------------------------------- Philox ---- */

static inline void philox_round(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
  const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  const uint32_t n0 = hi1 ^ c[1] ^ k[0];
  const uint32_t n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

/* Philox4x32 with 10 rounds: 4 x 32 random bits for one 128-bit counter. */
WD_SYNTH_API void wd_synth_philox4x32_10(uint64_t seed, const uint32_t ctr[4], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  for (int r = 0; r < 10; ++r) {
    philox_round(c, k);
    k[0] += 0x9E3779B9u;
    k[1] += 0xBB67AE85u;
  }
  memcpy(out, c, sizeof(c));
}

/* Uniform in (0,1) from 32 random bits: 2^-33 .. 1 - 2^-33, never 0 or 1. */
static inline double u01(uint32_t r) { return ((double)r + 0.5) * (1.0 / 4294967296.0); }

/* Natural log of u > 0 (normal double): u = m 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln u = e ln 2 + 2 atanh(t), t = (m-1)/(m+1), |t| < 0.172; the atanh series is
 * cut after t^11 (truncation below 1e-10).  Only IEEE +,-,*,/ are used, so the
 * result is the same on every machine that compiles without FMA contraction. */
static inline double ln_pos(double u) {
  uint64_t b;
  memcpy(&b, &u, 8);
  int e = (int)((b >> 52) & 0x7FF) - 1023;
  b = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
  double m;
  memcpy(&m, &b, 8);
  if (m > 1.4142135623730951) {
    m *= 0.5;
    e += 1;
  }
  const double t = (m - 1.0) / (m + 1.0), t2 = t * t;
  const double s =
      t * (2.0 + t2 * (2.0 / 3 + t2 * (2.0 / 5 + t2 * (2.0 / 7 + t2 * (2.0 / 9 + t2 * (2.0 / 11))))));
  return (double)e * 0.69314718055994530942 + s;
}

/* sin and cos of 2*pi*u for u in [0,1): quadrant q = floor(4u), phi in [0, pi/2),
 * Taylor series of sin to phi^13 and cos to phi^14 (truncation below 1e-9). */
static inline void sincos_2pi(double u, double* sn, double* cs) {
  const double v = u * 4.0;
  int q = (int)v;
  if (q > 3) q = 3;
  const double phi = (v - (double)q) * 1.57079632679489661923, p2 = phi * phi;
  /* Horner form with constant coefficients (+-1/n!) */
  const double s =
      phi * (1.0 + p2 * (-1.0 / 6 + p2 * (1.0 / 120 + p2 * (-1.0 / 5040 + p2 * (1.0 / 362880 +
      p2 * (-1.0 / 39916800 + p2 * (1.0 / 6227020800.0)))))));
  const double c = 1.0 + p2 * (-1.0 / 2 + p2 * (1.0 / 24 + p2 * (-1.0 / 720 + p2 * (1.0 / 40320 +
                   p2 * (-1.0 / 3628800 + p2 * (1.0 / 479001600.0 + p2 * (-1.0 / 87178291200.0)))))));
  const double a = (q & 1) ? c : s, b2 = (q & 1) ? -s : c, sg = (q & 2) ? -1.0 : 1.0;
  *sn = sg * a;
  *cs = sg * b2;
}

/* Four N(0,1) draws for counter (col4, row, kind<<24 | expert, layer):
 * Box-Muller on the uniform pairs (r0, r1) and (r2, r3). */
static inline void normal4(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t expert,
                           uint32_t row, uint32_t col4, float out[4]) {
  const uint32_t ctr[4] = {col4, row, (kind << 24) | (expert & 0xFFFFFFu), layer};
  uint32_t r[4];
  wd_synth_philox4x32_10(seed, ctr, r);
  for (int p = 0; p < 2; ++p) {
    const double rad = sqrt(-2.0 * ln_pos(u01(r[2 * p])));
    double sn, cs;
    sincos_2pi(u01(r[2 * p + 1]), &sn, &cs);
    out[2 * p] = (float)(rad * cs);
    out[2 * p + 1] = (float)(rad * sn);
  }
}

/* Row of `cols` normals (std = `std_dev`), counter columns start at 0. */
static void normal_row(uint64_t seed, uint32_t layer, uint32_t kind, uint32_t expert,
                       uint32_t row, int cols, float std_dev, float* out) {
  float v[4];
  for (int c = 0; c < cols; c += 4) {
    normal4(seed, layer, kind, expert, row, (uint32_t)(c >> 2), v);
    for (int j = 0; j < 4 && c + j < cols; ++j) out[c + j] = std_dev * v[j];
  }
}

/* ------------------------------------------------------ number encoders ---- */

/* FP32 -> BF16 bits, round to nearest even (NaN kept quiet). */
WD_SYNTH_API uint16_t wd_synth_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static inline uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static inline float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* FP32 -> OCP E4M3 code, round to nearest even, saturating to +-448.
 * E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
 * 0x7F/0xFF are NaN; largest finite magnitude 448 = 1.75 * 2^8;
 * smallest subnormal 2^-9. */
WD_SYNTH_API uint8_t wd_synth_f32_to_e4m3(float q) {
  const uint32_t u = f32_bits(q);
  const uint8_t s = (uint8_t)((u >> 24) & 0x80u);
  const uint32_t mag = u & 0x7FFFFFFFu;
  if (mag > 0x7F800000u) return (uint8_t)(s | 0x7F);       /* NaN */
  if (mag >= 0x43E00000u) return (uint8_t)(s | 0x7E);      /* >= 448: saturate */
  if (mag < 0x3C800000u) {                                 /* below 2^-6: step 2^-9 */
    /* a * 512 < 8, so adding 2^23 rounds it to an integer, ties to even */
    const float m = (bits_f32(mag) * 512.0f + 8388608.0f) - 8388608.0f;
    return (uint8_t)(s | (uint8_t)m);                      /* 8 -> code 0x08 = 2^-6 */
  }
  /* normal: keep 3 of 23 mantissa bits, ties to even; a carry bumps the exponent */
  const uint32_t r = mag + 0x7FFFFu + ((mag >> 20) & 1u);
  const int e = (int)(r >> 23) - 127;                      /* -6 .. 8 */
  int code = ((e + 7) << 3) | (int)((r >> 20) & 7u);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(s | code);
}

/* One 32-element block: E8M0 scale code and E4M3 element codes.
 * scale exponent = floor(log2(amax)) - 8 clamped to [-127, 127];
 * amax == 0 gives scale code 127 (1.0) and all-zero elements. */
WD_SYNTH_API void wd_synth_quantise_block(const float* v, int n, uint8_t* codes, uint8_t* scale) {
  float amax = 0.0f;
  for (int j = 0; j < n; ++j) amax = fmaxf(amax, fabsf(v[j]));
  if (amax == 0.0f || isnan(amax)) {
    *scale = 127;
    for (int j = 0; j < n; ++j) codes[j] = 0;
    return;
  }
  int fl; /* floor(log2(amax)) */
  const uint32_t ab = f32_bits(amax);
  if (ab >= 0x00800000u) {
    fl = (int)(ab >> 23) - 127;
  } else {
    int ex;
    (void)frexpf(amax, &ex);
    fl = ex - 1;
  }
  int se = fl - 8;
  if (se < -127) se = -127;
  if (se > 127) se = 127;
  *scale = (uint8_t)(se + 127);
  /* v * 2^-se is exact: |v| * 2^-se < 512 and 2^-se is a normal float for se in [-127, 119] */
  const float inv = (se > -127) ? bits_f32((uint32_t)(127 - se) << 23) : 1.7014118346046923e38f;
  for (int j = 0; j < n; ++j) codes[j] = wd_synth_f32_to_e4m3(v[j] * inv);
}

/* ------------------------------------------------------------- weights ---- */

typedef struct {
  uint64_t seed;
  uint32_t layer, kind;
  int e0, e1;    /* experts [e0, e1) */
  int rows, cols;
  float std_dev;
  uint8_t* codes;  /* [E, rows, cols] (only [e0,e1) written)      */
  uint8_t* scales; /* [E, rows, cols/32]                           */
  float* raw;      /* optional [E, rows, cols] FP32 pre-quantisation */
  int t, nt;       /* this thread's share of the (expert,row) list  */
} mx_job;

static void* mx_worker(void* arg) {
  mx_job* j = (mx_job*)arg;
  float* row = (float*)malloc(sizeof(float) * (size_t)j->cols);
  const long total = (long)(j->e1 - j->e0) * j->rows;
  const long lo = total * j->t / j->nt, hi = total * (j->t + 1) / j->nt;
  for (long i = lo; i < hi; ++i) {
    const int e = j->e0 + (int)(i / j->rows), r = (int)(i % j->rows);
    normal_row(j->seed, j->layer, j->kind, (uint32_t)e, (uint32_t)r, j->cols, j->std_dev, row);
    const size_t off = ((size_t)e * j->rows + r) * (size_t)j->cols;
    const size_t soff = ((size_t)e * j->rows + r) * (size_t)(j->cols / 32);
    if (j->raw) memcpy(j->raw + off, row, sizeof(float) * (size_t)j->cols);
    for (int b = 0; b < j->cols / 32; ++b)
      wd_synth_quantise_block(row + 32 * b, 32, j->codes + off + 32 * (size_t)b, j->scales + soff + b);
  }
  free(row);
  return NULL;
}

static int run_mx(mx_job proto, int nthreads) {
  if (proto.cols % 32 != 0 || proto.rows <= 0 || proto.e1 <= proto.e0) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  mx_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].t = t;
    jobs[t].nt = nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, mx_worker, &jobs[t]) != 0) break;
    started = t;
  }
  mx_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) mx_worker(&jobs[t]); /* threads that failed to start */
  return 0;
}

/* gate_up codes [E, 2I, H] + scales [E, 2I, H/32] for experts [e0, e1).
 * Rows [0, I) are the gate projection, rows [I, 2I) the up projection;
 * both have fan_in = H, so std = 1/sqrt(H).  `raw` (optional) gets the FP32
 * values before quantisation, same layout as `codes`. */
WD_SYNTH_API int wd_synth_gate_up(uint64_t seed, uint32_t layer, int e0, int e1, int H, int I,
                                  uint8_t* codes, uint8_t* scales, float* raw, int nthreads) {
  mx_job j = {seed, layer, KIND_GATE_UP, e0, e1, 2 * I, H, 1.0f / sqrtf((float)H),
              codes, scales, raw, 0, 1};
  return run_mx(j, nthreads);
}

/* down codes [E, H, I] + scales [E, H, I/32]; fan_in = I, std = 1/sqrt(I). */
WD_SYNTH_API int wd_synth_down(uint64_t seed, uint32_t layer, int e0, int e1, int H, int I,
                               uint8_t* codes, uint8_t* scales, float* raw, int nthreads) {
  mx_job j = {seed, layer, KIND_DOWN, e0, e1, H, I, 1.0f / sqrtf((float)I),
              codes, scales, raw, 0, 1};
  return run_mx(j, nthreads);
}

/* ---------------------------------------------------------- activations ---- */

/* x [B, H] as BF16 bits, N(0,1); `raw` (optional) gets the FP32 draws. */
WD_SYNTH_API int wd_synth_x(uint64_t seed, uint32_t layer, int B, int H, uint16_t* x, float* raw) {
  float* row = (float*)malloc(sizeof(float) * (size_t)H);
  if (!row) return 1;
  for (int b = 0; b < B; ++b) {
    normal_row(seed, layer, KIND_X, 0, (uint32_t)b, H, 1.0f, row);
    for (int j = 0; j < H; ++j) {
      x[(size_t)b * H + j] = wd_synth_f32_to_bf16(row[j]);
      if (raw) raw[(size_t)b * H + j] = row[j];
    }
  }
  free(row);
  return 0;
}

/* --------------------------------------------------------------- router ---- */

/* Routing modes. */
enum {
  ROUTE_UNIFORM = 0,  /* logits ~ N(0,1)                                        */
  ROUTE_ZIPF = 1,     /* logits + log p_e, p_e proportional to (e+1)^-s          */
  ROUTE_FIXED = 2,    /* every token takes the K ids in `fixed`                  */
  ROUTE_DISJOINT = 3  /* tokens take disjoint K-blocks of seeded permutations    */
};

/* Seeded Fisher-Yates permutation of 0..n-1 (permutation number `p`). */
static void seeded_perm(uint64_t seed, uint32_t layer, uint32_t p, int n, int* perm) {
  for (int i = 0; i < n; ++i) perm[i] = i;
  for (int i = n - 1; i > 0; --i) {
    const uint32_t ctr[4] = {(uint32_t)i, p, (uint32_t)KIND_PERM << 24, layer};
    uint32_t r[4];
    wd_synth_philox4x32_10(seed, ctr, r);
    const uint64_t wide = ((uint64_t)r[0] << 32) | r[1];
    const int j = (int)(wide % (uint64_t)(i + 1));
    const int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
}

/* Router outputs for B tokens: ids [B,K] int32 and weights [B,K] FP32.
 * The logits of token b are row b of kind LOGITS.  Weights are the softmax of
 * the chosen experts' logits (softmax over E, keep the top K, renormalise to
 * sum 1 -- the same numbers).  `fixed` holds K ids for ROUTE_FIXED;
 * `zipf_s` is the exponent for ROUTE_ZIPF.  Returns 0 on success. */
WD_SYNTH_API int wd_synth_route(uint64_t seed, uint32_t layer, int B, int E, int K, int mode,
                                double zipf_s, const int32_t* fixed, int32_t* ids, float* w,
                                float* logits_out) {
  if (K < 1 || K > E || B < 0) return 1;
  if (mode == ROUTE_DISJOINT && E % K != 0) return 1;
  float* lg = (float*)malloc(sizeof(float) * (size_t)E);
  int* order = (int*)malloc(sizeof(int) * (size_t)E);
  int* perm = (int*)malloc(sizeof(int) * (size_t)E);
  if (!lg || !order || !perm) return 2;
  double zsum = 0.0;
  if (mode == ROUTE_ZIPF)
    for (int e = 0; e < E; ++e) zsum += pow((double)(e + 1), -zipf_s);
  int cur_perm = -1;
  for (int b = 0; b < B; ++b) {
    normal_row(seed, layer, KIND_LOGITS, 0, (uint32_t)b, E, 1.0f, lg);
    if (mode == ROUTE_ZIPF)
      for (int e = 0; e < E; ++e) lg[e] += (float)log(pow((double)(e + 1), -zipf_s) / zsum);
    if (logits_out) memcpy(logits_out + (size_t)b * E, lg, sizeof(float) * (size_t)E);
    int32_t* id = ids + (size_t)b * K;
    if (mode == ROUTE_FIXED) {
      for (int k = 0; k < K; ++k) id[k] = fixed[k];
    } else if (mode == ROUTE_DISJOINT) {
      const int per = E / K; /* tokens served by one permutation */
      const int p = b / per, blk = b % per;
      if (p != cur_perm) {
        seeded_perm(seed, layer, (uint32_t)p, E, perm);
        cur_perm = p;
      }
      for (int k = 0; k < K; ++k) id[k] = perm[blk * K + k];
    } else {
      /* top-K by logit, ties to the lower id: selection by repeated argmax */
      for (int e = 0; e < E; ++e) order[e] = 0;
      for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!order[e] && (best < 0 || lg[e] > lg[best])) best = e;
        order[best] = 1;
        id[k] = best;
      }
    }
    double mx = -INFINITY, sum = 0.0;
    for (int k = 0; k < K; ++k) mx = fmax(mx, (double)lg[id[k]]);
    for (int k = 0; k < K; ++k) sum += exp((double)lg[id[k]] - mx);
    for (int k = 0; k < K; ++k) w[(size_t)b * K + k] = (float)(exp((double)lg[id[k]] - mx) / sum);
  }
  free(lg);
  free(order);
  free(perm);
  return 0;
}

/*
 * wd_oracle.c - CPU oracle for the small-batch MoE decode layer.
 *
 * TEST INFRASTRUCTURE.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library never
 * does, and it shares no code (no headers, helpers or tables) with the CUDA
 * kernels.
 *
 * What it computes (Cursor, "用 warp decode 实现更好的 MoE 模型推理"
 * [Better MoE inference with warp decode], section 两个 kernel 如何工作
 * [How the two kernels work], and section 精度提升 [Accuracy gains] for the
 * precision regime: BF16 activations, MXFP8 weights dequantised to real numbers,
 * wide accumulation):
 *
 *   for every token b and routed slot k (e = ids[b,k]), every neuron n < I:
 *       g = sum_j dq(gate_up[e, n,   j]) * x[b, j]
 *       u = sum_j dq(gate_up[e, I+n, j]) * x[b, j]
 *       h[b,k,n] = bf16( silu(g) * u ),  silu(g) = g / (1 + exp(-g))
 *   for every token b and output dim d < H:
 *       y[b,d] = sum_k w[b,k] * sum_i dq(down[e_k, d, i]) * h[b,k,i]
 *       out[b,d] = bf16(y[b,d])
 *
 * with dq(code at column j of a row) = E4M3(code) * E8M0(scale of that row at
 * column block j/32).  Everything is accumulated in FP64 (a superset of the
 * blog's FP32), in plain loops in the order written above.  h is rounded to
 * BF16 once, because the layer hands one BF16 value per neuron from the first
 * projection to the second (section 两个 kernel 如何工作: the gate/up warp
 * "writes out one intermediate value").
 *
 * Number formats (OCP Microscaling Formats (MX) Specification v1.0, section
 * on the E4M3 element format and the E8M0 scale format):
 *   E4M3 bits s eeee mmm, bias 7: e = 0 -> (-1)^s 2^-6 (m/8);
 *        otherwise (-1)^s 2^(e-7) (1 + m/8); s 1111 111 is NaN; no infinities.
 *   E8M0: code c -> 2^(c-127); c = 255 is NaN.
 *   BF16: the top 16 bits of an IEEE binary32; rounding to it is to nearest,
 *        ties to even, from the exact FP64 value (one rounding).
 *
 * Boundary behaviour (the library's documented contract, restated): an expert
 * id outside [0, E) contributes nothing (its h entries are 0) and is counted
 * in the returned number of bad ids.
 *
 * Parity status: every function here is pinned by tests that do not call it
 * twice (decode tables against an independent FP8 implementation, BF16 rounding
 * against exhaustive nearest-value search, the layer against a brute-force dense
 * evaluation over all experts, closed forms and invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------ formats ---- */

ORACLE_API double oracle_e4m3(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 0xF, m = code & 0x7;
  if (e == 0xF && m == 0x7) return NAN;
  const double mag = (e == 0) ? ldexp((double)m, -9)          /* 2^-6 * m/8      */
                              : ldexp((double)(8 + m), e - 10); /* 2^(e-7)(1+m/8) */
  return s ? -mag : mag;
}

ORACLE_API double oracle_e8m0(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

ORACLE_API double oracle_bf16_to_f64(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* FP64 -> BF16 bits, round to nearest, ties to even, single rounding. */
ORACLE_API uint16_t oracle_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  const uint16_t s = signbit(v) ? 0x8000 : 0x0000;
  const double a = fabs(v);
  if (a == 0.0) return s;
  if (isinf(a)) return (uint16_t)(s | 0x7F80);
  if (a < 0x1p-126) { /* subnormal: multiples of 2^-133 */
    const double q = nearbyint(a * 0x1p133); /* 0..128; 128 is the smallest normal */
    return (uint16_t)(s | (uint16_t)q);
  }
  int ex;
  const double fr = frexp(a, &ex);  /* a = fr 2^ex, fr in [0.5, 1) */
  int E = ex - 1;                   /* a in [2^E, 2^(E+1)) */
  double m = nearbyint((2.0 * fr - 1.0) * 128.0); /* 7 fraction bits */
  if (m == 128.0) {
    m = 0.0;
    E += 1;
  }
  if (E > 127) return (uint16_t)(s | 0x7F80); /* rounds past the largest finite value */
  return (uint16_t)(s | (uint16_t)((E + 127) << 7) | (uint16_t)m);
}

ORACLE_API double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* The two decode functions above, tabulated once when the library loads
 * (each entry is exactly the function's value for that code). */
static double e4m3_value[256], e8m0_value[256];

__attribute__((constructor)) static void fill_decode_tables(void) {
  for (int c = 0; c < 256; ++c) {
    e4m3_value[c] = oracle_e4m3((uint8_t)c);
    e8m0_value[c] = oracle_e8m0((uint8_t)c);
  }
}

/* Dequantised element (row r, column j) of an MXFP8 matrix whose rows hold
 * `cols` codes and cols/32 scales. */
static double dq(const uint8_t* codes, const uint8_t* scales, long row, int cols, int j) {
  return e4m3_value[codes[row * cols + j]] * e8m0_value[scales[row * (cols / 32) + j / 32]];
}

/* ------------------------------------------------------------ the layer ---- */

/* First projection.  x: BF16 bits [B,H]; ids: [B,K]; gate_up: codes [E,2I,H],
 * gate_up_scale: [E,2I,H/32].  Writes h: BF16 bits [B,K,I] and, if non-null,
 * h_f64 [B,K,I] = silu(g)*u before rounding.  Returns the number of bad ids. */
ORACLE_API long oracle_gate_up(const uint16_t* x, const int32_t* ids, const uint8_t* gate_up,
                               const uint8_t* gate_up_scale, int B, int H, int I, int E, int K,
                               uint16_t* h, double* h_f64) {
  long bad = 0;
  for (int b = 0; b < B; ++b) {
    for (int k = 0; k < K; ++k) {
      const int e = ids[b * K + k];
      const int valid = (e >= 0 && e < E);
      bad += !valid;
      for (int n = 0; n < I; ++n) {
        double val = 0.0;
        if (valid) {
          const long gate_row = (long)e * 2 * I + n;
          const long up_row = (long)e * 2 * I + I + n;
          double g = 0.0, u = 0.0;
          for (int j = 0; j < H; ++j) {
            const double xj = oracle_bf16_to_f64(x[(long)b * H + j]);
            g += dq(gate_up, gate_up_scale, gate_row, H, j) * xj;
            u += dq(gate_up, gate_up_scale, up_row, H, j) * xj;
          }
          val = oracle_silu(g) * u;
        }
        const long o = ((long)b * K + k) * I + n;
        h[o] = oracle_f64_to_bf16(val);
        if (h_f64) h_f64[o] = val;
      }
    }
  }
  return bad;
}

/* Second projection with the weighted top-k fold.  h: BF16 bits [B,K,I];
 * ids, w: [B,K]; down: codes [E,H,I], down_scale: [E,H,I/32].  Writes
 * out: BF16 bits [B,H] and, if non-null, y [B,H] before rounding. */
ORACLE_API long oracle_down(const uint16_t* h, const int32_t* ids, const float* w,
                            const uint8_t* down, const uint8_t* down_scale, int B, int H, int I,
                            int E, int K, uint16_t* out, double* y_f64) {
  long bad = 0;
  for (int b = 0; b < B; ++b)
    for (int k = 0; k < K; ++k) bad += !(ids[b * K + k] >= 0 && ids[b * K + k] < E);
  for (int b = 0; b < B; ++b) {
    for (int d = 0; d < H; ++d) {
      double y = 0.0;
      for (int k = 0; k < K; ++k) {
        const int e = ids[b * K + k];
        if (e < 0 || e >= E) continue;
        const long row = (long)e * H + d;
        double dot = 0.0;
        for (int i = 0; i < I; ++i)
          dot += dq(down, down_scale, row, I, i) * oracle_bf16_to_f64(h[((long)b * K + k) * I + i]);
        y += (double)w[b * K + k] * dot;
      }
      out[(long)b * H + d] = oracle_f64_to_bf16(y);
      if (y_f64) y_f64[(long)b * H + d] = y;
    }
  }
  return bad;
}

/* The whole layer: first projection, then the second.  `h` (BF16 bits
 * [B,K,I]) is caller-provided scratch and holds the intermediate on return. */
ORACLE_API long oracle_moe_decode(const uint16_t* x, const int32_t* ids, const float* w,
                                  const uint8_t* gate_up, const uint8_t* gate_up_scale,
                                  const uint8_t* down, const uint8_t* down_scale, int B, int H,
                                  int I, int E, int K, uint16_t* h, uint16_t* out, double* y_f64) {
  const long bad = oracle_gate_up(x, ids, gate_up, gate_up_scale, B, H, I, E, K, h, NULL);
  oracle_down(h, ids, w, down, down_scale, B, H, I, E, K, out, y_f64);
  return bad;
}

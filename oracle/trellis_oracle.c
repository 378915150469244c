/*
 * trellis_oracle.c -- plain, slow, obviously correct CPU reference for linear
 * layers over packed trellis-coded ("QTIP 1MAD") weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  The product path (the CUDA library
 * and its Python binding) never calls it and shares no code with it.
 *
 * Source: the "mlx-bun 0.2.0 -> 0.4.0" diff pages of trellis-linear.ts (the
 * file's header comment on the packed linear layer, and its kernel sources)
 * and of trellis-tiled-prefill.ts / trellis-vector-expand.ts.
 *
 * What is computed, in the pages' order:
 *   format   .weight is a uint32 bitstream [rows, cols*k/32], .scales is fp16
 *            [rows], one scale per stored row (trellis-linear.ts header).
 *   state    state_t of a T-long block is the L-bit window that starts at bit
 *            (T-1-t)*k of the block, bits read least-significant first inside
 *            little-endian words, wrapping to the start of the same block
 *            (trellis-linear.ts header; HEADER, trellis_state).
 *   code     1MAD: x = s*34038481 + 76625530 (mod 2^32), y = (sum of the four
 *            bytes of x) - 510; value = y / 147.800537109375
 *            (HEADER, trellis_y / trellis_val).
 *   expand   out[r][c] = bf16(value(s(r,c)) * scale[r]) with a correctly
 *            rounded value (EXPAND_SOURCE; trellis-vector-expand.ts).
 *   matvec   weights are fp32 value*scale with no bf16 rounding (the default
 *            decoder, "variant 6", in HEADER); axis 1 sums over stored columns
 *            (REDUCE_SOURCE), axis 0 over stored rows (SCATTER_SOURCE).
 *   gate/up  two axis-1 matvecs, then bf16 casts at gate, up, sigmoid, silu and
 *            product (GATEUP_SOURCE).
 *   prefill  out[m][r] = sum_c bf16 expand weight * x (trellis-tiled-prefill.ts).
 *
 * Arithmetic: window bits are collected one bit at a time; the four bytes of
 * x are taken by division and remainder by 256; sums run in double.  Build
 * with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_A 34038481u
#define OR_B 76625530u
#define OR_D 147.800537109375f

/* ---------- geometry ---------------------------------------------------- */

/* 0 if (k, L, T, rows, cols) describe a packed matrix the oracle can read:
 * T*k a whole number of 32-bit words, cols a whole number of blocks
 * (trellisGeometry in trellis-linear.ts), 1 <= k <= 8, 1 <= L <= 32. */
int or_geom_check(int k, int L, int T, int64_t rows, int64_t cols) {
  if (k < 1 || k > 8) return -1;
  if (L < 1 || L > 32) return -1;
  if (T < 1 || ((int64_t)T * k) % 32 != 0) return -1;
  if (rows < 1 || cols < 1 || cols % T != 0) return -1;
  return 0;
}

static int64_t words_per_block(int T, int k) { return (int64_t)T * k / 32; }

/* ---------- bit access and state ---------------------------------------- */

/* Bit j (0 <= j < T*k) of a block: LSB-first inside little-endian words. */
static uint32_t block_bit(const uint32_t *block, int64_t j) {
  return (block[j / 32] >> (j % 32)) & 1u;
}

/* state_t: L bits starting at (T-1-t)*k, wrapping inside the block. */
uint32_t or_state(const uint32_t *block, int T, int k, int L, int t) {
  const int64_t nbits = (int64_t)T * k;
  const int64_t start = (int64_t)(T - 1 - t) * k;
  uint64_t s = 0;
  for (int i = 0; i < L; ++i) {
    const int64_t j = (start + i) % nbits;
    s |= (uint64_t)block_bit(block, j) << i;
  }
  return (uint32_t)s;
}

/* ---------- the 1MAD code ---------------------------------------------- */

/* y(s): x = s*a + b mod 2^32, y = sum of the four bytes of x minus 510. */
int or_code_y(uint32_t s) {
  uint64_t x = ((uint64_t)s * (uint64_t)OR_A + (uint64_t)OR_B) % 4294967296ull;
  int sum = 0;
  for (int i = 0; i < 4; ++i) {
    sum += (int)(x % 256u);
    x /= 256u;
  }
  return sum - 510;
}

/* value(y) = y / d, one IEEE single-precision division (correctly rounded). */
float or_code_val(int y) {
  volatile float num = (float)y;
  volatile float den = OR_D;
  return num / den;
}

/* Table of y and value for every state s < 2^L (L <= 24), built by a second
 * route that shares nothing with or_code_y: x is walked through the states
 * by repeated addition of a in 32-bit unsigned arithmetic (x(0) = b,
 * x(s+1) = x(s) + a, wrapping mod 2^32), and the byte sum is the "two
 * byte-pair adds" form of the HEADER source's trellis_y: add the even bytes
 * to the odd bytes as two 16-bit lanes, then add the two lanes.  Tests
 * compare this table with or_code_y over every state. */
void or_lut(int L, int32_t *ytab, float *vtab) {
  const uint32_t n = 1u << L;
  uint32_t x = OR_B;
  for (uint32_t s = 0; s < n; ++s, x += OR_A) {
    const uint32_t pairs = (x & 0x00FF00FFu) + ((x >> 8) & 0x00FF00FFu); /* two lanes, each <= 510 */
    const int y = (int)((pairs & 0xFFFFu) + (pairs >> 16)) - 510;
    if (ytab) ytab[s] = y;
    if (vtab) vtab[s] = or_code_val(y);
  }
}

/* ---------- number formats ---------------------------------------------- */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* fp16 storage bits -> fp32 value (exact; handles subnormals, inf, nan). */
float or_f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) & 1u;
  const uint32_t e = (uint32_t)(h >> 10) & 31u;
  const uint32_t m = (uint32_t)h & 1023u;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024u + m), (int)e - 25);
  return (float)(sign ? -v : v);
}

/* bf16 storage bits -> fp32 value (exact). */
float or_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* fp32 -> bf16 storage bits, round to nearest, ties to even.  The kept part
 * is the upper half of the fp32 pattern; it is bumped by one when the
 * discarded half is above one half, or exactly one half with an odd kept
 * part.  NaN stays NaN. */
uint16_t or_bf16_rne(float v) {
  const uint32_t u = f32_to_bits(v);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t keep = u >> 16;
  const uint32_t rest = u & 0xFFFFu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

/* double -> bf16 bits, rounding once (nearest, ties to even). */
uint16_t or_bf16_rne_f64(double v) {
  if (isnan(v)) return 0x7FC0u;
  const uint16_t sgn = (uint16_t)(signbit(v) ? 0x8000u : 0u);
  double a = fabs(v);
  if (a == 0.0) return sgn;
  /* candidates: truncate the fp32 nearest-below to bf16, then the next one */
  float f = (float)a;               /* nearest fp32 */
  if ((double)f > a) f = nextafterf(f, 0.0f);  /* largest fp32 <= a */
  uint32_t lo = f32_to_bits(f) >> 16;          /* bf16 <= a */
  const double vlo = (double)bits_to_f32(lo << 16);
  const double vhi = (double)bits_to_f32((lo + 1u) << 16);
  uint32_t pick;
  if (a - vlo < vhi - a) pick = lo;
  else if (a - vlo > vhi - a) pick = lo + 1u;
  else pick = (lo & 1u) ? lo + 1u : lo;
  return (uint16_t)(sgn | pick);
}

/* ---------- decoded weights --------------------------------------------- */

static const uint32_t *block_ptr(const uint32_t *codes, int T, int k, int64_t cols,
                                 int64_t r, int64_t c) {
  const int64_t wpb = words_per_block(T, k);
  return codes + r * (cols / T) * wpb + (c / T) * wpb;
}

/* The correctly rounded value of stored entry (r, c), before scaling. */
static float entry_value(const uint32_t *codes, int T, int k, int L, int64_t cols,
                         int64_t r, int64_t c) {
  const uint32_t s = or_state(block_ptr(codes, T, k, cols, r, c), T, k, L, (int)(c % T));
  return or_code_val(or_code_y(s));
}

/* Packed-matvec weight: fp32 value * fp32 scale, not rounded to bf16. */
static float entry_weight_f32(const uint32_t *codes, const uint16_t *scales, int T, int k,
                              int L, int64_t cols, int64_t r, int64_t c) {
  volatile float v = entry_value(codes, T, k, L, cols, r, c);
  volatile float s = or_f16_to_f32(scales[r]);
  return v * s;
}

/* States, y values or fp32 matvec weights of a list of stored rows
 * (out is [n_rows, cols]); any of the three outputs may be NULL. */
void or_decode_rows(const uint32_t *codes, const uint16_t *scales, int k, int L, int T,
                    int64_t rows, int64_t cols, const int64_t *row_idx, int64_t n_rows,
                    uint32_t *states, int32_t *ys, float *weights) {
  (void)rows;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = row_idx[i];
    for (int64_t c = 0; c < cols; ++c) {
      const uint32_t s = or_state(block_ptr(codes, T, k, cols, r, c), T, k, L, (int)(c % T));
      if (states) states[i * cols + c] = s;
      if (ys) ys[i * cols + c] = or_code_y(s);
      if (weights) weights[i * cols + c] = entry_weight_f32(codes, scales, T, k, L, cols, r, c);
    }
  }
}

/* ---------- expand ------------------------------------------------------- */

/* out[i][c] = bf16(fl32(value(s(r,c)) * scale[r])) for r = row_idx[i]. */
void or_expand_bf16(const uint32_t *codes, const uint16_t *scales, int k, int L, int T,
                    int64_t rows, int64_t cols, const int64_t *row_idx, int64_t n_rows,
                    uint16_t *out) {
  (void)rows;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = row_idx[i];
    for (int64_t c = 0; c < cols; ++c)
      out[i * cols + c] = or_bf16_rne(entry_weight_f32(codes, scales, T, k, L, cols, r, c));
  }
}

/* ---------- matvec along axis 1 (reduce over stored columns) ------------- */

/* ref[m][i] = sum_c w(r,c) x[m][c] and absum[m][i] = sum_c |w(r,c) x[m][c]|
 * for r = row_idx[i]; w is the fp32 packed-matvec weight; sums in double.
 * x is bf16 [M, cols]; ref/absum are [M, n_rows]. */
void or_matvec_axis1(const uint32_t *codes, const uint16_t *scales, const uint16_t *x, int M,
                     int k, int L, int T, int64_t rows, int64_t cols, const int64_t *row_idx,
                     int64_t n_rows, double *ref, double *absum) {
  (void)rows;
  float *w = (float *)malloc(sizeof(float) * (size_t)cols);
  if (!w) return;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = row_idx[i];
    for (int64_t c = 0; c < cols; ++c) w[c] = entry_weight_f32(codes, scales, T, k, L, cols, r, c);
    for (int m = 0; m < M; ++m) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t c = 0; c < cols; ++c) {
        const double p = (double)w[c] * (double)or_bf16_to_f32(x[(int64_t)m * cols + c]);
        acc += p;
        aacc += fabs(p);
      }
      ref[(int64_t)m * n_rows + i] = acc;
      absum[(int64_t)m * n_rows + i] = aacc;
    }
  }
  free(w);
}

/* ---------- matvec along axis 0 (reduce over stored rows) ---------------- */

/* The stored matrix is W^T [rows = in, cols = out].  For c = col_idx[j]:
 * ref[m][j] = sum_r w(r,c) x[m][r], absum likewise with |.|.
 * x is bf16 [M, rows]; ref/absum are [M, n_cols]. */
void or_matvec_axis0(const uint32_t *codes, const uint16_t *scales, const uint16_t *x, int M,
                     int k, int L, int T, int64_t rows, int64_t cols, const int64_t *col_idx,
                     int64_t n_cols, double *ref, double *absum) {
  float *w = (float *)malloc(sizeof(float) * (size_t)rows);
  if (!w) return;
  for (int64_t j = 0; j < n_cols; ++j) {
    const int64_t c = col_idx[j];
    for (int64_t r = 0; r < rows; ++r) w[r] = entry_weight_f32(codes, scales, T, k, L, cols, r, c);
    for (int m = 0; m < M; ++m) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t r = 0; r < rows; ++r) {
        const double p = (double)w[r] * (double)or_bf16_to_f32(x[(int64_t)m * rows + r]);
        acc += p;
        aacc += fabs(p);
      }
      ref[(int64_t)m * n_cols + j] = acc;
      absum[(int64_t)m * n_cols + j] = aacc;
    }
  }
  free(w);
}

/* Axis-0 matvec with the bf16-rounded weight numerics (decoder variants 0-3
 * of the HEADER source): w = bf16(fl32(value * scale)), the expand weight. */
void or_matvec_axis0_bf16w(const uint32_t *codes, const uint16_t *scales, const uint16_t *x, int M, int k,
                           int L, int T, int64_t rows, int64_t cols, const int64_t *col_idx, int64_t n_cols,
                           double *ref, double *absum) {
  double *w = (double *)malloc(sizeof(double) * (size_t)rows);
  if (!w) return;
  for (int64_t j = 0; j < n_cols; ++j) {
    const int64_t c = col_idx[j];
    for (int64_t r = 0; r < rows; ++r)
      w[r] = (double)or_bf16_to_f32(or_bf16_rne(entry_weight_f32(codes, scales, T, k, L, cols, r, c)));
    for (int m = 0; m < M; ++m) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t r = 0; r < rows; ++r) {
        const double p = w[r] * (double)or_bf16_to_f32(x[(int64_t)m * rows + r]);
        acc += p;
        aacc += fabs(p);
      }
      ref[(int64_t)m * n_cols + j] = acc;
      absum[(int64_t)m * n_cols + j] = aacc;
    }
  }
  free(w);
}

/* ---------- fused gate/up SwiGLU ---------------------------------------- */

/* The activation chain on bf16 gate and up values, evaluated in fp32 with
 * a bf16 rounding after every step: sigmoid = bf16(1 / (1 + exp(-g))),
 * silu = bf16(g * sigmoid), out = bf16(silu * u). */
uint16_t or_swiglu_bf16(uint16_t g_bits, uint16_t u_bits) {
  volatile float g = or_bf16_to_f32(g_bits);
  volatile float u = or_bf16_to_f32(u_bits);
  volatile float e = expf(-g);
  volatile float den = 1.0f + e;
  volatile float sig = or_bf16_to_f32(or_bf16_rne(1.0f / den));
  volatile float silu = or_bf16_to_f32(or_bf16_rne(g * sig));
  volatile float prod = silu * u;
  return or_bf16_rne(prod);
}

void or_swiglu_bf16_many(const uint16_t *g, const uint16_t *u, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_swiglu_bf16(g[i], u[i]);
}

/* Gate and up sums of the fused layer for r = row_idx[i] (each an axis-1
 * matvec with fp32 packed weights); outputs [M, n_rows] in double. */
void or_gateup_sums(const uint32_t *gcodes, const uint16_t *gscales, const uint32_t *ucodes,
                    const uint16_t *uscales, const uint16_t *x, int M, int k, int L, int T,
                    int64_t rows, int64_t cols, const int64_t *row_idx, int64_t n_rows,
                    double *gref, double *gabs, double *uref, double *uabs) {
  or_matvec_axis1(gcodes, gscales, x, M, k, L, T, rows, cols, row_idx, n_rows, gref, gabs);
  or_matvec_axis1(ucodes, uscales, x, M, k, L, T, rows, cols, row_idx, n_rows, uref, uabs);
}

/* ---------- prefill GEMM ------------------------------------------------- */

/* ref[m][i] = sum_c e(r,c) x[m][c] for r = row_idx[i], with e the bf16
 * expand weight (the prefill's numerical contract); absum likewise. */
void or_prefill(const uint32_t *codes, const uint16_t *scales, const uint16_t *x, int M, int k,
                int L, int T, int64_t rows, int64_t cols, const int64_t *row_idx, int64_t n_rows,
                double *ref, double *absum) {
  (void)rows;
  double *e = (double *)malloc(sizeof(double) * (size_t)cols);
  if (!e) return;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = row_idx[i];
    for (int64_t c = 0; c < cols; ++c)
      e[c] = (double)or_bf16_to_f32(or_bf16_rne(entry_weight_f32(codes, scales, T, k, L, cols, r, c)));
    for (int m = 0; m < M; ++m) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t c = 0; c < cols; ++c) {
        const double p = e[c] * (double)or_bf16_to_f32(x[(int64_t)m * cols + c]);
        acc += p;
        aacc += fabs(p);
      }
      ref[(int64_t)m * n_rows + i] = acc;
      absum[(int64_t)m * n_rows + i] = aacc;
    }
  }
  free(e);
}

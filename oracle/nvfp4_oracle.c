/*
 * NVFP4 FC2 oracle: a plain, slow CPU restatement of the FC2 step of the
 * video DiT MLP (SwiGLU -> two-pass NVFP4 quantisation -> block-scaled GEMM).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can check the CUDA library against an
 * independent definition.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Sources (page title, section):
 *   - "FC2 NVFP4 Scheduling Results", Canonical Operation: the GEMM shape,
 *     E2M1 elements with vector-16 UE4M3 block scales, FP32 accumulation and
 *     scalars, BF16 output, producer padding of M.
 *   - "GB10 component-2 nsys summary", nvfp4 (absmax_partial ->
 *     scale_finalize -> block_scale_zero -> activation_pack: the two-pass
 *     order, global scale before block scales) and native_pack_validation
 *     (the general 128-row by 4-scale-column tiled scale offset).
 *   - "GB10 component-2 nsys summary", other_boundaries (unfused SwiGLU:
 *     a separate BF16 silu and a separate BF16 multiply).
 *   - The two-level NVFP4 recipe (not printed on the pages):
 *     global = amax/(6*448), block = RNE-E4M3(block_amax/(6*global)),
 *     element = RNE-E2M1(x/(block*global)).
 *
 * Readings where the pages are silent:
 *   - silu is rounded once, correctly, to BF16; the SwiGLU product
 *     (exact in binary32) is rounded once to BF16; gate = columns [0,K),
 *     up = columns [K,2K).
 *   - 6*global is formed first, then block_amax is divided by it.
 *   - element codes keep the sign of zero; a zero scale gives code 0x0.
 *   - even element in the low nibble.
 *   - rows padded to a multiple of 128, pad rows and pad scale columns zero.
 *   - a non-finite amax gives status 4, global scale NaN, all-zero output.
 *
 * Parity pins live in tests/test_oracle_pins.py (brute-force code tables,
 * hand-worked blocks, round-trip bounds, closed-form byte counts, an
 * independent FP64 matmul on tiny shapes) and tests/test_gpu_pins.py: the
 * nibble order, which a GEMM of two packed operands cannot show (the same
 * swap in both cancels), against the tensor core's own reading of these
 * bytes; the tiled scale layout against a library's block-scaled NVFP4
 * matmul on these bytes.
 *
 * Arithmetic: every float operation below is one IEEE binary32 (or binary64
 * where stated) operation; build with -ffp-contract=off so that no two are
 * fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENONFINITE 4

typedef struct {
  float global_scale;
  uint32_t amax_bits;
  uint32_t status;
  uint32_t pad;
} oracle_scale_rec;

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------- BF16 ---------------------------------------------------- */

float oracle_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Round a binary32 value to the nearest BF16, ties to the even significand.
 * Written as "choose the nearer of the two neighbours": lo keeps the upper 16
 * bits (truncation toward zero), hi is the next BF16 away from zero. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
  uint32_t lo = u & 0xFFFF0000u;
  uint32_t rem = u & 0x0000FFFFu;
  uint16_t lo16 = (uint16_t)(lo >> 16);
  if (rem < 0x8000u) return lo16;
  if (rem > 0x8000u) return (uint16_t)(lo16 + 1u);
  return (lo16 & 1u) ? (uint16_t)(lo16 + 1u) : lo16; /* tie: even significand */
}

/* ---------------- E2M1 (element format) ------------------------------------ */

/* Value of a 4-bit E2M1 code from its bit fields: bit 3 sign, bits 2..1
 * exponent (bias 1), bit 0 mantissa.  Exponent 0 is subnormal: m * 0.5. */
double oracle_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Round-to-nearest-even into E2M1 with saturation to +-6 (satfinite).
 * Nearest magnitude among the eight codes 0..7; on a tie the even code wins.
 * The sign bit is copied from q, so -0 and small negatives give 0x8. */
int oracle_e2m1_encode(float q) {
  double a = fabs((double)q);
  int best = 0;
  double best_d = INFINITY;
  if (a > 6.0) {
    best = 7;
  } else {
    for (int c = 0; c < 8; ++c) {
      double d = fabs(a - oracle_e2m1_value(c));
      if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
        best = c;
        best_d = d;
      }
    }
  }
  return best | (signbit(q) ? 8 : 0);
}

/* ---------------- E4M3 (block-scale format, E4M3FN) ------------------------ */

/* Value of an 8-bit E4M3FN code: bit 7 sign, bits 6..3 exponent (bias 7),
 * bits 2..0 mantissa; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is
 * NaN; the largest finite magnitude is 448. */
double oracle_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp((double)m, -9);
  else mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Round-to-nearest-even into E4M3FN, saturating finite values above 448 to
 * 448 (code 0x7E).  Nearest magnitude among codes 0x00..0x7E, ties to the
 * even code; the sign bit is copied.  NaN maps to 0x7F. */
int oracle_e4m3_encode(float r) {
  if (isnan(r)) return 0x7F;
  double a = fabs((double)r);
  int best = 0;
  if (a >= 448.0) {
    best = 0x7E;
  } else {
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
      double d = fabs(a - oracle_e4m3_value(c));
      if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
        best = c;
        best_d = d;
      }
    }
  }
  return best | (signbit(r) ? 0x80 : 0);
}

/* ---------------- SwiGLU ---------------------------------------------------- */

/* BF16 silu, correctly rounded: silu(g) = g / (1 + e^-g) taken exactly and
 * rounded once to BF16 (nearest, ties to even).  Evaluated in binary64;
 * a result within 2^-40 (relative) of a BF16 midpoint is a near tie and is
 * settled by the fact silu(g) > g/2 for g != 0: the only near ties are the
 * ones where binary64 returns g/2 exactly (|g| tiny), and then the exact
 * value lies above the midpoint.  Any other near tie is reported through
 * *unresolved (the pin test asserts there is none).
 * Non-finite gates: silu(+inf) = +inf; silu(-inf) and silu(NaN) are NaN, so
 * a non-finite input always makes the SwiGLU output non-finite. */
static uint16_t silu_bf16_impl(uint16_t gb, int* unresolved) {
  float gf = oracle_bf16_to_f32(gb);
  if (isnan(gf)) return 0x7FC0;
  if (isinf(gf)) return gf > 0 ? 0x7F80 : 0x7FC0;
  if (gf == 0.0f) return gb; /* silu(+-0) = +-0 */
  double g = (double)gf;
  double v = g / (1.0 + exp(-g));
  if (v == 0.0) return (uint16_t)(signbit(v) ? 0x8000 : 0x0000);
  /* Neighbours of v in BF16: truncate to BF16 toward zero (lo) and step one
   * unit away from zero (hi).  v is below 2^128 in magnitude because
   * |silu(g)| <= |g| for every g. */
  float vf = (float)v; /* only used to read the binade; the decision is in double */
  uint32_t vb = f32_bits(vf);
  uint16_t lo16 = (uint16_t)(vb >> 16);
  double lo = (double)oracle_bf16_to_f32(lo16);
  if (fabs(lo) > fabs(v)) { lo16 = (uint16_t)(lo16 - 1u); lo = (double)oracle_bf16_to_f32(lo16); }
  if (lo == v) return lo16; /* already a BF16 value (also keeps hi finite below) */
  uint16_t hi16 = (uint16_t)(lo16 + 1u);
  double hi = (double)oracle_bf16_to_f32(hi16);
  double mid = 0.5 * (lo + hi);
  double dist = fabs(v) - fabs(mid);
  if (fabs(dist) <= ldexp(fabs(mid), -40)) {
    if (fabs(g) < 0x1p-60) {
      /* exact value is above v = g/2: toward +inf */
      return (v > 0) ? hi16 : lo16;
    }
    if (unresolved) *unresolved += 1;
  }
  if (dist < 0) return lo16;
  if (dist > 0) return hi16;
  return (lo16 & 1u) ? hi16 : lo16;
}

uint16_t oracle_silu_bf16(uint16_t g) { return silu_bf16_impl(g, NULL); }

/* Fill a 65536-entry table of correctly rounded BF16 silu; returns the
 * number of unresolved near ties (expected 0). */
int oracle_silu_table(uint16_t* out) {
  int unresolved = 0;
  for (uint32_t g = 0; g < 65536u; ++g) out[g] = silu_bf16_impl((uint16_t)g, &unresolved);
  return unresolved;
}

/* h = RNE_bf16(float(silu_bf16(g)) * float(u)); the product of two BF16
 * values is exact in binary32, so there is one rounding. */
uint16_t oracle_swiglu_bf16(uint16_t g, uint16_t u, const uint16_t* silu_tab) {
  float s = oracle_bf16_to_f32(silu_tab ? silu_tab[g] : oracle_silu_bf16(g));
  float p = s * oracle_bf16_to_f32(u);
  return oracle_f32_to_bf16(p);
}

/* h [rows, cols] (row stride cols) = the SwiGLU of every element of a
 * gate|up matrix x [rows, ld] (gate in columns [0, cols), up in [cols,
 * 2 cols)): h = RNE_bf16(silu_bf16(g) * u) as above, the tensor the
 * producer quantises ("GB10 component-2 nsys summary", other_boundaries: a
 * BF16 silu, then a BF16 multiply). */
int oracle_swiglu_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint16_t* h) {
  if (!x || !h || rows < 0 || cols < 1 || ld < 2 * cols) return ORACLE_EINVAL;
  uint16_t* silu_tab = (uint16_t*)malloc(65536 * sizeof(uint16_t));
  if (!silu_tab) return ORACLE_EINVAL;
  oracle_silu_table(silu_tab);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < cols; ++j)
      h[r * cols + j] = oracle_swiglu_bf16(x[r * ld + j], x[r * ld + cols + j], silu_tab);
  free(silu_tab);
  return ORACLE_OK;
}

/* ---------------- Sizes and the scale layout ------------------------------- */

int64_t oracle_padded_rows(int64_t rows) { return (rows + 127) / 128 * 128; }
int64_t oracle_scale_cols_padded(int64_t cols) { return ((cols / 16) + 3) / 4 * 4; }

/* General 128-row by 4-scale-column tiled offset of scale (r, c) in a matrix
 * with `cols` elements per row.  A tile holds 128 rows x 4 scale columns in
 * 512 bytes; tiles run along the scale columns first, then down the rows.
 * Inside a tile, row r sits at (r mod 32) * 16 + ((r / 32) mod 4) * 4 and
 * column c at c mod 4. */
int64_t oracle_scale_offset(int64_t r, int64_t c, int64_t cols) {
  int64_t cpad = oracle_scale_cols_padded(cols);
  int64_t tile = (r / 128) * (cpad / 4) + (c / 4);
  return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

/* ---------------- Two-pass NVFP4 quantisation ------------------------------ */

/* Element (r, j) of the tensor being quantised: the SwiGLU output for the
 * activation producer, or the BF16 input itself for a weight. */
static uint16_t elem(const uint16_t* x, int64_t ld, int64_t cols, int swiglu,
                     const uint16_t* silu_tab, int64_t r, int64_t j) {
  const uint16_t* row = x + r * ld;
  return swiglu ? oracle_swiglu_bf16(row[j], row[cols + j], silu_tab) : row[j];
}

/* Quantise a [rows, cols] tensor (cols % 16 == 0) to NVFP4.
 *   x: BF16 input, row stride ld elements; with swiglu != 0 each row holds
 *      gate in [0, cols) and up in [cols, 2 cols).
 *   qdata: padded_rows * cols/2 bytes; scales: padded_rows * scale_cols_padded
 *   bytes in the tiled layout; rec: global scale record.
 * Pass 1: amax = max |h|; global g = amax / 2688 (2688 = 6 * 448).
 * Pass 2: per 16-element block, d = 6 g, bs = E4M3(block_amax / d),
 *         s = E4M3val(bs) * g, code = E2M1(h / s), two codes per byte. */
int oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int swiglu,
                    uint8_t* qdata, uint8_t* scales, oracle_scale_rec* rec) {
  if (rows < 1 || cols < 16 || cols % 16 != 0 || !x || !qdata || !scales || !rec)
    return ORACLE_EINVAL;
  int64_t mpad = oracle_padded_rows(rows);
  int64_t nblk = cols / 16;
  int64_t cpad = oracle_scale_cols_padded(cols);
  uint16_t* silu_tab = NULL;
  if (swiglu) {
    silu_tab = (uint16_t*)malloc(65536 * sizeof(uint16_t));
    if (!silu_tab) return ORACLE_EINVAL;
    oracle_silu_table(silu_tab);
  }
  memset(qdata, 0, (size_t)(mpad * cols / 2));
  memset(scales, 0, (size_t)(mpad * cpad));

  /* pass 1: the largest |h| as a bit pattern (|h| >= 0, so the unsigned bit
   * order is the value order; NaN patterns sort above +inf) */
  uint32_t amax_bits = 0;
#pragma omp parallel for reduction(max : amax_bits) schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < cols; ++j) {
      uint32_t b = ((uint32_t)elem(x, ld, cols, swiglu, silu_tab, r, j) << 16) & 0x7FFFFFFFu;
      if (b > amax_bits) amax_bits = b;
    }
  }
  rec->amax_bits = amax_bits;
  rec->pad = 0;
  if (amax_bits >= 0x7F800000u) {
    rec->status = ORACLE_ENONFINITE;
    rec->global_scale = bits_f32(0x7FC00000u);
    free(silu_tab);
    return ORACLE_OK;
  }
  rec->status = ORACLE_OK;
  float amax = bits_f32(amax_bits);
  float g = amax / 2688.0f;
  rec->global_scale = g;
  float d = 6.0f * g;

  /* pass 2 */
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float h[16];
    for (int64_t b = 0; b < nblk; ++b) {
      float bmax = 0.0f;
      for (int i = 0; i < 16; ++i) {
        h[i] = oracle_bf16_to_f32(elem(x, ld, cols, swiglu, silu_tab, r, b * 16 + i));
        float a = fabsf(h[i]);
        if (a > bmax) bmax = a;
      }
      float ratio = (d == 0.0f) ? 0.0f : bmax / d;
      int bs = oracle_e4m3_encode(ratio);
      float s = (float)oracle_e4m3_value(bs) * g;
      scales[oracle_scale_offset(r, b, cols)] = (uint8_t)bs;
      for (int i = 0; i < 16; i += 2) {
        int c0 = (s == 0.0f) ? 0 : oracle_e2m1_encode(h[i] / s);
        int c1 = (s == 0.0f) ? 0 : oracle_e2m1_encode(h[i + 1] / s);
        qdata[r * (cols / 2) + b * 8 + i / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
  free(silu_tab);
  return ORACLE_OK;
}

/* ---------------- Dequantisation and the block-scaled GEMM ------------------ */

/* Dequantise rows `row_ids[0..nrows)` of an NVFP4 tensor into binary64:
 * out[i, k] = E2M1val(code) * E4M3val(scale) * global.  Exact: the product
 * needs 2 + 4 + 24 significant bits. */
void oracle_dequantize_rows(const uint8_t* qdata, const uint8_t* scales, float global,
                            int64_t cols, const int64_t* row_ids, int64_t nrows, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = row_ids[i];
    for (int64_t k = 0; k < cols; ++k) {
      uint8_t byte = qdata[r * (cols / 2) + k / 2];
      int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      int sc = scales[oracle_scale_offset(r, k / 16, cols)];
      out[i * cols + k] = oracle_e2m1_value(code) * oracle_e4m3_value(sc) * (double)global;
    }
  }
}

/* ref[i, n] = sum_k deqA[row_ids[i], k] * deqW[n, k], in binary64, k in
 * increasing order (the unrounded GEMM value; the CUDA output is compared to
 * it under the stated tolerance). */
int oracle_gemm_rows(const uint8_t* a_q, const uint8_t* a_s, float ga,
                     const uint8_t* w_q, const uint8_t* w_s, float gw,
                     int64_t n, int64_t k, const int64_t* row_ids, int64_t nrows, double* out) {
  if (n < 1 || k < 16 || k % 16 != 0 || nrows < 0) return ORACLE_EINVAL;
  double* wd = (double*)malloc((size_t)(n * k) * sizeof(double));
  double* ad = (double*)malloc((size_t)((nrows ? nrows : 1) * k) * sizeof(double));
  int64_t* wrows = (int64_t*)malloc((size_t)n * sizeof(int64_t));
  if (!wd || !ad || !wrows) { free(wd); free(ad); free(wrows); return ORACLE_EINVAL; }
  for (int64_t j = 0; j < n; ++j) wrows[j] = j;
  oracle_dequantize_rows(w_q, w_s, gw, k, wrows, n, wd);
  oracle_dequantize_rows(a_q, a_s, ga, k, row_ids, nrows, ad);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t i = 0; i < nrows; ++i) {
    for (int64_t j0 = 0; j0 < n; j0 += 8) {
      const double* a = ad + i * k;
      double acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      int64_t jn = (n - j0 < 8) ? n - j0 : 8;
      /* eight independent sums, each in increasing k */
      for (int64_t kk = 0; kk < k; ++kk)
        for (int64_t t = 0; t < jn; ++t) acc[t] += a[kk] * wd[(j0 + t) * k + kk];
      for (int64_t t = 0; t < jn; ++t) out[i * n + j0 + t] = acc[t];
    }
  }
  free(wd); free(ad); free(wrows);
  return ORACLE_OK;
}

/* The GEMM epilogue's rounding of accumulator values ("FC2 NVFP4 Scheduling
 * Results", Canonical Operation: FP32 accumulation and scalars, BF16
 * output): out[i] = RNE_bf16(RN_f32(acc_i * alpha)) with acc_i the binary32
 * accumulator, taken here as (float)ref[i].  That equals the tensor core's
 * accumulator whenever every partial sum of the dot product is exact in
 * binary32 (e.g. E2M1 values with unit block scales: multiples of 1/4 far
 * below 2^22), so for such inputs the whole GEMM output is known exactly. */
void oracle_epilogue_bf16(const double* ref, int64_t n, float alpha, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float acc = (float)ref[i];
    out[i] = oracle_f32_to_bf16(acc * alpha);
  }
}

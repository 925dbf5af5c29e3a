/*
 * fp8_oracle.c -- plain CPU oracle for the FP8 scaled matrix multiply with a
 * fused global amax.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  The CUDA path
 * shares no code with it and never calls it.
 *
 * What it computes, and where each step comes from:
 *
 *   C[l,m,n] = round_out( sum_c  S_A(l,m,c) * S_B(l,n,c) * sum_{k in c} dec(A[l,m,k]) * dec(B[l,n,k]) )
 *   Amax     = max |C|
 *
 *   - torch._scaled_mm semantics: the product of two FP8 matrices, the result
 *     multiplied by both one-element fp32 scales, then cast to out_dtype
 *     (mmaemu "API reference (v0.1)", section mmaemu.scaled_mm, argument table).
 *   - Per-tensor, 1x128 and 128x128 block scales along K
 *     (TileOPs "Linear Algebra Operators", tileops.gemm.GemmFP8FwdOp).
 *   - Block-scaled MX form: dequantize A and B with one UE8M0 factor per
 *     sf_vec_size = 32 elements along K, then a plain sum over K, then
 *     Amax = max over m, n, l of |C|  (cuDNN "GEMM + Amax (SM100)", Shapes,
 *     Equations and the "Using JAX arrays" note on the physical atom layout).
 *     The same page's FP4 operands (E2M1) with factors per 32 (UE8M0) or per
 *     16 (float8_e4m3fn) elements follow the same steps.
 *   - Optional bias [N] added before the rounding (TileOPs GemmFP8FwdOp), and
 *     FP8 outputs scaled by scale_result (mmaemu.scaled_mm).
 *
 * Everything is evaluated in float64 with one final rounding to the output
 * format (round to nearest, ties to even).  For E4M3 operands every product is
 * a multiple of 2^-18 below 2^17.7 in magnitude, so for K < 2^17 the unscaled
 * float64 sum is exact; the scaled results are then exact up to the one
 * rounding of each scale multiplication.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): E4M3 is float8_e4m3fn (no infinities, S.1111.111 is NaN, largest
 * finite 448); E5M2 follows IEEE rules (exponent 31: mantissa 0 is Inf,
 * otherwise NaN); UE8M0 code e means 2^(e-127) and 0xFF is NaN; non-finite
 * values propagate by IEEE arithmetic; bf16/fp16/fp32 outputs overflow to Inf;
 * FP8 outputs are the result times scale_result, rounded once and saturated.
 *
 * Parity pins (tests/test_oracle_*.py): decode tables against torch's float8
 * casts; brute-force exact rationals on tiny K; power-of-two scale linearity;
 * NT/NN/TN/TT stride equivalence; constant block scales equal per-tensor; MX
 * factors read back through the page's logical-to-physical permutation;
 * output rounding against C's and numpy's conversions; FP8 outputs against
 * torch's float8 casts; bias against exact rationals; FP4 against torch's
 * own FP4 packing and blocked-layout routines.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FMT_E4M3 0
#define OR_FMT_E5M2 1
#define OR_FMT_E2M1 2

#define OR_OUT_F32 0
#define OR_OUT_BF16 1
#define OR_OUT_F16 2
#define OR_OUT_E4M3 3
#define OR_OUT_E5M2 4

#define OR_SCALE_TENSOR 0
#define OR_SCALE_A1x128_B1x128 1
#define OR_SCALE_A1x128_B128x128 2
#define OR_SCALE_MX32_UE8M0 3
#define OR_SCALE_NV16_E4M3 4

/* ------------------------------------------------------------------------ */
/* FP8 decode, bit by bit.                                                   */
/* ------------------------------------------------------------------------ */

/* float8_e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Normal:    (1 + m/8) * 2^(e-7)  =  (8 + m) * 2^(e-10)
 * Subnormal: (m/8) * 2^-6         =  m * 2^-9
 * e = 15, m = 7 is NaN; there is no infinity, so e = 15, m = 6 gives 448. */
double oracle_decode_e4m3(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp((double)(8 + m), e - 10);
  return sign ? -mag : mag;
}

/* float8_e5m2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits.
 * Normal:    (1 + m/4) * 2^(e-15)  =  (4 + m) * 2^(e-17)
 * Subnormal: (m/4) * 2^-14         =  m * 2^-16
 * e = 31: m = 0 is +-Inf, m != 0 is NaN (IEEE-style); largest finite 57344. */
double oracle_decode_e5m2(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 2) & 0x1F;
  int m = code & 0x3;
  double mag;
  if (e == 0x1F) {
    if (m != 0) return NAN;
    mag = INFINITY;
  } else if (e == 0) {
    mag = ldexp((double)m, -16);
  } else {
    mag = ldexp((double)(4 + m), e - 17);
  }
  return sign ? -mag : mag;
}

/* float4_e2m1 (cuDNN "GEMM + Amax (SM100)", Dtypes: float4_e2m1fn_x2, two
 * values per byte): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, in
 * the low four bits of `code`.
 * Normal:    (1 + m/2) * 2^(e-1)  =  (2 + m) * 2^(e-2)
 * Subnormal: (m/2)                =  m * 2^-1
 * No infinity and no NaN; largest finite 6. */
double oracle_decode_e2m1(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 0x3;
  int m = code & 0x1;
  double mag = (e == 0) ? ldexp((double)m, -1) : ldexp((double)(2 + m), e - 2);
  return sign ? -mag : mag;
}

double oracle_decode(int fmt, uint8_t code) {
  if (fmt == OR_FMT_E2M1) return oracle_decode_e2m1(code);
  return fmt == OR_FMT_E5M2 ? oracle_decode_e5m2(code) : oracle_decode_e4m3(code);
}

/* UE8M0 scale factor (float8_e8m0fnu): code e is 2^(e-127); 0xFF is NaN. */
double oracle_decode_ue8m0(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* ------------------------------------------------------------------------ */
/* Rounding to a binary floating-point format, round to nearest even.        */
/* p = significand bits including the implicit one; emin = exponent of the   */
/* smallest normal; emax = exponent of the largest binade.  The value is     */
/* rounded as if the exponent range were unbounded above, and a result       */
/* above the largest finite number becomes +-Inf (IEEE 754 overflow).        */
/* ------------------------------------------------------------------------ */
static double round_binary(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  int ex;
  frexp(x, &ex); /* x = f * 2^ex with 0.5 <= |f| < 1, so the binade is ex-1 */
  int binade = ex - 1;
  if (binade < emin) binade = emin;
  double quantum = ldexp(1.0, binade - (p - 1));
  double r = nearbyint(x / quantum) * quantum; /* default mode: ties to even */
  double maxfinite = ldexp(2.0 - ldexp(1.0, -(p - 1)), emax);
  if (fabs(r) > maxfinite) return x > 0 ? INFINITY : -INFINITY;
  return r;
}

double oracle_round_f32(double x) { return round_binary(x, 24, -126, 127); }
double oracle_round_bf16(double x) { return round_binary(x, 8, -126, 127); }
double oracle_round_f16(double x) { return round_binary(x, 11, -14, 15); }

uint8_t oracle_encode_e4m3_sat(double x);
uint8_t oracle_encode_e5m2_sat(double x);

/* FP8 outputs (mmaemu "API reference (v0.1)", mmaemu.scaled_mm: out_dtype
 * may be float8_e4m3fn or float8_e5m2).  Reading: one rounding to nearest
 * even on the FP8 grid, saturated to the largest finite value (Inf too); NaN
 * stays NaN. */
double oracle_round_out(int out_dtype, double x) {
  switch (out_dtype) {
    case OR_OUT_BF16: return oracle_round_bf16(x);
    case OR_OUT_F16: return oracle_round_f16(x);
    case OR_OUT_E4M3: return oracle_decode_e4m3(oracle_encode_e4m3_sat(x));
    case OR_OUT_E5M2: return oracle_decode_e5m2(oracle_encode_e5m2_sat(x));
    default: return oracle_round_f32(x);
  }
}

/* ------------------------------------------------------------------------ */
/* FP8 encode with saturation (used to cross-check the input generators).    */
/* Round to nearest even on the format's grid, clamp the magnitude to the    */
/* largest finite value; NaN maps to the canonical 0x7F.                     */
/* ------------------------------------------------------------------------ */
static uint8_t encode_by_table(int fmt, double x) {
  /* The rounded value is exactly representable; find its code (positive
   * codes first, then apply the sign so that -0 keeps its sign bit). */
  double ax = fabs(x);
  for (int c = 0; c < 0x80; ++c) {
    double v = oracle_decode(fmt, (uint8_t)c);
    if (v == ax) return (uint8_t)(signbit(x) ? (c | 0x80) : c);
  }
  return 0x7F; /* unreachable for rounded inputs */
}

uint8_t oracle_encode_e4m3_sat(double x) {
  if (isnan(x)) return 0x7F;
  double r = round_binary(x, 4, -6, 8); /* E4M3 grid: 3 mantissa bits, emin -6 */
  if (isinf(r) || fabs(r) > 448.0) r = copysign(448.0, x);
  return encode_by_table(OR_FMT_E4M3, r);
}

uint8_t oracle_encode_e5m2_sat(double x) {
  if (isnan(x)) return 0x7F;
  double r = round_binary(x, 3, -14, 15); /* E5M2 grid: 2 mantissa bits, emin -14 */
  if (isinf(r) || fabs(r) > 57344.0) r = copysign(57344.0, x);
  return encode_by_table(OR_FMT_E5M2, r);
}

/* ------------------------------------------------------------------------ */
/* Scale lookup.                                                             */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t L, M, N, K;
  const uint8_t *A;
  int64_t sAl, sAm, sAk; /* element strides of A[l][m][k] */
  int a_fmt;
  const uint8_t *B;
  int64_t sBl, sBn, sBk; /* element strides of B[l][n][k] */
  int b_fmt;
  int scale_mode;
  const void *scale_a, *scale_b;
  int out_dtype;
  double scale_result;             /* multiplies the result before an FP8 output's rounding */
  const double *bias;              /* [N] values added to every row, or NULL */
  double *C_exact, *C_out, *absum; /* [L][M][N], any may be NULL */
  int64_t m0, m1;                  /* rows [m0, m1) are computed; C arrays hold m1-m0 rows */
  double dec_a[256], dec_b[256];
} job_t;

/* 1x128 block scales: fp32 [L][rows][ceil(K/128)] (GemmFP8FwdOp, scale_a). */
static double scale_1x128(const float *s, int64_t l, int64_t rows, int64_t r, int64_t c, int64_t KB) {
  return (double)s[(l * rows + r) * KB + c];
}

/* 128x128 block scales: fp32 [L][ceil(N/128)][ceil(K/128)] (GemmFP8FwdOp, scale_b). */
static double scale_128x128(const float *s, int64_t l, int64_t N, int64_t n, int64_t c, int64_t KB) {
  int64_t NB = (N + 127) / 128;
  return (double)s[(l * NB + n / 128) * KB + c];
}

/* Block scale factors in the physical atom layout of "GEMM + Amax (SM100)":
 * with sf_vec_size v the logical tensor has shape
 * (32, 4, ceil(MN/128), 4, ceil(K/(4v)), L) and is the physical C-contiguous
 * (L, ceil(MN/128), ceil(K/(4v)), 32, 4, 4) allocation permuted by
 * (3, 4, 1, 5, 2, 0).  Reading the logical modes with the first index
 * fastest, row r = i32 + 32*i4 + 128*mb and factor index f = j4 + 4*kb, where
 * factor f covers k in [v*f, v*f + v).  So the byte offset is
 * ((l*MB + mb)*KB + kb)*512 + i32*16 + i4*4 + j4.  The factors are UE8M0
 * for v = 32 and float8_e4m3fn for v = 16 (Dtypes: an E4M3 factor only with
 * sf_vec_size 16). */
static double scale_blocked(const uint8_t *sf, int64_t l, int64_t rows, int64_t r, int64_t k, int64_t K,
                            int vec) {
  int64_t MB = (rows + 127) / 128;
  int64_t KB = (K + 4 * vec - 1) / (4 * vec);
  int64_t mb = r / 128, rin = r % 128, i4 = rin / 32, i32 = rin % 32;
  int64_t f = k / vec, kb = f / 4, j4 = f % 4;
  int64_t off = ((l * MB + mb) * KB + kb) * 512 + i32 * 16 + i4 * 4 + j4;
  return vec == 16 ? oracle_decode_e4m3(sf[off]) : oracle_decode_ue8m0(sf[off]);
}

/* ------------------------------------------------------------------------ */
/* One output element.                                                       */
/* ------------------------------------------------------------------------ */
static void one_element(const job_t *j, int64_t l, int64_t m, int64_t n, double *exact, double *abssum) {
  const uint8_t *a = j->A + l * j->sAl + m * j->sAm;
  const uint8_t *b = j->B + l * j->sBl + n * j->sBn;
  int64_t K = j->K;
  int64_t KB = (K + 127) / 128;
  double c = 0.0, s = 0.0;

  if (j->scale_mode == OR_SCALE_TENSOR) {
    /* (A * s_a) @ (B * s_b)^T with one-element scales: the plain sum over K,
     * multiplied by both scales. */
    double sa = (double)((const float *)j->scale_a)[0];
    double sb = (double)((const float *)j->scale_b)[0];
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double p = j->dec_a[a[k * j->sAk]] * j->dec_b[b[k * j->sBk]];
      acc += p;
      aacc += fabs(p);
    }
    c = (sa * sb) * acc;
    s = fabs(sa * sb) * aacc;
  } else if (j->scale_mode == OR_SCALE_MX32_UE8M0 || j->scale_mode == OR_SCALE_NV16_E4M3) {
    /* A_hat = dequantize(A, SFA), B_hat likewise, C = sum_k A_hat * B_hat. */
    const int vec = j->scale_mode == OR_SCALE_NV16_E4M3 ? 16 : 32;
    for (int64_t k = 0; k < K; ++k) {
      double ah = j->dec_a[a[k * j->sAk]] * scale_blocked((const uint8_t *)j->scale_a, l, j->M, m, k, K, vec);
      double bh = j->dec_b[b[k * j->sBk]] * scale_blocked((const uint8_t *)j->scale_b, l, j->N, n, k, K, vec);
      c += ah * bh;
      s += fabs(ah * bh);
    }
  } else {
    /* Block scales along K in chunks of 128: each chunk's sum is multiplied by
     * its two scales and the chunk results are added. */
    for (int64_t cidx = 0; cidx < KB; ++cidx) {
      double sa = scale_1x128((const float *)j->scale_a, l, j->M, m, cidx, KB);
      double sb = (j->scale_mode == OR_SCALE_A1x128_B1x128)
                      ? scale_1x128((const float *)j->scale_b, l, j->N, n, cidx, KB)
                      : scale_128x128((const float *)j->scale_b, l, j->N, n, cidx, KB);
      double acc = 0.0, aacc = 0.0;
      int64_t k1 = (cidx + 1) * 128 < K ? (cidx + 1) * 128 : K;
      for (int64_t k = cidx * 128; k < k1; ++k) {
        double p = j->dec_a[a[k * j->sAk]] * j->dec_b[b[k * j->sBk]];
        acc += p;
        aacc += fabs(p);
      }
      c += (sa * sb) * acc;
      s += fabs(sa * sb) * aacc;
    }
  }
  *exact = c;
  *abssum = s;
}

typedef struct {
  const job_t *job;
  int64_t r_begin, r_end; /* flattened (l, m) rows in [0, L*(m1-m0)) */
} slice_t;

static void *run_slice(void *arg) {
  const slice_t *sl = (const slice_t *)arg;
  const job_t *j = sl->job;
  int64_t rows = j->m1 - j->m0;
  for (int64_t r = sl->r_begin; r < sl->r_end; ++r) {
    int64_t l = r / rows, m = j->m0 + r % rows;
    for (int64_t n = 0; n < j->N; ++n) {
      double e, s;
      one_element(j, l, m, n, &e, &s);
      /* d = (a s_a) @ (b s_b)^T + bias, bias [N] (TileOPs "Linear Algebra
       * Operators", GemmFP8FwdOp): added to the exact value, before the one
       * rounding. */
      if (j->bias) e += j->bias[n];
      int64_t idx = r * j->N + n;
      if (j->C_exact) j->C_exact[idx] = e;
      if (j->absum) j->absum[idx] = s;
      if (j->C_out) {
        /* scale_result is "used only for FP8 outputs" (mmaemu.scaled_mm): the
         * result is multiplied by it, then rounded once. */
        const int fp8_out = j->out_dtype == OR_OUT_E4M3 || j->out_dtype == OR_OUT_E5M2;
        j->C_out[idx] = oracle_round_out(j->out_dtype, fp8_out ? e * j->scale_result : e);
      }
    }
  }
  return NULL;
}

/* Computes rows [m0, m1) of every batch.  Returns 0 on success, -1 on bad
 * arguments.  nthreads <= 0 means one thread. */
int oracle_scaled_gemm(int64_t L, int64_t M, int64_t N, int64_t K,
                       const uint8_t *A, int64_t sAl, int64_t sAm, int64_t sAk, int a_fmt,
                       const uint8_t *B, int64_t sBl, int64_t sBn, int64_t sBk, int b_fmt,
                       int scale_mode, const void *scale_a, const void *scale_b, int out_dtype,
                       double scale_result, const double *bias,
                       double *C_exact, double *C_out, double *absum,
                       int64_t m0, int64_t m1, int nthreads) {
  if (L < 0 || M < 0 || N < 0 || K < 0 || m0 < 0 || m1 > M || m0 > m1) return -1;
  if (scale_mode < 0 || scale_mode > 4) return -1;
  if (a_fmt < 0 || a_fmt > 2 || b_fmt < 0 || b_fmt > 2) return -1;
  if (out_dtype < 0 || out_dtype > 4) return -1;
  if (bias && (out_dtype == OR_OUT_E4M3 || out_dtype == OR_OUT_E5M2)) return -1; /* not defined by the pages */
  job_t *j = (job_t *)calloc(1, sizeof(job_t));
  if (!j) return -1;
  j->L = L; j->M = M; j->N = N; j->K = K;
  j->A = A; j->sAl = sAl; j->sAm = sAm; j->sAk = sAk; j->a_fmt = a_fmt;
  j->B = B; j->sBl = sBl; j->sBn = sBn; j->sBk = sBk; j->b_fmt = b_fmt;
  j->scale_mode = scale_mode; j->scale_a = scale_a; j->scale_b = scale_b;
  j->out_dtype = out_dtype;
  j->scale_result = scale_result;
  j->bias = bias;
  j->C_exact = C_exact; j->C_out = C_out; j->absum = absum;
  j->m0 = m0; j->m1 = m1;
  for (int c = 0; c < 256; ++c) {
    j->dec_a[c] = oracle_decode(a_fmt, (uint8_t)c);
    j->dec_b[c] = oracle_decode(b_fmt, (uint8_t)c);
  }
  int64_t total = L * (m1 - m0);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > total) nthreads = total > 0 ? (int)total : 1;
  slice_t sl[256];
  pthread_t th[256];
  int started[256] = {0};
  for (int t = 0; t < nthreads; ++t) {
    sl[t].job = j;
    sl[t].r_begin = total * t / nthreads;
    sl[t].r_end = total * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) started[t] = pthread_create(&th[t], NULL, run_slice, &sl[t]) == 0;
  run_slice(&sl[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(th[t], NULL);
    else
      run_slice(&sl[t]);
  }
  free(j);
  return 0;
}

/* Amax = max |C| (cuDNN "GEMM + Amax (SM100)", Equations).  |-0| = +0; any
 * NaN makes the result NaN; an empty C gives +0. */
double oracle_amax(const double *C, int64_t count) {
  double m = 0.0;
  for (int64_t i = 0; i < count; ++i) {
    double v = fabs(C[i]);
    if (isnan(v)) return NAN;
    if (v > m) m = v;
  }
  return m;
}

/*
 * CPU oracle for the dense multiply-accumulate D = A*B + C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or helper with the CUDA path, and the product path never
 * loads it: only the test suite, the smoke check and the bench's CPU-baseline
 * leg call into it.
 *
 * What it follows (page title -- section):
 *   - "CDNA2 dense MFMA builtins" -- Naming convention: one instruction adds
 *     the contribution of an M x K panel of A and a K x N panel of B to an
 *     M x N tile; the caller loops over K for the full product.  Here the
 *     whole K loop is written out, so the result is the plain definition
 *       D[i][j] = C[i][j] + sum_k A[i][k] * B[k][j].
 *   - "CDNA2 dense MFMA builtins" -- Builtin reference: FP16/BF16 inputs
 *     accumulate in FP32, INT8 inputs in INT32, FP64 in FP64 with
 *     round-to-nearest-even.
 *   - "RDNA3 dense WMMA builtins" -- Builtin reference: each builtin returns
 *     srcA x srcB + srcC; INT8 inputs are signed (a_neg/b_neg select signed).
 *   - "Common MFMA parameters" -- Shared parameters (cbsz, abid): with a
 *     group of G = 2^cbsz neighbouring blocks, every block of the group uses
 *     the A values of block abid of that group.
 *
 * Precision of the oracle itself:
 *   - FP16/BF16 -> FP32: operands are decoded exactly to double; each product
 *     is exact in double (at most 11 x 11 significant bits); the K products
 *     are summed in double in sequential k order; C is added in double and
 *     the sum is rounded once to FP32 (round to nearest even).
 *   - INT8 -> INT32: exact 64-bit integer sum, plus C; results that do not
 *     fit in INT32 are counted (overflow is never silent) and wrap in two's
 *     complement.
 *   - FP64: Ogita-Rump-Oishi compensated dot product "Dot2" (TwoProduct by
 *     fma, TwoSum by Knuth), with C as one more term, so the oracle's error
 *     is about eps^2 relative to sum |a*b| plus one final rounding.  When a
 *     term (a product or C) is infinite or NaN the compensation terms are
 *     meaningless (inf - inf), and the result is the IEEE value of the
 *     plain sum instead: NaN if a term is NaN or infinities of both signs
 *     meet, else the infinity.
 *
 * Build: plain C11, -O2 -fopenmp -ffp-contract=off (no contraction, no
 * reassociation, no fast-math); only the loop over output rows is parallel.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes, matching the numeric values of the public enum */
enum { OR_F16 = 1, OR_BF16 = 2, OR_I8 = 3, OR_F64 = 4, OR_F32 = 5, OR_I32 = 6 };
/* B layouts: column-major (B[k][j] at B[j*ldb + k]) or row-major */
enum { OR_B_COL = 0, OR_B_ROW = 1 };

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- c1: exact decode of 16-bit float bit patterns -------------------- */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
  const int neg = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x400), e - 25); /* (2^10 + f) * 2^(e-15-10) */
  return neg ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t h) {
  const int neg = (h >> 15) & 1;
  const int e = (h >> 7) & 0xff;
  const int f = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133); /* subnormal: f * 2^(1-127-7) */
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x80), e - 134); /* (2^7 + f) * 2^(e-127-7) */
  return neg ? -v : v;
}

static double *decode_table(int kind) {
  double *t = (double *)malloc(65536 * sizeof(double));
  if (!t) return NULL;
  for (int b = 0; b < 65536; ++b)
    t[b] = kind == OR_F16 ? oracle_f16_to_double((uint16_t)b)
                          : oracle_bf16_to_double((uint16_t)b);
  return t;
}

static inline int64_t b_index(int b_layout, int64_t k, int64_t j, int64_t ldb) {
  return b_layout == OR_B_COL ? j * ldb + k : k * ldb + j;
}

/* ---- c2: FP16/BF16 inputs, FP32 accumulate ---------------------------- *
 * A: M x K row-major (A[i][k] at A[i*lda + k]); B per b_layout; C, D: M x N
 * row-major.  C may be NULL (C = 0).  If absab is not NULL it receives
 * (|A|*|B|)[i][j] in double (the scale of the parity tolerance).        */
static void f16_row(const double *tab, int64_t i, int64_t N, int64_t K,
                    const uint16_t *A, int64_t lda, const uint16_t *B,
                    int64_t ldb, int b_layout, const float *C, int64_t ldc,
                    float *D, int64_t ldd, double *absab, int64_t ldabs) {
  for (int64_t j = 0; j < N; ++j) {
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = tab[A[i * lda + k]];
      const double b = tab[B[b_index(b_layout, k, j, ldb)]];
      s += a * b;
      if (absab) sa += fabs(a) * fabs(b);
    }
    const double c = C ? (double)C[i * ldc + j] : 0.0;
    D[i * ldd + j] = (float)(s + c);
    if (absab) absab[i * ldabs + j] = sa;
  }
}

/* Returns 0, or -1 on bad arguments / allocation failure. */
int oracle_gemm_f16f32(int in_kind, int64_t M, int64_t N, int64_t K,
                       const uint16_t *A, int64_t lda, const uint16_t *B,
                       int64_t ldb, int b_layout, const float *C, int64_t ldc,
                       float *D, int64_t ldd, double *absab, int64_t ldabs) {
  if (in_kind != OR_F16 && in_kind != OR_BF16) return -1;
  if (M < 0 || N < 0 || K < 0) return -1;
  double *tab = decode_table(in_kind);
  if (!tab) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i)
    f16_row(tab, i, N, K, A, lda, B, ldb, b_layout, C, ldc, D, ldd, absab,
            ldabs);
  free(tab);
  return 0;
}

/* ---- c2b: FP16/BF16 inputs, 16-bit accumulator and output ------------- *
 * "RDNA3 dense WMMA builtins" -- FP16/BF16-accumulate builtins: the addend
 * and the result are 16-bit.  The oracle keeps the exact-product double sum
 * of c2, adds the decoded C and rounds once to the 16-bit format (nearest,
 * ties to even).  (The builtins round the 16-bit accumulator after every
 * K step; one final rounding is the plain definition of D = A*B + C in
 * the output format.)                                                    */

/* Round a double to the 16-bit format with `mant` stored fraction bits,
 * exponent bias `bias` and all-ones exponent `emax_field`; nearest, ties to
 * even; overflow to infinity; NaN to a quiet NaN.                        */
static uint16_t round_double_16(double x, int mant, int bias, int emax_field) {
  const uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
  const uint16_t inf = (uint16_t)(sign | ((unsigned)emax_field << mant));
  if (isnan(x)) return (uint16_t)(inf | (1u << (mant - 1)));
  double a = fabs(x);
  if (isinf(a)) return inf;
  if (a == 0.0) return sign;
  const int emin = 1 - bias;                 /* smallest normal exponent */
  int e;
  frexp(a, &e);                              /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;                                    /* a in [2^e, 2^(e+1)) */
  if (e < emin) e = emin;                    /* subnormal quantum */
  const double q = ldexp(1.0, e - mant);     /* spacing of the format at a */
  const double m = rint(a / q);              /* exact division; RNE */
  const double v = m * q;                    /* the rounded magnitude */
  if (v >= ldexp(1.0, emax_field - bias)) return inf;
  if (v < ldexp(1.0, emin)) return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, emin - mant)));
  int ev;
  frexp(v, &ev);
  ev -= 1;
  const unsigned frac = (unsigned)(v / ldexp(1.0, ev - mant)) - (1u << mant);
  return (uint16_t)(sign | ((unsigned)(ev + bias) << mant) | frac);
}

uint16_t oracle_double_to_f16(double x) { return round_double_16(x, 10, 15, 31); }
uint16_t oracle_double_to_bf16(double x) { return round_double_16(x, 7, 127, 255); }

static void h16_row(const double *tab, int in_kind, int64_t i, int64_t N,
                    int64_t K, const uint16_t *A, int64_t lda,
                    const uint16_t *B, int64_t ldb, int b_layout,
                    const uint16_t *C, int64_t ldc, uint16_t *D, int64_t ldd,
                    double *absab, int64_t ldabs) {
  for (int64_t j = 0; j < N; ++j) {
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = tab[A[i * lda + k]];
      const double b = tab[B[b_index(b_layout, k, j, ldb)]];
      s += a * b;
      if (absab) sa += fabs(a) * fabs(b);
    }
    const double c = C ? tab[C[i * ldc + j]] : 0.0;
    D[i * ldd + j] = in_kind == OR_F16 ? oracle_double_to_f16(s + c)
                                       : oracle_double_to_bf16(s + c);
    if (absab) absab[i * ldabs + j] = sa;
  }
}

/* C and D have the input's 16-bit type.  Returns 0, or -1. */
int oracle_gemm_f16f16(int in_kind, int64_t M, int64_t N, int64_t K,
                       const uint16_t *A, int64_t lda, const uint16_t *B,
                       int64_t ldb, int b_layout, const uint16_t *C,
                       int64_t ldc, uint16_t *D, int64_t ldd, double *absab,
                       int64_t ldabs) {
  if (in_kind != OR_F16 && in_kind != OR_BF16) return -1;
  if (M < 0 || N < 0 || K < 0) return -1;
  double *tab = decode_table(in_kind);
  if (!tab) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i)
    h16_row(tab, in_kind, i, N, K, A, lda, B, ldb, b_layout, C, ldc, D, ldd,
            absab, ldabs);
  free(tab);
  return 0;
}

/* ---- c3: INT8 inputs, INT32 accumulate -------------------------------- *
 * Exact int64 sum.  Outputs that do not fit in INT32 wrap in two's
 * complement and are counted.                                           */
static int64_t i8_row(int64_t i, int64_t N, int64_t K, const int8_t *A,
                      int64_t lda, const int8_t *B, int64_t ldb, int b_layout,
                      const int32_t *C, int64_t ldc, int32_t *D, int64_t ldd) {
  int64_t overflow = 0;
  for (int64_t j = 0; j < N; ++j) {
    int64_t s = 0;
    for (int64_t k = 0; k < K; ++k)
      s += (int64_t)A[i * lda + k] * (int64_t)B[b_index(b_layout, k, j, ldb)];
    const int64_t d = s + (C ? (int64_t)C[i * ldc + j] : 0);
    if (d < INT32_MIN || d > INT32_MAX) ++overflow;
    D[i * ldd + j] = (int32_t)(uint32_t)(uint64_t)d;
  }
  return overflow;
}

/* Returns the number of outputs that overflowed INT32, or -1. */
int64_t oracle_gemm_i8i32(int64_t M, int64_t N, int64_t K, const int8_t *A,
                          int64_t lda, const int8_t *B, int64_t ldb,
                          int b_layout, const int32_t *C, int64_t ldc,
                          int32_t *D, int64_t ldd) {
  if (M < 0 || N < 0 || K < 0) return -1;
  int64_t overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : overflow)
  for (int64_t i = 0; i < M; ++i)
    overflow += i8_row(i, N, K, A, lda, B, ldb, b_layout, C, ldc, D, ldd);
  return overflow;
}

/* ---- c3b: INT8 / UINT8 inputs in any signedness, optional clamp ------- *
 * "RDNA3 dense WMMA builtins" -- INT8 and UINT8 inputs: a_neg / b_neg select
 * signed (else unsigned) 8-bit A / B; `clamp` saturates the INT32 result on
 * overflow (else it wraps modulo 2^32).  Exact int64 sum plus C.  Returns
 * the number of outputs whose exact value did not fit in INT32.          */
int64_t oracle_gemm_i8i32_ex(int64_t M, int64_t N, int64_t K, const void *A,
                             int64_t lda, int a_signed, const void *B,
                             int64_t ldb, int b_signed, int b_layout,
                             const int32_t *C, int64_t ldc, int32_t *D,
                             int64_t ldd, int clamp) {
  if (M < 0 || N < 0 || K < 0) return -1;
  const int8_t *As = (const int8_t *)A;
  const uint8_t *Au = (const uint8_t *)A;
  const int8_t *Bs = (const int8_t *)B;
  const uint8_t *Bu = (const uint8_t *)B;
  int64_t overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : overflow)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      int64_t s = 0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t ia = i * lda + k, ib = b_index(b_layout, k, j, ldb);
        const int64_t a = a_signed ? (int64_t)As[ia] : (int64_t)Au[ia];
        const int64_t b = b_signed ? (int64_t)Bs[ib] : (int64_t)Bu[ib];
        s += a * b;
      }
      int64_t d = s + (C ? (int64_t)C[i * ldc + j] : 0);
      if (d < INT32_MIN || d > INT32_MAX) {
        ++overflow;
        if (clamp) d = d < 0 ? INT32_MIN : INT32_MAX;
      }
      D[i * ldd + j] = (int32_t)(uint32_t)(uint64_t)d;
    }
  }
  return overflow;
}

/* ---- c4: FP64, compensated dot product (Dot2) ------------------------- */

/* Knuth's TwoSum: s + e == a + b exactly, s = fl(a + b). */
static inline void two_sum(double a, double b, double *s, double *e) {
  const double x = a + b;
  const double z = x - a;
  *e = (a - (x - z)) + (b - z);
  *s = x;
}

/* TwoProduct with a fused multiply-add: p + e == a * b exactly. */
static inline void two_prod(double a, double b, double *p, double *e) {
  const double x = a * b;
  *e = fma(a, b, -x);
  *p = x;
}

static void f64_row(int64_t i, int64_t N, int64_t K, const double *A,
                    int64_t lda, const double *B, int64_t ldb, int b_layout,
                    const double *C, int64_t ldc, double *D, int64_t ldd,
                    double *absab, int64_t ldabs) {
  for (int64_t j = 0; j < N; ++j) {
    double p = 0.0, s = 0.0, sa = 0.0;
    double plain = 0.0;   /* IEEE sum of the terms, for non-finite ones */
    int special = 0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = A[i * lda + k];
      const double b = B[b_index(b_layout, k, j, ldb)];
      double h, r, q;
      two_prod(a, b, &h, &r);
      two_sum(p, h, &p, &q);
      s += q + r;
      plain += h;
      if (!isfinite(h)) special = 1;
      if (absab) sa += fabs(a) * fabs(b);
    }
    if (C) {
      const double c = C[i * ldc + j];
      double q;
      two_sum(p, c, &p, &q);
      s += q;
      plain += c;
      if (!isfinite(c)) special = 1;
    }
    D[i * ldd + j] = special ? plain : p + s;
    if (absab) absab[i * ldabs + j] = sa;
  }
}

int oracle_gemm_f64(int64_t M, int64_t N, int64_t K, const double *A,
                    int64_t lda, const double *B, int64_t ldb, int b_layout,
                    const double *C, int64_t ldc, double *D, int64_t ldd,
                    double *absab, int64_t ldabs) {
  if (M < 0 || N < 0 || K < 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i)
    f64_row(i, N, K, A, lda, B, ldb, b_layout, C, ldc, D, ldd, absab, ldabs);
  return 0;
}

/* ---- c5: batched tiles with A-block broadcast ------------------------- *
 * Tile b of each operand is stored contiguously: A tile t at A + t*M*lda,
 * B tile b at B + b*N*ldb (column-major B) or B + b*K*ldb (row-major B),
 * C and D tile b at b*M*ldc and b*M*ldd.  With a broadcast group of G
 * entries and source index abid, entry b reads A tile
 *     src(b) = (b / G) * G + abid,
 * while B, C and D are never broadcast.  G is 1, 2, 4, 8 or 16, G must
 * divide batch and 0 <= abid < G.  Returns 0 (or the INT8 overflow count), -1 on bad
 * arguments.                                                            */
/* B-group source of an entry, read from "Common MFMA parameters", section
 * "Dense MFMA parameters" (blgp): the page swizzles B between the four
 * 16-lane quarters of a 64-lane operand.  At matrix level the batch is cut
 * into groups of four consecutive entries, entry q of a group playing lane
 * quarter q; returns the quarter whose B the entry at quarter q reads, or
 * -1 for a pattern outside 0..7.                                          */
int oracle_blgp_source(int blgp, int q) {
  switch (blgp) {
    case 0: return q;                  /* no swizzling                     */
    case 1: return q & 1;              /* lanes 0-31 copied into 32-63     */
    case 2: return 2 + (q & 1);        /* lanes 32-63 copied into 0-31     */
    case 3: return (q + 1) & 3;        /* rotated down by 16 lanes: lane 16
                                          feeds lane 0, lane 0 lane 48     */
    case 4: return 0;                  /* lanes 0-15 to all quarters       */
    case 5: return 1;                  /* lanes 16-31 to all quarters      */
    case 6: return 2;                  /* lanes 32-47 to all quarters      */
    case 7: return 3;                  /* lanes 48-63 to all quarters      */
    default: return -1;
  }
}

int64_t oracle_gemm_batched(int dtype_in, int64_t M, int64_t N, int64_t K,
                            const void *A, int64_t lda, const void *B,
                            int64_t ldb, int b_layout, const void *C,
                            int64_t ldc, void *D, int64_t ldd, int64_t batch,
                            int64_t G, int64_t abid, int blgp) {
  if (M < 0 || N < 0 || K < 0) return -1;
  /* G = 2^cbsz with cbsz in 0..4 ("Common MFMA parameters", cbsz row) */
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return -1;
  if (batch < 0 || abid < 0 || abid >= G || batch % G != 0) return -1;
  if (oracle_blgp_source(blgp, 0) < 0) return -1;
  if (blgp != 0 && batch % 4 != 0) return -1;
  if (dtype_in != OR_F16 && dtype_in != OR_BF16 && dtype_in != OR_I8 &&
      dtype_in != OR_F64)
    return -1;
  double *tab = NULL;
  if (dtype_in == OR_F16 || dtype_in == OR_BF16) {
    tab = decode_table(dtype_in);
    if (!tab) return -1;
  }
  const int64_t b_tile = (b_layout == OR_B_COL ? N : K) * ldb;
  int64_t overflow = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : overflow)
  for (int64_t b = 0; b < batch; ++b) {
    const int64_t src = (b / G) * G + abid;
    /* (pattern 0 maps every entry to itself, whatever the batch) */
    const int64_t bs = (b / 4) * 4 + oracle_blgp_source(blgp, (int)(b % 4));
    for (int64_t i = 0; i < M; ++i) {
      if (dtype_in == OR_I8)
        overflow += i8_row(i, N, K, (const int8_t *)A + src * M * lda, lda,
                           (const int8_t *)B + bs * b_tile, ldb, b_layout,
                           C ? (const int32_t *)C + b * M * ldc : NULL, ldc,
                           (int32_t *)D + b * M * ldd, ldd);
      else if (dtype_in == OR_F64)
        f64_row(i, N, K, (const double *)A + src * M * lda, lda,
                (const double *)B + bs * b_tile, ldb, b_layout,
                C ? (const double *)C + b * M * ldc : NULL, ldc,
                (double *)D + b * M * ldd, ldd, NULL, 0);
      else
        f16_row(tab, i, N, K, (const uint16_t *)A + src * M * lda, lda,
                (const uint16_t *)B + bs * b_tile, ldb, b_layout,
                C ? (const float *)C + b * M * ldc : NULL, ldc,
                (float *)D + b * M * ldd, ldd, NULL, 0);
    }
  }
  free(tab);
  return overflow;
}

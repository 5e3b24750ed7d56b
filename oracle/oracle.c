/*
 * CPU oracle for the dense matrix multiply-accumulate D = A*B + C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; it exists so that the tests, the smoke check and the CPU
 * baseline of the benchmark have an obviously correct result to compare the
 * CUDA library against.  It shares no code, header or constant table with
 * the CUDA library.
 *
 * What it computes (plain definition, no blocking, no fusion, no reordering):
 *
 *   D[i,j] = C[i,j] + sum_{k=0}^{K-1} A[i,k] * B[k,j]
 *
 * The sum over k is formed first and C is added once afterwards, as in the
 * plain HIP kernel "MatMulAdd_kernel2" (forum.sourcefind.cn, "DCU K100 ..."
 * article, section 5.2), where each thread forms the K-sum and then writes
 * sum + C.  The sum over k ascends, as in the Triton "matmul_kernel" of the
 * "Hopper Support in Triton" slides (slide 5: one fp32 accumulator that
 * receives tl.dot of successive BLOCK_K slices).
 *
 * Floating point: fp16/bf16 operands are widened exactly to fp64 and the
 * whole sum is formed in fp64 (every fp16/bf16 product is exact in fp64).
 * The same holds for the two 8-bit float operand types, E4M3 and E5M2: the
 * pages name a scaled low-precision matrix product (mfma_scaled) as the
 * next data type without defining the encodings, so the encodings are the
 * ones of the OCP 8-bit floating point specification (OFP8): E4M3 has 4
 * exponent bits (bias 7) and 3 fraction bits, no infinities, and only the
 * all-ones pattern S.1111.111 is NaN (largest finite 448); E5M2 has 5
 * exponent bits (bias 15) and 2 fraction bits with IEEE 754 infinities and
 * NaNs (largest finite 57344).
 * Integer: int8 operands, int32 C, and the sum is formed in int64 (exact).
 *
 * Indexing follows the storage order of each operand.  Row-major X[r,c] is
 * X[r*ld + c]; column-major X[r,c] is X[r + c*ld] (the article's kernel
 * reads a column-major A as A[row + k*M] and a row-major B as B[k*N + col]).
 *
 * Output rounding to fp16/bf16 is a single round-to-nearest-even of the
 * fp64 value, written out from the IEEE 754 definition.  The pages show the
 * fp32 accumulator being narrowed to fp16 on store (slides 5-6, the
 * arith.truncf before tt.store) but never state the rounding mode; the plain
 * reading is the IEEE default, nearest with ties to even.
 *
 * Build: cc -O2 -fopenmp -shared -fPIC oracle.c -o liboracle.so -lm
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element type codes understood by this file. */
#define OR_F16 1
#define OR_BF16 2
#define OR_F32 3
#define OR_I8 4
#define OR_I32 5
#define OR_E4M3 6
#define OR_E5M2 7

/* Fault-planting hook for the oracle's own self-tests: a build with
 * -DORACLE_MUTANT=n plants one plausible mistake so that the tests can show
 * that their pins catch it.  The default build (n = 0) plants nothing.
 *   1: a square A read transposed
 *   2: C dropped            3: C subtracted
 *   4: last k dropped       5: rounding ties away from zero
 *   6: integer sum starts at k = 1
 *   7: subnormal scale off by a factor of two in the widening
 *   8: A's k index reversed (A[i, K-1-k] paired with B[k, j])
 *   9: E4M3 read with IEEE specials (exponent field 15 as inf / NaN)
 *  10: block-scaled product with blocks of 16 K elements instead of 32
 *  11: E8M0 scale read with bias 128 instead of 127
 *  12: block-scaled product ignores B's scales
 *  13: block-scaled product applies each row's first block scale to all K
 *  14: C's storage order ignored (C always read row-major)
 *  15: a square B read transposed
 *  16: the rows variant ignores its row list (output row q from A's row q)
 *  17: the points variant swaps the coordinates of square problems
 *  18: the magnitude sum S adds signed products */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------------------
 * Binary16, bfloat16 and the two OFP8 encodings.
 *   binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
 *   bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.
 *   E5M2:     1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE specials.
 *   E4M3:     1 sign, 4 exponent (bias 7), 3 fraction bits; the all-ones
 *             exponent holds normal numbers except S.1111.111 (NaN).
 * ------------------------------------------------------------------------- */
typedef struct {
  int frac_bits; /* stored fraction bits */
  int exp_bits;
  int bias;
  int ieee_specials; /* all-ones exponent = inf (fraction 0) or NaN */
} or_format;

static const or_format FMT_F16 = {10, 5, 15, 1};
static const or_format FMT_BF16 = {7, 8, 127, 1};
static const or_format FMT_E5M2 = {2, 5, 15, 1};
#if ORACLE_MUTANT == 9
static const or_format FMT_E4M3 = {3, 4, 7, 1};
#else
static const or_format FMT_E4M3 = {3, 4, 7, 0};
#endif

/* Exact value of an encoding. */
static double widen_bits(uint32_t bits, or_format f) {
  const uint32_t frac_mask = (1u << f.frac_bits) - 1u;
  const uint32_t exp_mask = (1u << f.exp_bits) - 1u;
  const uint32_t frac = bits & frac_mask;
  const uint32_t e = (bits >> f.frac_bits) & exp_mask;
  const int neg = (int)((bits >> (f.frac_bits + f.exp_bits)) & 1u);
  double v;
  if (e == exp_mask && f.ieee_specials) {
    v = frac ? NAN : INFINITY;
  } else if (e == exp_mask && frac == frac_mask) {
    v = NAN; /* E4M3: the only NaN pattern; no infinities */
  } else if (e == 0) {
    /* subnormal: frac * 2^(1 - bias - frac_bits) */
#if ORACLE_MUTANT == 7
    v = ldexp((double)frac, -f.bias - f.frac_bits);
#else
    v = ldexp((double)frac, 1 - f.bias - f.frac_bits);
#endif
  } else {
    v = ldexp((double)((1u << f.frac_bits) | frac), (int)e - f.bias - f.frac_bits);
  }
  return neg ? -v : v;
}

/* Round x to the nearest value of format f, ties to the even significand.
 * The exponent is unbounded above (a result beyond the largest finite value
 * becomes infinity) and underflow is gradual (subnormals are produced).
 * Returns the encoding. */
static uint32_t round_bits(double x, or_format f) {
  const int p = f.frac_bits + 1;          /* precision in bits */
  const int emin = 1 - f.bias;            /* exponent of the smallest normal */
  const int emax = f.bias;                /* exponent of the largest normal */
  const uint32_t exp_all = (1u << f.exp_bits) - 1u;
  const uint32_t sign = signbit(x) ? (1u << (f.frac_bits + f.exp_bits)) : 0u;
  if (isnan(x)) return sign | (exp_all << f.frac_bits) | (1u << (f.frac_bits - 1));
  const double a = fabs(x);
  if (isinf(a)) return sign | (exp_all << f.frac_bits);
  if (a == 0.0) return sign;

  int E;
  (void)frexp(a, &E);            /* a = m * 2^E with m in [0.5, 1) */
  int e = E - 1;                 /* a in [2^e, 2^(e+1)) */
  if (e < emin) e = emin;        /* below the normal range the spacing is fixed */
  const int qexp = e - (p - 1);  /* log2 of the spacing of the format near a */
  const double r = ldexp(a, -qexp); /* exact: scaling by a power of two */
  double n = floor(r);
  const double rem = r - n;      /* exact */
#if ORACLE_MUTANT == 5
  if (rem >= 0.5) n += 1.0;
#else
  if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
#endif
  const double v = ldexp(n, qexp); /* the rounded magnitude */

  const double max_finite = ldexp((double)((1u << p) - 1u), emax - (p - 1));
  if (v > max_finite) return sign | (exp_all << f.frac_bits);

  if (v < ldexp(1.0, emin)) {
    /* subnormal or zero: the fraction field is v / 2^(emin - (p-1)) */
    return sign | (uint32_t)ldexp(v, -(emin - (p - 1)));
  }
  int E2;
  (void)frexp(v, &E2);
  const int e2 = E2 - 1;
  const uint32_t sig = (uint32_t)ldexp(v, -(e2 - (p - 1))); /* in [2^(p-1), 2^p) */
  const uint32_t ef = (uint32_t)(e2 + f.bias);
  return sign | (ef << f.frac_bits) | (sig - (1u << (p - 1)));
}

/* Exported: exact widening of n encoded values of type t (OR_F16/OR_BF16). */
int oracle_widen(const uint16_t* bits, int64_t n, int t, double* out) {
  if (t != OR_F16 && t != OR_BF16) return -1;
  const or_format f = (t == OR_F16) ? FMT_F16 : FMT_BF16;
  for (int64_t i = 0; i < n; ++i) out[i] = widen_bits(bits[i], f);
  return 0;
}

/* Exported: exact widening of n 8-bit float encodings (OR_E4M3/OR_E5M2). */
int oracle_widen8(const uint8_t* bits, int64_t n, int t, double* out) {
  if (t != OR_E4M3 && t != OR_E5M2) return -1;
  const or_format f = (t == OR_E4M3) ? FMT_E4M3 : FMT_E5M2;
  for (int64_t i = 0; i < n; ++i) out[i] = widen_bits(bits[i], f);
  return 0;
}

/* Exported: one round-to-nearest-even of each fp64 value to type t. */
int oracle_round(const double* x, int64_t n, int t, uint16_t* out_bits) {
  if (t != OR_F16 && t != OR_BF16) return -1;
  const or_format f = (t == OR_F16) ? FMT_F16 : FMT_BF16;
  for (int64_t i = 0; i < n; ++i) out_bits[i] = (uint16_t)round_bits(x[i], f);
  return 0;
}

/* Exported: number of threads the parallel loops below use. */
int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Exported: set the number of threads of the parallel loops below (n >= 1);
 * used only to time the oracle on one core and on all of them.  Returns the
 * count now in effect. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* Element (r, c) of an operand stored with leading dimension ld. */
static int64_t at(int64_t r, int64_t c, int col_major, int64_t ld) {
  return col_major ? r + c * ld : r * ld + c;
}

/* Element (i, k) of A, an M x K operand. */
static int64_t at_a(int64_t i, int64_t k, int64_t M, int64_t K, int col_major, int64_t ld) {
#if ORACLE_MUTANT == 1
  if (M == K) return at(k, i, col_major, ld);
#elif ORACLE_MUTANT == 8
  return at(i, K - 1 - k, col_major, ld);
#endif
  (void)M;
  (void)K;
  return at(i, k, col_major, ld);
}

/* Floating-point element, widened to fp64. */
static double load_f(const void* base, int t, int64_t idx) {
  switch (t) {
    case OR_F16: return widen_bits(((const uint16_t*)base)[idx], FMT_F16);
    case OR_BF16: return widen_bits(((const uint16_t*)base)[idx], FMT_BF16);
    case OR_F32: return (double)((const float*)base)[idx];
    case OR_E4M3: return widen_bits(((const uint8_t*)base)[idx], FMT_E4M3);
    case OR_E5M2: return widen_bits(((const uint8_t*)base)[idx], FMT_E5M2);
    default: return NAN;
  }
}

/* Element (i, j) of C. */
static int64_t at_c(int64_t i, int64_t j, int col_major, int64_t ld) {
#if ORACLE_MUTANT == 14
  (void)col_major;
  return at(i, j, 0, ld);
#else
  return at(i, j, col_major, ld);
#endif
}

/* Element (k, j) of B, a K x N operand. */
static int64_t at_b(int64_t k, int64_t j, int64_t K, int64_t N, int col_major, int64_t ld) {
#if ORACLE_MUTANT == 15
  if (K == N) return at(j, k, col_major, ld);
#endif
  (void)K;
  (void)N;
  return at(k, j, col_major, ld);
}

/* |p| for the magnitude sum S of the error bound. */
static double mag(double p) {
#if ORACLE_MUTANT == 18
  return p;
#else
  return fabs(p);
#endif
}

/* Output row of entry q of a rows call (rows == NULL: every row). */
static int64_t row_of(const int64_t* rows, int64_t q, int64_t M) {
#if ORACLE_MUTANT == 16
  return rows ? q % M : q;
#else
  (void)M;
  return rows ? rows[q] : q;
#endif
}

/* Coordinates of point q of a points call. */
static int64_t point_row(const int64_t* pi, const int64_t* pj, int64_t q, int64_t M, int64_t N) {
#if ORACLE_MUTANT == 17
  if (M == N) return pj[q];
#endif
  (void)pj;
  (void)M;
  (void)N;
  return pi[q];
}

static int64_t point_col(const int64_t* pi, const int64_t* pj, int64_t q, int64_t M, int64_t N) {
#if ORACLE_MUTANT == 17
  if (M == N) return pi[q];
#endif
  (void)pi;
  (void)M;
  (void)N;
  return pj[q];
}

static double add_c(double sum, double c) {
#if ORACLE_MUTANT == 2
  (void)c;
  return sum;
#elif ORACLE_MUTANT == 3
  return sum - c;
#else
  return sum + c;
#endif
}

static int64_t k_end(int64_t K) {
#if ORACLE_MUTANT == 4
  return K > 0 ? K - 1 : 0;
#else
  return K;
#endif
}

static int fp_types_ok(int ab_type, int c_type, const void* C) {
  if (ab_type != OR_F16 && ab_type != OR_BF16 && ab_type != OR_E4M3 && ab_type != OR_E5M2)
    return 0;
  if (C && c_type != OR_F16 && c_type != OR_BF16 && c_type != OR_F32) return 0;
  return 1;
}

/* ---------------------------------------------------------------------------
 * Floating-point oracle over whole rows.
 *   rows == NULL: every row i in [0, M); otherwise the nrows rows listed.
 *   D : nrows x N fp64, dense row-major (D[q*N + j] is row rows[q]).
 *   S : optional, same shape: sum_k |A[i,k] * B[k,j]|, for the error bound.
 *   C : may be NULL, meaning C = 0 (C is then never read).
 * Loop order i, k, j over operands widened once; for every output the sum
 * over k ascends.  Returns 0, -1 on bad arguments, -2 when out of memory.
 * ------------------------------------------------------------------------- */
int oracle_gemm_f64_rows(int64_t M, int64_t N, int64_t K, int ab_type, int c_type,
                         int a_col, int b_col, int c_col,
                         int64_t lda, int64_t ldb, int64_t ldc,
                         const void* A, const void* B, const void* C,
                         const int64_t* rows, int64_t nrows, double* D, double* S) {
  if (M < 0 || N < 0 || K < 0 || !fp_types_ok(ab_type, c_type, C)) return -1;
  const int64_t nr = rows ? nrows : M;
  for (int64_t q = 0; q < nr; ++q)
    if (rows && (rows[q] < 0 || rows[q] >= M)) return -1;
  if (nr == 0 || N == 0) return 0;

  double* Bw = (double*)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(double));
  double* Aw = (double*)malloc((size_t)(K > 0 ? K : 1) * (size_t)nr * sizeof(double));
  if (!Bw || !Aw) {
    free(Bw);
    free(Aw);
    return -2;
  }
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j) Bw[k * N + j] = load_f(B, ab_type, at_b(k, j, K, N, b_col, ldb));

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < nr; ++q) {
    const int64_t i = row_of(rows, q, M);
    double* a = Aw + q * K;
    double* d = D + q * N;
    double* s = S ? S + q * N : NULL;
    for (int64_t k = 0; k < K; ++k) a[k] = load_f(A, ab_type, at_a(i, k, M, K, a_col, lda));
    for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
    if (s)
      for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
    const int64_t ke = k_end(K);
    for (int64_t k = 0; k < ke; ++k) {
      const double aik = a[k];
      const double* brow = Bw + k * N;
      for (int64_t j = 0; j < N; ++j) d[j] += aik * brow[j];
      if (s)
        for (int64_t j = 0; j < N; ++j) s[j] += mag(aik * brow[j]);
    }
    if (C)
      for (int64_t j = 0; j < N; ++j) d[j] = add_c(d[j], load_f(C, c_type, at_c(i, j, c_col, ldc)));
  }
  free(Bw);
  free(Aw);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Floating-point oracle at single elements (pi[q], pj[q]), q < npts: the
 * same definition, one length-K dot product per element with k ascending.
 * D[q] and (optional) S[q] receive the value and sum_k |a*b|.
 * ------------------------------------------------------------------------- */
int oracle_gemm_f64_points(int64_t M, int64_t N, int64_t K, int ab_type, int c_type,
                           int a_col, int b_col, int c_col,
                           int64_t lda, int64_t ldb, int64_t ldc,
                           const void* A, const void* B, const void* C,
                           const int64_t* pi, const int64_t* pj, int64_t npts,
                           double* D, double* S) {
  if (M < 0 || N < 0 || K < 0 || !fp_types_ok(ab_type, c_type, C)) return -1;
  for (int64_t q = 0; q < npts; ++q)
    if (pi[q] < 0 || pi[q] >= M || pj[q] < 0 || pj[q] >= N) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < npts; ++q) {
    const int64_t i = point_row(pi, pj, q, M, N), j = point_col(pi, pj, q, M, N);
    double d = 0.0, s = 0.0;
    const int64_t ke = k_end(K);
    for (int64_t k = 0; k < ke; ++k) {
      const double p = load_f(A, ab_type, at_a(i, k, M, K, a_col, lda)) *
                       load_f(B, ab_type, at_b(k, j, K, N, b_col, ldb));
      d += p;
      s += mag(p);
    }
    if (C) d = add_c(d, load_f(C, c_type, at_c(i, j, c_col, ldc)));
    D[q] = d;
    if (S) S[q] = s;
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Block-scaled 8-bit float product (microscaling).
 *
 * The pages name a scaled low-precision matrix product (the mfma_scaled
 * entry point of the "Tuning Triton" page, section 6, for the microscaled
 * data types) without defining the scaling.  The plain reading is the OCP
 * Microscaling (MX) definition: along K, every block of 32 consecutive
 * elements of a row of A (and of a column of B) shares one scale X, stored
 * as an 8-bit power-of-two exponent (E8M0: X = 2^(e - 127), e = 255 is NaN);
 * the element's value is X times its 8-bit float value.  So
 *
 *   D[i,j] = C[i,j] + sum_k (XA[i, k/32] A[i,k]) * (XB[j, k/32] B[k,j])
 *
 * with k ascending and C added after the sum, as above.  Every product is
 * exact in fp64 (8-bit floats times powers of two within 2^+-254).  A last
 * block shorter than 32 (K not a multiple of 32) keeps its own scale.
 *   SA: M x nb scale exponents, row-major (SA[i*nb + b]), nb = ceil(K/32);
 *   SB: N x nb scale exponents, row-major (SB[j*nb + b]) -- per column of B.
 * Rows variant only (D, S, rows, C as in oracle_gemm_f64_rows).
 * ------------------------------------------------------------------------- */
/* Scale block of element k (nb blocks per row). */
static int64_t mx_block(int64_t k, int64_t nb) {
#if ORACLE_MUTANT == 10
  return (k / 16) % nb; /* kept inside the row's nb scales */
#else
  (void)nb;
  return k / 32;
#endif
}

static double e8m0(uint8_t e) {
  if (e == 255) return NAN;
#if ORACLE_MUTANT == 11
  return ldexp(1.0, (int)e - 128);
#else
  return ldexp(1.0, (int)e - 127);
#endif
}

int oracle_gemm_mx_rows(int64_t M, int64_t N, int64_t K, int ab_type, int c_type,
                        int a_col, int b_col, int c_col,
                        int64_t lda, int64_t ldb, int64_t ldc,
                        const void* A, const void* B, const void* C,
                        const uint8_t* SA, const uint8_t* SB,
                        const int64_t* rows, int64_t nrows, double* D, double* S) {
  if (M < 0 || N < 0 || K < 0 || (ab_type != OR_E4M3 && ab_type != OR_E5M2) ||
      !fp_types_ok(ab_type, c_type, C) || (K > 0 && (!SA || !SB)))
    return -1;
  const int64_t nr = rows ? nrows : M;
  for (int64_t q = 0; q < nr; ++q)
    if (rows && (rows[q] < 0 || rows[q] >= M)) return -1;
  if (nr == 0 || N == 0) return 0;
  const int64_t nb = (K + 31) / 32; /* scale blocks per row (the stored layout) */

  /* B widened and scaled once: Bw[k*N + j] = XB[j, k/32] * B[k,j]. */
  double* Bw = (double*)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(double));
  double* Aw = (double*)malloc((size_t)(K > 0 ? K : 1) * (size_t)nr * sizeof(double));
  if (!Bw || !Aw) {
    free(Bw);
    free(Aw);
    return -2;
  }
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j) {
#if ORACLE_MUTANT == 12
      const double xb = 1.0;
#else
      const double xb = e8m0(SB[j * nb + mx_block(k, nb)]);
#endif
      Bw[k * N + j] = xb * load_f(B, ab_type, at_b(k, j, K, N, b_col, ldb));
    }

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < nr; ++q) {
    const int64_t i = row_of(rows, q, M);
    double* a = Aw + q * K;
    double* d = D + q * N;
    double* s = S ? S + q * N : NULL;
    for (int64_t k = 0; k < K; ++k) {
#if ORACLE_MUTANT == 13
      const double xa = e8m0(SA[i * nb]);
#else
      const double xa = e8m0(SA[i * nb + mx_block(k, nb)]);
#endif
      a[k] = xa * load_f(A, ab_type, at_a(i, k, M, K, a_col, lda));
    }
    for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
    if (s)
      for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double aik = a[k];
      const double* brow = Bw + k * N;
      for (int64_t j = 0; j < N; ++j) d[j] += aik * brow[j];
      if (s)
        for (int64_t j = 0; j < N; ++j) s[j] += mag(aik * brow[j]);
    }
    if (C)
      for (int64_t j = 0; j < N; ++j) d[j] = add_c(d[j], load_f(C, c_type, at_c(i, j, c_col, ldc)));
  }
  free(Bw);
  free(Aw);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Integer oracle: int8 A and B, int32 C (or NULL), int64 sums (exact).
 * Rows variant: D is nrows x N int64, dense row-major.
 * ------------------------------------------------------------------------- */
static int64_t int_k_begin(void) {
#if ORACLE_MUTANT == 6
  return 1;
#else
  return 0;
#endif
}

int oracle_gemm_i64_rows(int64_t M, int64_t N, int64_t K, int a_col, int b_col, int c_col,
                         int64_t lda, int64_t ldb, int64_t ldc,
                         const int8_t* A, const int8_t* B, const int32_t* C,
                         const int64_t* rows, int64_t nrows, int64_t* D) {
  if (M < 0 || N < 0 || K < 0) return -1;
  const int64_t nr = rows ? nrows : M;
  for (int64_t q = 0; q < nr; ++q)
    if (rows && (rows[q] < 0 || rows[q] >= M)) return -1;
  if (nr == 0 || N == 0) return 0;
  int64_t* Bw = (int64_t*)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(int64_t));
  if (!Bw) return -2;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j) Bw[k * N + j] = B[at_b(k, j, K, N, b_col, ldb)];

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < nr; ++q) {
    const int64_t i = row_of(rows, q, M);
    int64_t* d = D + q * N;
    for (int64_t j = 0; j < N; ++j) d[j] = 0;
    for (int64_t k = int_k_begin(); k < K; ++k) {
      const int64_t aik = A[at_a(i, k, M, K, a_col, lda)];
      const int64_t* brow = Bw + k * N;
      for (int64_t j = 0; j < N; ++j) d[j] += aik * brow[j];
    }
    if (C)
      for (int64_t j = 0; j < N; ++j) d[j] += C[at_c(i, j, c_col, ldc)];
  }
  free(Bw);
  return 0;
}

int oracle_gemm_i64_points(int64_t M, int64_t N, int64_t K, int a_col, int b_col, int c_col,
                           int64_t lda, int64_t ldb, int64_t ldc,
                           const int8_t* A, const int8_t* B, const int32_t* C,
                           const int64_t* pi, const int64_t* pj, int64_t npts, int64_t* D) {
  if (M < 0 || N < 0 || K < 0) return -1;
  for (int64_t q = 0; q < npts; ++q)
    if (pi[q] < 0 || pi[q] >= M || pj[q] < 0 || pj[q] >= N) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < npts; ++q) {
    const int64_t i = point_row(pi, pj, q, M, N), j = point_col(pi, pj, q, M, N);
    int64_t d = 0;
    for (int64_t k = int_k_begin(); k < K; ++k)
      d += (int64_t)A[at_a(i, k, M, K, a_col, lda)] * (int64_t)B[at_b(k, j, K, N, b_col, ldb)];
    if (C) d += C[at_c(i, j, c_col, ldc)];
    D[q] = d;
  }
  return 0;
}

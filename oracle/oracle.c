/*
 * oracle.c -- plain CPU oracle for the TN GEMM  C = A x B.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, header, table or constant with the CUDA library: its number codecs
 * are written here from the format definitions (IEEE 754-2008 binary16, the
 * bfloat16 layout, and the OCP 8-bit floating point E4M3 format).
 *
 * What it computes (the plain definition, nothing reordered):
 *
 *   C[m,n] = sum_{k=0}^{K-1} A[m,k] * B[k,n]
 *     -- hello-gpu ch.11 "GEMM-Like", section 11.1 (the definition of C_{m,n}
 *        and the worked 2x3 by 3x2 example, Fig. 11.1).
 *
 *   Storage is the TN layout of the AMD ROCm blog "FP16 GEMM optimization on
 *   AMD RDNA 3 and RDNA 4", section "What we compute": A row-major (M x K,
 *   A[m*lda + k]), B column-major (K x N, B[k + n*ldb]), so both are
 *   K-contiguous; C column-major with leading dimension ldc (C[m + n*ldc]).
 *
 *   The sum runs sequentially in k (k = 0, 1, ..., K-1) in IEEE double,
 *   starting from +0.0, and is rounded ONCE to the output format with
 *   round-to-nearest-even.  Products of two binary16 or two E4M3 values are
 *   exact in double.
 *
 *   Alongside C the oracle returns, per output,
 *     X[m,n] = the double sum before the final rounding, and
 *     S[m,n] = sum_k |A[m,k] * B[k,n]|  (the magnitude sum used by the
 *              acceptance tolerance), both in double.
 *
 *   Scaled-score variant (QK^T with the softmax's row statistics): see
 *   oracle_gemm_f16_tn_softmax_stats below.
 *
 *   Before the F8 GEMM, an operand may be quantised to E4M3 per tensor
 *   (oracle_quantize_e4m3 below; amax over the tensor, scale to 448).
 *
 *   F8 variant: A and B hold E4M3 codes; a = decode(qa), b = decode(qb);
 *   X = sum a*b (double), C = bf16_rne((X * scale_a) * scale_b) and
 *   S = (sum |a*b|) * scale_a * scale_b.  scale_a / scale_b are the
 *   dequantisation factors the caller passes with the codes.
 *
 * Parallelism: output columns n are distributed over OpenMP threads; each
 * output's k-loop is untouched, so the result does not depend on the thread
 * count.  Build: cc -O2 -fopenmp -shared -fPIC (no -ffast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* binary16 (IEEE 754-2008): 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits.  Exponent field 0 = zero/subnormal (value f * 2^-24),
 * field 31 = infinity (f == 0) or NaN (f != 0), otherwise (1024 + f) * 2^(e-25). */
double oracle_fp16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round a non-negative finite double to the nearest multiple of 2^q_exp,
 * ties to even; returns the integer multiple (as double, exact). */
static double round_to_quantum(double ax, int q_exp)
{
    double n = ldexp(ax, -q_exp);      /* exact: power-of-two scaling */
    double fl = floor(n);
    double diff = n - fl;              /* exact while n < 2^53 */
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16, round to nearest even, overflow to +-Inf, subnormals
 * kept, NaN -> quiet NaN with the input's sign. */
uint16_t oracle_fp16_encode(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return sign | 0x7e00;
    double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7c00;
    if (ax == 0.0) return sign;
    int e2;
    frexp(ax, &e2);                    /* ax in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                    /* ax in [2^E, 2^(E+1)) */
    if (E < -14) {                     /* subnormal range: quantum 2^-24 */
        double r = round_to_quantum(ax, -24);   /* 0 .. 1024 */
        return sign | (uint16_t)r;     /* r == 1024 is exactly 2^-14 (0x0400) */
    }
    if (E > 15) return sign | 0x7c00;
    double r = round_to_quantum(ax, E - 10);    /* 1024 .. 2048 */
    if (r >= 2048.0) { E += 1; r = 1024.0; }
    if (E > 15) return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/* bfloat16: the upper half of binary32 -- 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits.  double -> bf16 with one RNE rounding,
 * overflow to +-Inf, subnormals kept (quantum 2^-133), NaN -> quiet NaN. */
uint16_t oracle_bf16_encode(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return sign | 0x7fc0;
    double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7f80;
    if (ax == 0.0) return sign;
    int e2;
    frexp(ax, &e2);
    int E = e2 - 1;
    if (E < -126) {
        double r = round_to_quantum(ax, -133);  /* 0 .. 128 */
        return sign | (uint16_t)r;
    }
    if (E > 127) return sign | 0x7f80;
    double r = round_to_quantum(ax, E - 7);     /* 128 .. 256 */
    if (r >= 256.0) { E += 1; r = 128.0; }
    if (E > 127) return sign | 0x7f80;
    return sign | (uint16_t)(((E + 127) << 7) | ((int)r - 128));
}

double oracle_bf16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

/* OCP OFP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits, no infinities; S.1111.111 is NaN.  Exponent field 0 is zero or a
 * subnormal f * 2^-9; otherwise (8 + f) * 2^(e-10).  Largest finite 448. */
double oracle_e4m3_decode(uint8_t q)
{
    int sign = (q >> 7) & 1;
    int e = (q >> 3) & 0xf;
    int f = q & 7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

/* double -> E4M3, round to nearest even; magnitudes from 448 (the largest
 * finite E4M3 value) up -- Inf included -- give +-448 (saturation), NaN gives
 * the NaN code S.1111.111.  Zero keeps its sign.  Normal values have the
 * quantum 2^(E-3) for |x| in [2^E, 2^(E+1)), E >= -6; below 2^-6 the quantum
 * is 2^-9 (subnormals). */
uint8_t oracle_e4m3_encode(double x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return sign | 0x7f;
    double ax = fabs(x);
    if (ax >= 448.0) return sign | 0x7e;
    if (ax == 0.0) return sign;
    int e2;
    frexp(ax, &e2);
    int E = e2 - 1;                    /* ax in [2^E, 2^(E+1)) */
    if (E < -6) {
        double r = round_to_quantum(ax, -9);    /* 0 .. 8; 8 is exactly 2^-6 (0x08) */
        return sign | (uint8_t)r;
    }
    double r = round_to_quantum(ax, E - 3);     /* 8 .. 16 */
    if (r >= 16.0) { E += 1; r = 8.0; }
    return sign | (uint8_t)(((E + 7) << 3) | ((int)r - 8));
}

/* ------------------------------------------------------------------------- */
/* Per-tensor E4M3 quantisation with the amax over the whole tensor:
 *   amax = max |x|,  s_q = 448 / amax (binary32),  q = E4M3(binary32(x * s_q)),
 *   scale = amax / 448 (binary32),
 * with s_q = 0 for amax = 0 and s_q = FLT_MAX when 448 / amax overflows.  The
 * pages give no FP8 rule; this is the plain per-tensor scaling to the E4M3
 * maximum.  The code of each element is an integer decided by floating point,
 * so the oracle takes that decision in the precision the rule names (binary32
 * for s_q and for the product), not in double.
 * x_type: 0 binary32, 1 binary16, 2 bfloat16; x is rows x cols with row
 * stride ldx elements, q rows x cols with row stride ldq bytes. */
#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the quantiser needs binary32 arithmetic evaluated in binary32"
#endif

static double load_elem(const void *x, int x_type, int64_t i)
{
    if (x_type == 0) {
        float f;
        memcpy(&f, (const char *)x + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)x + 2 * i, 2);
    return x_type == 1 ? oracle_fp16_decode(h) : oracle_bf16_decode(h);
}

int oracle_quantize_e4m3(const void *x, int x_type, int64_t rows, int64_t cols, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *scale)
{
    if (x_type < 0 || x_type > 2 || rows < 0 || cols < 0) return -1;
    double amax = 0.0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            double v = fabs(load_elem(x, x_type, r * ldx + c));
            if (v > amax) amax = v;
        }
    float amax32 = (float)amax;        /* exact: every input is a binary32 value */
    float s_q = 0.0f;
    if (amax32 > 0.0f) {
        s_q = 448.0f / amax32;
        if (isinf(s_q)) s_q = FLT_MAX;
    }
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float xv = (float)load_elem(x, x_type, r * ldx + c);
            float prod = xv * s_q;
            q[r * ldq + c] = oracle_e4m3_encode((double)prod);
        }
    *scale = amax32 / 448.0f;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Decoding tables, filled once from the decoders above. */
static double g_f16[65536];
static double g_e4m3[256];
static int g_tables_ready = 0;

static void tables_init(void)
{
    if (g_tables_ready) return;
    for (int i = 0; i < 65536; ++i) g_f16[i] = oracle_fp16_decode((uint16_t)i);
    for (int i = 0; i < 256; ++i) g_e4m3[i] = oracle_e4m3_decode((uint8_t)i);
    g_tables_ready = 1;
}

/* One output of the F16 variant: the k-loop of the definition. */
static void dot_f16(int64_t K, const uint16_t *a_row, const uint16_t *b_col,
                    double *x_out, double *s_out)
{
    double x = 0.0, s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = g_f16[a_row[k]] * g_f16[b_col[k]];
        x += p;
        s += fabs(p);
    }
    *x_out = x;
    *s_out = s;
}

static void dot_e4m3(int64_t K, const uint8_t *a_row, const uint8_t *b_col,
                     double *x_out, double *s_out)
{
    double x = 0.0, s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = g_e4m3[a_row[k]] * g_e4m3[b_col[k]];
        x += p;
        s += fabs(p);
    }
    *x_out = x;
    *s_out = s;
}

/* Full F16 GEMM.  C (binary16 codes) is column-major with ldc; S and X, when
 * not NULL, are column-major with leading dimension M.  Returns 0, or -1 on
 * a bad argument. */
int oracle_gemm_f16_tn(int64_t M, int64_t N, int64_t K,
                       const uint16_t *A, int64_t lda,
                       const uint16_t *B, int64_t ldb,
                       uint16_t *C, int64_t ldc, double *S, double *X)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1) || ldc < (M > 1 ? M : 1)) return -1;
    tables_init();
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double x, s;
            dot_f16(K, A + m * lda, B + n * ldb, &x, &s);
            C[m + n * ldc] = oracle_fp16_encode(x);
            if (S) S[m + n * M] = s;
            if (X) X[m + n * M] = x;
        }
    }
    return 0;
}

/* Scaled scores and the softmax's row statistics (the QK^T step of attention,
 * followed by the two reductions a softmax over n needs):
 *   Y[m,n]     = scale * sum_k A[m,k] * B[k,n]          (double)
 *   C[m,n]     = binary16(Y[m,n])                       (one RNE rounding)
 *   row_max[m] = max_n Y[m,n]
 *   row_sum[m] = sum_n exp(Y[m,n] - row_max[m])         (double, n ascending)
 * S[m,n] (optional) = |scale| * sum_k |A[m,k] * B[k,n]|.  N = 0 leaves the
 * statistics unwritten. */
int oracle_gemm_f16_tn_softmax_stats(int64_t M, int64_t N, int64_t K,
                                     const uint16_t *A, int64_t lda,
                                     const uint16_t *B, int64_t ldb, double scale,
                                     uint16_t *C, int64_t ldc,
                                     double *row_max, double *row_sum, double *S)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1) || ldc < (M > 1 ? M : 1)) return -1;
    tables_init();
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        double mx = -INFINITY;
        for (int64_t n = 0; n < N; ++n) {
            double x, s;
            dot_f16(K, A + m * lda, B + n * ldb, &x, &s);
            const double y = scale * x;
            C[m + n * ldc] = oracle_fp16_encode(y);
            if (S) S[m + n * M] = fabs(scale) * s;
            if (y > mx) mx = y;
        }
        if (N == 0) continue;
        double sum = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double x, s;
            dot_f16(K, A + m * lda, B + n * ldb, &x, &s);
            sum += exp(scale * x - mx);
        }
        row_max[m] = mx;
        row_sum[m] = sum;
    }
    return 0;
}

/* F16 outputs at `count` chosen positions (m_idx[i], n_idx[i]); c_out gets the
 * binary16 codes, s_out / x_out (optional) the magnitude and exact sums. */
int oracle_gemm_f16_tn_at(int64_t M, int64_t N, int64_t K,
                          const uint16_t *A, int64_t lda,
                          const uint16_t *B, int64_t ldb,
                          int64_t count, const int64_t *m_idx, const int64_t *n_idx,
                          uint16_t *c_out, double *s_out, double *x_out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1)) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N) return -1;
    tables_init();
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double x, s;
        dot_f16(K, A + m_idx[i] * lda, B + n_idx[i] * ldb, &x, &s);
        c_out[i] = oracle_fp16_encode(x);
        if (s_out) s_out[i] = s;
        if (x_out) x_out[i] = x;
    }
    return 0;
}

/* Full F8 (E4M3 in, bf16 out) GEMM; layouts as for the F16 variant. */
int oracle_gemm_f8e4m3_tn(int64_t M, int64_t N, int64_t K,
                          const uint8_t *A, int64_t lda,
                          const uint8_t *B, int64_t ldb,
                          float scale_a, float scale_b,
                          uint16_t *C, int64_t ldc, double *S, double *X)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1) || ldc < (M > 1 ? M : 1)) return -1;
    tables_init();
    const double sa = (double)scale_a, sb = (double)scale_b;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double x, s;
            dot_e4m3(K, A + m * lda, B + n * ldb, &x, &s);
            C[m + n * ldc] = oracle_bf16_encode((x * sa) * sb);
            if (S) S[m + n * M] = (s * sa) * sb;
            if (X) X[m + n * M] = x;
        }
    }
    return 0;
}

int oracle_gemm_f8e4m3_tn_at(int64_t M, int64_t N, int64_t K,
                             const uint8_t *A, int64_t lda,
                             const uint8_t *B, int64_t ldb,
                             float scale_a, float scale_b,
                             int64_t count, const int64_t *m_idx, const int64_t *n_idx,
                             uint16_t *c_out, double *s_out, double *x_out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (K > 1 ? K : 1)) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N) return -1;
    tables_init();
    const double sa = (double)scale_a, sb = (double)scale_b;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double x, s;
        dot_e4m3(K, A + m_idx[i] * lda, B + n_idx[i] * ldb, &x, &s);
        c_out[i] = oracle_bf16_encode((x * sa) * sb);
        if (s_out) s_out[i] = (s * sa) * sb;
        if (x_out) x_out[i] = x;
    }
    return 0;
}

/* Threads the OpenMP runtime will use for the loops above. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * synth.c -- seeded synthetic inputs for the TN GEMM workloads.
 *
 * This module only MAKES inputs; it holds none of the GEMM's arithmetic and is
 * shared by the tests and the benchmark (the CUDA library and the CPU oracle
 * never include it).
 *
 * Random stream: element i of a stream with seed s is the i-th output of the
 * SplitMix64 generator (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the finaliser constants are Vigna's
 * published SplitMix64 variant) started at state s:
 *     z = s + (i + 1) * 0x9E3779B97F4A7C15
 *     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *     z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *     z =  z ^ (z >> 31)
 * It is counter based, so any element can be produced on its own and the
 * result does not depend on the thread count.
 *
 *   sign     : bit 63 of z_i picks -1 (set) or +1.
 *   gaussian : Box-Muller on two draws, u1 = ((z_{2i} >> 11) + 1) 2^-53 in
 *              (0,1], u2 = (z_{2i+1} >> 11) 2^-53 in [0,1):
 *              x_i = sqrt(-2 ln u1) cos(2 pi u2)    (double).
 *   fp16     : x_i rounded once to binary16, nearest-even.
 *   e4m3     : clamp(x_i * mult, -448, 448) rounded once to OCP E4M3FN,
 *              nearest-even (the clamp makes it saturating).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64_at(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline double gauss_at(uint64_t seed, uint64_t i)
{
    const double two_m53 = 1.0 / 9007199254740992.0;
    double u1 = (double)((splitmix64_at(seed, 2 * i) >> 11) + 1) * two_m53;
    double u2 = (double)(splitmix64_at(seed, 2 * i + 1) >> 11) * two_m53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* Round the 53-bit significand `sig` right by `shift` bits, ties to even. */
static inline uint64_t rne_shift(uint64_t sig, int shift)
{
    if (shift <= 0) return sig << (-shift);
    if (shift > 60) return 0;
    uint64_t q = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
    return q;
}

/* finite double -> binary16 by its bit fields (inputs here are |x| < 2^15). */
static inline uint16_t to_fp16(double x)
{
    uint64_t u;
    memcpy(&u, &x, 8);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000);
    int bexp = (int)((u >> 52) & 0x7ff);
    if (bexp == 0) return sign;                 /* zero (double subnormals flush) */
    int e = bexp - 1023;
    uint64_t sig = (u & ((1ull << 52) - 1)) | (1ull << 52);
    if (e >= -14) {
        uint64_t q = rne_shift(sig, 42);        /* 11-bit significand */
        if (q == 2048) { q = 1024; ++e; }
        if (e + 15 >= 31) return sign | 0x7c00;
        return sign | (uint16_t)(((e + 15) << 10) | (int)(q - 1024));
    }
    uint64_t q = rne_shift(sig, 42 + (-14 - e)); /* subnormal quantum 2^-24 */
    return sign | (uint16_t)q;                  /* q == 1024 encodes 2^-14 */
}

/* finite double with |x| <= 448 -> E4M3FN by its bit fields. */
static inline uint8_t to_e4m3(double x)
{
    uint64_t u;
    memcpy(&u, &x, 8);
    uint8_t sign = (uint8_t)((u >> 56) & 0x80);
    int bexp = (int)((u >> 52) & 0x7ff);
    if (bexp == 0) return sign;
    int e = bexp - 1023;
    uint64_t sig = (u & ((1ull << 52) - 1)) | (1ull << 52);
    if (e >= -6) {
        uint64_t q = rne_shift(sig, 49);        /* 4-bit significand */
        if (q == 16) { q = 8; ++e; }
        int field = e + 7;
        if (field > 15 || (field == 15 && q - 8 == 7)) return sign | 0x7e;
        return sign | (uint8_t)((field << 3) | (int)(q - 8));
    }
    uint64_t q = rne_shift(sig, 49 + (-6 - e));  /* subnormal quantum 2^-9 */
    return sign | (uint8_t)q;                   /* q == 8 encodes 2^-6 */
}

/* finite double -> bfloat16 by its bit fields (inputs here are normal,
 * |x| < 2^127; smaller than 2^-126 gives signed zero). */
static inline uint16_t to_bf16(double x)
{
    uint64_t u;
    memcpy(&u, &x, 8);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000);
    int bexp = (int)((u >> 52) & 0x7ff);
    int e = bexp - 1023;
    if (bexp == 0 || e < -126) return sign;
    uint64_t sig = (u & ((1ull << 52) - 1)) | (1ull << 52);
    uint64_t q = rne_shift(sig, 45);            /* 8-bit significand */
    if (q == 256) { q = 128; ++e; }
    return sign | (uint16_t)(((e + 127) << 7) | (int)(q - 128));
}

void synth_sign_fp16(uint16_t *out, int64_t n, uint64_t seed)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (splitmix64_at(seed, (uint64_t)i) >> 63) ? 0xbc00 : 0x3c00;
}

void synth_gauss_f64(double *out, int64_t n, uint64_t seed)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gauss_at(seed, (uint64_t)i);
}

void synth_gauss_fp16(uint16_t *out, int64_t n, uint64_t seed)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = to_fp16(gauss_at(seed, (uint64_t)i));
}

void synth_gauss_bf16(uint16_t *out, int64_t n, uint64_t seed)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(gauss_at(seed, (uint64_t)i));
}

double synth_gauss_absmax(int64_t n, uint64_t seed)
{
    double mx = 0.0;
    #pragma omp parallel for schedule(static) reduction(max : mx)
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs(gauss_at(seed, (uint64_t)i));
        if (a > mx) mx = a;
    }
    return mx;
}

void synth_gauss_e4m3(uint8_t *out, int64_t n, uint64_t seed, double mult)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double v = gauss_at(seed, (uint64_t)i) * mult;
        if (v > 448.0) v = 448.0;
        if (v < -448.0) v = -448.0;
        out[i] = to_e4m3(v);
    }
}

/* Generic helpers for the tests: raw stream values and conversions of given
 * doubles (so the converters can be checked against library routines). */
void synth_raw(uint64_t *out, int64_t n, uint64_t seed)
{
    for (int64_t i = 0; i < n; ++i) out[i] = splitmix64_at(seed, (uint64_t)i);
}

void synth_f64_to_fp16(uint16_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = to_fp16(in[i]);
}

void synth_f64_to_e4m3(uint8_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = in[i];
        if (v > 448.0) v = 448.0;
        if (v < -448.0) v = -448.0;
        out[i] = to_e4m3(v);
    }
}

void synth_f64_to_bf16(uint16_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(in[i]);
}

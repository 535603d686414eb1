/*
 * ORACLE for the stochastic-rounding option of the bf16 outputs -- TEST
 * INFRASTRUCTURE ONLY.
 *
 * The encoder page's wte and wpe kernels round their fp32 sums to bf16
 * stochastically, with a deterministic seed per element; the page calls a
 * helper whose body it does not print. This file states the option the
 * library offers (mmbwd_run_sr), from the definition of stochastic rounding:
 * a value between two neighbouring bf16 numbers lo < |x| < hi (same sign)
 * becomes hi with probability (|x| - lo) / (hi - lo), else lo. Only the tests,
 * the smoke check and the benchmark's CPU leg may load it; it shares no code
 * with the CUDA library.
 *
 * Readings taken where the page leaves a step open:
 *   - The draw: element e (row-major index) of output tensor k takes the
 *     16-bit integer r = bits 16 (e mod 4) .. 16 (e mod 4) + 15 of output
 *     number n = (k << 58) | (e / 4) of the splitmix64 generator seeded with
 *     the caller's seed (Steele, Lea and Flood 2014; the n-th output, counting
 *     from 0, is mix(seed + (n + 1) * 0x9E3779B97F4A7C15)).
 *   - The decision: with f = 65536 (|x| - lo) / (hi - lo) (an integer for an
 *     fp32 x), the value rounds up exactly when r + f >= 65536, so that
 *     P(up) = f / 65536.
 *   - The value rounded is the fp32 value of the exact result (the type the
 *     library accumulates in); infinities and NaNs keep their class (NaN quiet).
 *
 * Parity pins (CPU tests, independent of this code): published splitmix64
 * outputs, the decision rule restated on bit patterns, representable values
 * kept, unbiasedness and independence of the draws, distinct tensors.
 *
 * ORACLE_MUTANT 19..22 plants one mistake each (see the #if blocks).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* The n-th output (n = 0, 1, ...) of splitmix64 seeded with `seed`. */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t n) {
    uint64_t z = seed + (n + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* The 16-bit draw of element e of tensor k. */
uint32_t oracle_sr_draw(uint64_t seed, int k, int64_t e) {
#if ORACLE_MUTANT == 21 /* the tensor is not part of the counter */
    (void)k;
    const uint64_t w = oracle_splitmix64(seed, (uint64_t)e >> 2);
#else
    const uint64_t w = oracle_splitmix64(seed, ((uint64_t)k << 58) | ((uint64_t)e >> 2));
#endif
#if ORACLE_MUTANT == 20 /* the same 16 bits for the four elements of a word */
    return (uint32_t)w & 0xFFFFu;
#else
    return (uint32_t)(w >> (16 * (e & 3))) & 0xFFFFu;
#endif
}

/* x (an fp32 value) rounded to bf16 with draw r; returns the bf16 bit pattern. */
static uint16_t round_one(float x, uint32_t r) {
    uint32_t xb;
    memcpy(&xb, &x, 4);
    const uint16_t sign = (uint16_t)((xb >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)((xb >> 16) | 0x40u);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
    if (x == 0.0f) return sign;
    const double a = fabs((double)x);
    int E;
    frexp(a, &E); /* a = m 2^E, 0.5 <= m < 1 */
    /* bf16 keeps 8 significant bits: neighbours 2^(E-8) apart in this binade,
       2^-133 apart below 2^-126 (the subnormal spacing) */
#if ORACLE_MUTANT == 22 /* the spacing of the binade above */
    int se = E - 7;
#else
    int se = E - 8;
#endif
    if (se < -133) se = -133;
    const double sp = ldexp(1.0, se);
    const double lo = floor(a / sp) * sp;
    const double f = (a - lo) / sp * 65536.0; /* exact: x is a multiple of sp / 65536 */
#if ORACLE_MUTANT == 19 /* the decision taken on the other side of the draw */
    const int up = (double)r < f;
#else
    const int up = (double)r + f >= 65536.0;
#endif
    const float y = (float)(lo + (up ? sp : 0.0)); /* representable, or 2^128 -> inf */
    uint32_t yb;
    memcpy(&yb, &y, 4);
    return (uint16_t)((yb >> 16) | sign);
}

/*
 * out[i] = stochastic bf16 rounding of (float) v[i], the element index of
 * v[i] being e0 + i in tensor k.
 */
void oracle_sr_round(const double* v, uint16_t* out, int64_t n, uint64_t seed, int k, int64_t e0) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_one((float)v[i], oracle_sr_draw(seed, k, e0 + i));
}

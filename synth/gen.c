/*
 * Seeded synthetic inputs for the matmul_backward workloads.
 *
 * This module only draws random numbers and rounds them to a storage type.
 * It holds none of the backward pass's arithmetic, so both the CPU oracle and
 * the CUDA path can take their inputs from it without sharing any of the
 * method's code.
 *
 * Generator (counter-based, so any element can be drawn on its own and the
 * output does not depend on the number of threads):
 *   key       = mix64(seed XOR (stream * 0xD6E8FEB86659FD93))
 *   word(c)   = mix64(key + (c + 1) * 0x9E3779B97F4A7C15)     (the c-th output
 *               of a splitmix64 sequence whose state starts at key)
 *   U(c)      = ((word(c) >> 11) + 1) * 2^-53                 (uniform on (0,1])
 *   Box-Muller on the pair (U(2j), U(2j+1)):
 *     r = sqrt(-2 ln U(2j)), phi = 2 pi U(2j+1)
 *     z(2j) = r cos(phi),  z(2j+1) = r sin(phi)
 *   value(i)  = mean + std * z(i), in double, then rounded to the storage type:
 *               f32 by round-to-nearest-even, bf16 by rounding to f32 first and
 *               then to bf16 with round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_F32 0
#define SYNTH_BF16 1
#define SYNTH_F64 2

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed ^ (stream * 0xD6E8FEB86659FD93ULL));
}

static inline double uniform01(uint64_t key, uint64_t c) {
    uint64_t w = mix64(key + (c + 1) * 0x9E3779B97F4A7C15ULL);
    return (double)((w >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double std_normal(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t j = i >> 1;
    double u1 = uniform01(key, 2 * j);
    double u2 = uniform01(key, 2 * j + 1);
    double r = sqrt(-2.0 * log(u1));
    double phi = two_pi * u2;
    return (i & 1) ? r * sin(phi) : r * cos(phi);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

static inline void store_value(void* out, int64_t i, int dtype, double v) {
    if (dtype == SYNTH_F32) {
        ((float*)out)[i] = (float)v;
    } else if (dtype == SYNTH_BF16) {
        ((uint16_t*)out)[i] = f32_to_bf16_rne((float)v);
    } else {
        ((double*)out)[i] = v;
    }
}

/* Fill out[0..n) with mean + std * N(0,1) from (seed, stream). Returns 0, or -1
 * on a bad dtype or negative n. */
int synth_normal(void* out, int64_t n, int dtype, uint64_t seed, uint64_t stream, double mean,
                 double std) {
    if (n < 0 || dtype < 0 || dtype > 2) return -1;
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) store_value(out, i, dtype, mean + std * std_normal(key, (uint64_t)i));
    return 0;
}

/* Language-model-head gradient stand-in, row-major (rows, cols):
 *   value(r, c) = std * z(r*cols + c) from (seed, stream_noise)
 *               + spike  if c == floor(U_r * cols), U_r = U(r) from (seed, stream_index)
 * the sum being formed in double before the single rounding to the storage
 * type. This mimics softmax-minus-one-hot: small dense values plus one
 * negative entry per row. */
int synth_lmhead_dout(void* out, int64_t rows, int64_t cols, int dtype, uint64_t seed,
                      uint64_t stream_noise, uint64_t stream_index, double std, double spike) {
    if (rows < 0 || cols <= 0 || dtype < 0 || dtype > 2) return -1;
    uint64_t kn = stream_key(seed, stream_noise);
    uint64_t ki = stream_key(seed, stream_index);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t hot = (int64_t)floor(uniform01(ki, (uint64_t)r) * (double)cols);
        if (hot >= cols) hot = cols - 1; /* U == 1 exactly */
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            double v = std * std_normal(kn, (uint64_t)i);
            if (c == hot) v += spike;
            store_value(out, i, dtype, v);
        }
    }
    return 0;
}

/* The hot column of row r used by synth_lmhead_dout (for tests). */
int64_t synth_lmhead_hot_index(int64_t r, int64_t cols, uint64_t seed, uint64_t stream_index) {
    uint64_t ki = stream_key(seed, stream_index);
    int64_t hot = (int64_t)floor(uniform01(ki, (uint64_t)r) * (double)cols);
    return hot >= cols ? cols - 1 : hot;
}

/* Uniform draws on (0,1] (for tests of the generator itself). */
int synth_uniform(double* out, int64_t n, uint64_t seed, uint64_t stream) {
    if (n < 0) return -1;
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = uniform01(key, (uint64_t)i);
    return 0;
}

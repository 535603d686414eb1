/*
 * ORACLE for the GPT-2 encoder backward -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain CPU statement of what the encoder backward of llm.c's
 * llmc/encoder.cuh computes (the forward adds a token row of wte and a
 * position row of wpe; the backward sends the gradient of each output row to
 * both). Only the tests, the smoke check and the benchmark's CPU leg may load
 * it; the CUDA library never does, and it shares no code with it.
 *
 * Shapes: dout (B, T, C); inp (B, T) token ids in [0, V); dwte (V, C); dwpe (T, C).
 *
 *   dwte[ix, c] = dwte_init[ix, c] + sum over (b, t) with inp[b, t] == ix of dout[b, t, c]
 *   dwpe[t, c]  = dwpe_init[t, c]  + sum over b of dout[b, t, c]
 *
 * Readings taken where the page leaves a step open:
 *   - Both gradients accumulate into what the caller passes (the page's kernels
 *     read dwte / dwpe and add).
 *   - Sums are formed in double in a fixed order (b then t ascending for dwte;
 *     b ascending for dwpe) and added to the initial value once; outputs stay
 *     in double. The page rounds its fp32 sums to bf16 stochastically; the
 *     library rounds once to nearest-even, like every other output here.
 *   - A token id outside [0, V) is an error (this function returns -2).
 *
 * Parity pins (CPU tests, independent of this code): exact integer sums,
 * conservation of the column totals, one-hot and single-token cases, and
 * invariance under reordering of the (b, t) positions.
 *
 * ORACLE_MUTANT 16..18 plants one mistake each (see the #if blocks).
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ENC_F32 0
#define ENC_BF16 1
#define ENC_F64 2

static double enc_load(const void* p, int dtype, int64_t i) {
    if (dtype == ENC_F32) return (double)((const float*)p)[i];
    if (dtype == ENC_F64) return ((const double*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/*
 * dwte (V*C) and dwpe (T*C) in double. Inits may be NULL (zero).
 * Returns 0, -1 on bad sizes, -2 on a token id outside [0, V).
 */
int oracle_encoder_backward(double* dwte, double* dwpe, const void* dwte_init, const void* dwpe_init,
                            const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C, int64_t V,
                            int dtype) {
    if (B < 0 || T < 0 || C < 0 || V < 0 || dtype < 0 || dtype > 2) return -1;
    for (int64_t bt = 0; bt < B * T; ++bt)
        if (inp[bt] < 0 || inp[bt] >= V) return -2;
    for (int64_t i = 0; i < V * C; ++i) dwte[i] = 0.0;
    for (int64_t i = 0; i < T * C; ++i) dwpe[i] = 0.0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t) {
            int64_t bt = b * T + t;
#if ORACLE_MUTANT == 16 /* wrong index: the token of the neighbouring position */
            int64_t ix = inp[(bt + 1) % (B * T)];
#else
            int64_t ix = inp[bt];
#endif
            for (int64_t c = 0; c < C; ++c) {
                double d = enc_load(dout, dtype, bt * C + c);
                dwte[ix * C + c] += d;
#if ORACLE_MUTANT == 17 /* position gradient summed over t instead of b */
                dwpe[b % T * C + c] += d;
#else
                dwpe[t * C + c] += d;
#endif
            }
        }
    for (int64_t i = 0; i < V * C; ++i)
        if (dwte_init) dwte[i] += enc_load(dwte_init, dtype, i);
    for (int64_t i = 0; i < T * C; ++i) {
#if ORACLE_MUTANT == 18 /* '=' instead of '+=': the initial dwpe is dropped */
        (void)dwpe_init;
#else
        if (dwpe_init) dwpe[i] += enc_load(dwpe_init, dtype, i);
#endif
    }
    return 0;
}

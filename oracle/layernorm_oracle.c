/*
 * ORACLE for layernorm_backward -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU statement of the GPT-2 LayerNorm backward, written from the
 * CPU reference `layernorm_backward_cpu` of llm.c's dev/cuda/layernorm_backward.cu
 * (and `layernorm_forward_cpu` of the same file, which makes the cached row
 * statistics). Only the tests, the smoke check and the benchmark's CPU leg may
 * load it; the CUDA library never does, and it shares no code with it.
 *
 * Shapes (row-major, contiguous): inp, dout, dinp (BT, C); weight, bias,
 * dweight, dbias (C); mean, rstd (BT), with BT = B*T.
 *
 * Forward (layernorm_forward_cpu), per row bt:
 *   m = (1/C) sum_i x_i,  v = (1/C) sum_i (x_i - m)^2,  s = 1 / sqrt(v + 1e-5)
 *   out_i = s (x_i - m) w_i + b_i;  mean[bt] = m, rstd[bt] = s
 *
 * Backward (layernorm_backward_cpu), per row bt with m = mean[bt], s = rstd[bt]:
 *   n_i  = (x_i - m) s                 (the normalised input)
 *   g_i  = w_i dout_i                  (gradient reaching n)
 *   a    = (1/C) sum_i g_i,   c = (1/C) sum_i g_i n_i       (first pass)
 *   dinp[bt,i] += s (g_i - a - n_i c)                        (second pass)
 *   dweight[i] += sum_bt n_i dout_i,   dbias[i] += sum_bt dout_i
 *
 * Readings taken where the page leaves a step open:
 *   - All three gradients accumulate into what the caller passes (`+=` in
 *     layernorm_backward_cpu); the initial values are explicit arguments here
 *     because the outputs are double.
 *   - mean and rstd are inputs, as cached by the forward; they are read with
 *     their own element type (fp32 as in the CPU reference, or double).
 *   - Every sum is formed in double, in the page's loop order (i ascending for
 *     the two row means; b then t ascending for dweight and dbias), and added to
 *     the initial value once at the end. Outputs stay in double.
 * Compiled with -ffp-contract=off. The OpenMP build splits the dinp rows over
 * threads; the order of operations inside each element is unchanged.
 *
 * Parity pins (CPU tests, independent of this code): the library LayerNorm of
 * torch in float64 (forward values, and the input, weight and bias gradients by
 * autograd), central differences of L = sum(dout * out) through the forward,
 * shift invariance of each row's input gradient, exact column sums for dbias.
 *
 * ORACLE_MUTANT 11..15 plants one mistake each (see the #if blocks).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define LN_F32 0
#define LN_BF16 1
#define LN_F64 2

static double ln_load(const void* p, int dtype, int64_t i) {
    if (dtype == LN_F32) return (double)((const float*)p)[i];
    if (dtype == LN_F64) return ((const double*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static int ln_bad(int64_t BT, int64_t C, int dtype) { return BT < 0 || C < 0 || dtype < 0 || dtype > 2; }

/*
 * Forward of the layer norm in double (eps 1e-5). out (BT*C), mean (BT), rstd (BT);
 * out may be NULL (statistics only); bias may be NULL (zero).
 */
int oracle_layernorm_forward(double* out, double* mean, double* rstd, const void* inp, const void* weight,
                             const void* bias, int64_t BT, int64_t C, int dtype) {
    if (ln_bad(BT, C, dtype) || C == 0) return -1;
    for (int64_t bt = 0; bt < BT; ++bt) {
        double m = 0.0;
        for (int64_t i = 0; i < C; ++i) m += ln_load(inp, dtype, bt * C + i);
        m = m / (double)C;
        double v = 0.0;
        for (int64_t i = 0; i < C; ++i) {
            double d = ln_load(inp, dtype, bt * C + i) - m;
            v += d * d;
        }
        v = v / (double)C;
        double s = 1.0 / sqrt(v + 1e-5);
        if (out)
            for (int64_t i = 0; i < C; ++i) {
                double n = s * (ln_load(inp, dtype, bt * C + i) - m);
                out[bt * C + i] = n * ln_load(weight, dtype, i) + (bias ? ln_load(bias, dtype, i) : 0.0);
            }
        mean[bt] = m;
        rstd[bt] = s;
    }
    return 0;
}

/*
 * dinp rows of the backward. For r in [0, nrows): bt = rows ? rows[r] : r,
 *   out[r*C + i] = dinp_init[bt,i] + s (g_i - a - n_i c)
 * dinp_init may be NULL (zero). mean/rstd are read as stat_dtype (LN_F32 or LN_F64).
 */
int oracle_layernorm_dinp_rows(double* out, const int64_t* rows, int64_t nrows, const void* dinp_init,
                               const void* dout, const void* inp, const void* weight, const void* mean,
                               const void* rstd, int stat_dtype, int64_t BT, int64_t C, int dtype) {
    if (ln_bad(BT, C, dtype) || nrows < 0 || (!rows && nrows != BT)) return -1;
    if (stat_dtype != LN_F32 && stat_dtype != LN_F64) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= BT)) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bt = rows ? rows[r] : r;
        double m = ln_load(mean, stat_dtype, bt), s = ln_load(rstd, stat_dtype, bt);
        /* first pass: the two row means */
        double a = 0.0, c = 0.0;
        for (int64_t i = 0; i < C; ++i) {
            double n = (ln_load(inp, dtype, bt * C + i) - m) * s;
            double g = ln_load(weight, dtype, i) * ln_load(dout, dtype, bt * C + i);
            a += g;
            c += g * n;
        }
        a = a / (double)C;
        c = c / (double)C;
        /* second pass: the input gradient */
        for (int64_t i = 0; i < C; ++i) {
            double n = (ln_load(inp, dtype, bt * C + i) - m) * s;
            double g = ln_load(weight, dtype, i) * ln_load(dout, dtype, bt * C + i);
#if ORACLE_MUTANT == 11 /* dropped term: the mean of g is not subtracted */
            double dval = g - n * c;
#elif ORACLE_MUTANT == 12 /* wrong sign of the third term */
            double dval = g - a + n * c;
#elif ORACLE_MUTANT == 13 /* final scale squared */
            double dval = (g - a - n * c) * s;
#else
            double dval = g - a - n * c;
#endif
            dval *= s;
            out[r * C + i] = (dinp_init ? ln_load(dinp_init, dtype, bt * C + i) : 0.0) + dval;
        }
    }
    return 0;
}

/*
 * dweight and dbias of the backward (length C each):
 *   dweight[i] = dweight_init[i] + sum_bt n_i dout_i,  dbias[i] = dbias_init[i] + sum_bt dout_i
 * Inits may be NULL (zero).
 */
int oracle_layernorm_params(double* dweight, double* dbias, const void* dweight_init, const void* dbias_init,
                            const void* dout, const void* inp, const void* mean, const void* rstd,
                            int stat_dtype, int64_t BT, int64_t C, int dtype) {
    if (ln_bad(BT, C, dtype)) return -1;
    if (stat_dtype != LN_F32 && stat_dtype != LN_F64) return -1;
    for (int64_t i = 0; i < C; ++i) dweight[i] = dbias[i] = 0.0;
    for (int64_t bt = 0; bt < BT; ++bt) {
        double m = ln_load(mean, stat_dtype, bt), s = ln_load(rstd, stat_dtype, bt);
        for (int64_t i = 0; i < C; ++i) {
            double d = ln_load(dout, dtype, bt * C + i);
#if ORACLE_MUTANT == 14 /* the raw input instead of the normalised one */
            double n = ln_load(inp, dtype, bt * C + i);
            (void)m;
            (void)s;
#else
            double n = (ln_load(inp, dtype, bt * C + i) - m) * s;
#endif
            dbias[i] += d;
            dweight[i] += n * d;
        }
    }
    for (int64_t i = 0; i < C; ++i) {
#if ORACLE_MUTANT == 15 /* '=' instead of '+=': the initial dbias is dropped */
        (void)dbias_init;
#else
        if (dbias_init) dbias[i] += ln_load(dbias_init, dtype, i);
#endif
        if (dweight_init) dweight[i] += ln_load(dweight_init, dtype, i);
    }
    return 0;
}

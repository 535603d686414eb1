/*
 * ORACLE for matmul_backward -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the GPT-2 linear-layer
 * backward computes, written from the CPU reference `matmul_backward_cpu` of
 * llm.c's dev/cuda/matmul_backward.cu. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the CUDA library never does, and it
 * shares no code with the CUDA library.
 *
 * Shapes (row-major, contiguous, as in matmul_backward_cpu's indexing):
 *   dout (BT, OC), inp (BT, C), weight (OC, C)  -> dinp (BT, C), dweight (OC, C), dbias (OC)
 *   with BT = B*T.
 *
 * What it computes (matmul_backward_cpu, "backward into inp" and "backward into
 * weight/bias" loops):
 *   dinp[bt,i]    = dinp_init[bt,i]    + sum_o  dout[bt,o] * weight[o,i]
 *   dweight[o,i]  = dweight_init[o,i]  + sum_bt dout[bt,o] * inp[bt,i]
 *   dbias[o]      = sum_bt dout[bt,o]            (overwritten, never accumulated)
 *
 * Readings taken where the page leaves a step open:
 *   - The page accumulates dinp/dweight in float and the bias in double; here
 *     every sum is accumulated in double, inputs being converted exactly.
 *   - The sum over o (for dinp) and over bt (for dweight, dbias) is formed first,
 *     in the page's loop order (o ascending; b then t ascending), and added to the
 *     initial value once at the end.
 *   - dbias is overwritten (`dbias[o] = sum` on the page), not accumulated.
 *   - Outputs stay in double: no rounding to the storage type.
 * Compiled with -ffp-contract=off so that no fused multiply-add changes the
 * rounding between machines. The single-threaded and OpenMP builds come from
 * this one source; the per-element order of operations is the same in both.
 *
 * Parity pins (checked by the CPU tests, independent of this code): brute
 * force in exact integer arithmetic, the column-sum invariant of dbias,
 * adjoint identities, central finite differences of the scalar
 * L = sum(dout * (inp weight^T + bias)), and special cases (identity weight,
 * one-hot dout, zero dout).
 *
 * The file also states the forward of the layer (oracle_forward_rows).
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake so that
 * the tests can show that their pins catch it; it is never set in a real build.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

/* Exact value of element i of a typed array. */
static double load(const void* p, int dtype, int64_t i) {
    if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
    if (dtype == ORACLE_F64) return ((const double*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static int bad_args(int64_t BT, int64_t C, int64_t OC, int dtype) {
    return BT < 0 || C < 0 || OC < 0 || dtype < 0 || dtype > 2;
}

/*
 * dinp rows. For r in [0, nrows): bt = rows ? rows[r] : r, and
 *   out[r*C + i] = dinp_init[bt,i] + sum_{o=0..OC-1} dout[bt,o] * weight[o,i]
 * dinp_init may be NULL (zero). Returns 0, or -1 on bad arguments.
 */
int oracle_dinp_rows(double* out, const int64_t* rows, int64_t nrows, const void* dinp_init,
                     const void* dout, const void* weight, int64_t BT, int64_t C, int64_t OC,
                     int dtype) {
    if (bad_args(BT, C, OC, dtype) || nrows < 0 || (!rows && nrows != BT)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= BT)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bt = rows ? rows[r] : r;
        double* acc = out + r * C;
        for (int64_t i = 0; i < C; ++i) acc[i] = 0.0;
        for (int64_t o = 0; o < OC; ++o) {
#if ORACLE_MUTANT == 1 /* dropped term: the last output channel is skipped */
            if (o == OC - 1) continue;
#endif
            double d = load(dout, dtype, bt * OC + o);
            for (int64_t i = 0; i < C; ++i) {
#if ORACLE_MUTANT == 2 /* wrong index: the weight column is shifted by one */
                acc[i] += load(weight, dtype, o * C + (i + 1) % C) * d;
#else
                acc[i] += load(weight, dtype, o * C + i) * d;
#endif
            }
        }
        for (int64_t i = 0; i < C; ++i) {
#if ORACLE_MUTANT == 3 /* '=' instead of '+=': the initial value is dropped */
            (void)dinp_init;
#else
            if (dinp_init) acc[i] += load(dinp_init, dtype, bt * C + i);
#endif
        }
    }
    return 0;
}

/*
 * dweight rows (and optionally dbias). For r in [0, nrows): o = rows ? rows[r] : r,
 *   out[r*C + i]  = dweight_init[o,i] + sum_{bt=0..BT-1} dout[bt,o] * inp[bt,i]
 *   dbias_out[r]  = sum_{bt=0..BT-1} dout[bt,o]          (when dbias_out != NULL)
 * dweight_init may be NULL (zero). Returns 0, or -1 on bad arguments.
 */
int oracle_dweight_rows(double* out, double* dbias_out, const int64_t* rows, int64_t nrows,
                        const void* dweight_init, const void* dout, const void* inp, int64_t BT,
                        int64_t C, int64_t OC, int dtype) {
    if (bad_args(BT, C, OC, dtype) || nrows < 0 || (!rows && nrows != OC)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= OC)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t o = rows ? rows[r] : r;
        double* acc = out + r * C;
        double sum = 0.0;
        for (int64_t i = 0; i < C; ++i) acc[i] = 0.0;
        for (int64_t bt = 0; bt < BT; ++bt) {
#if ORACLE_MUTANT == 4 /* wrong index: dout read from the neighbouring channel */
            double d = load(dout, dtype, bt * OC + (o + 1) % OC);
#else
            double d = load(dout, dtype, bt * OC + o);
#endif
#if ORACLE_MUTANT == 5 /* off-by-one: the bias sum misses the last row */
            if (bt < BT - 1) sum += d;
#elif ORACLE_MUTANT == 6 /* wrong sign of the bias gradient */
            sum -= d;
#else
            sum += d;
#endif
            for (int64_t i = 0; i < C; ++i) {
#if ORACLE_MUTANT == 7 /* transposed operand: inp indexed by (i, bt) on the square case */
                acc[i] += load(inp, dtype, (BT == C ? i * C + bt : bt * C + i)) * d;
#else
                acc[i] += load(inp, dtype, bt * C + i) * d;
#endif
            }
        }
        if (dweight_init)
            for (int64_t i = 0; i < C; ++i) acc[i] += load(dweight_init, dtype, o * C + i);
#if ORACLE_MUTANT == 8 /* single-precision accumulation of the bias sum */
        sum = (double)(float)sum;
#endif
        if (dbias_out) dbias_out[r] = sum;
    }
    return 0;
}

/*
 * The whole backward pass, in the argument order of matmul_backward_cpu (with
 * the initial gradients passed explicitly because the outputs are double):
 *   dinp (BT*C), dweight (OC*C), dbias (OC, or NULL to skip the bias).
 */
int oracle_matmul_backward(double* dinp, double* dweight, double* dbias, const void* dout,
                           const void* inp, const void* weight, const void* dinp_init,
                           const void* dweight_init, int64_t B, int64_t T, int64_t C, int64_t OC,
                           int dtype) {
    if (B < 0 || T < 0) return -1;
    int64_t BT = B * T;
    if (oracle_dinp_rows(dinp, NULL, BT, dinp_init, dout, weight, BT, C, OC, dtype)) return -1;
    return oracle_dweight_rows(dweight, dbias, NULL, OC, dweight_init, dout, inp, BT, C, OC, dtype);
}

/*
 * Forward of the same linear layer, the product `matmul_backward1`'s comment
 * recalls ("the forward pass was calculated with alpha = 1.0f, beta = 0.0f":
 * out = inp . weight^T, overwritten), with the optional bias of a GPT-2 linear
 * layer added. For r in [0, nrows): bt = rows ? rows[r] : r,
 *   out[r*OC + o] = bias[o] + sum_{i=0..C-1} inp[bt,i] * weight[o,i]
 * summed in double over i ascending; bias may be NULL (no bias term).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_forward_rows(double* out, const int64_t* rows, int64_t nrows, const void* inp,
                        const void* weight, const void* bias, int64_t BT, int64_t C, int64_t OC,
                        int dtype) {
    if (bad_args(BT, C, OC, dtype) || nrows < 0 || (!rows && nrows != BT)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= BT)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bt = rows ? rows[r] : r;
        for (int64_t o = 0; o < OC; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < C; ++i) {
#if ORACLE_MUTANT == 10 /* transposed operand: weight indexed by (i, o) on the square case */
                acc += load(inp, dtype, bt * C + i) * load(weight, dtype, (C == OC ? i * C + o : o * C + i));
#else
                acc += load(inp, dtype, bt * C + i) * load(weight, dtype, o * C + i);
#endif
            }
#if ORACLE_MUTANT == 9 /* dropped term: the bias is not added */
            (void)bias;
#else
            if (bias) acc += load(bias, dtype, o);
#endif
            out[r * OC + o] = acc;
        }
    }
    return 0;
}

/* Number of threads a parallel region of this compiled variant uses (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_mutant(void) { return ORACLE_MUTANT; }

/*
 * layernorm_backward.h -- C ABI of the GPT-2 LayerNorm backward in the same
 * library (libmmbwd.so) as the linear-layer backward.
 *
 * The operation is `layernorm_backward_cpu` of llm.c's
 * dev/cuda/layernorm_backward.cu: the gradient of the layer norm of each row
 * (`layernorm_forward_cpu`: out = (x - mean) * rstd * weight + bias, rstd =
 * 1/sqrt(var + 1e-5)) given the gradient `dout` of its output. With BT = B*T,
 * every tensor row-major and contiguous, and per row bt
 *
 *     n_i = (inp[bt,i] - mean[bt]) * rstd[bt]           the normalised input
 *     g_i = weight[i] * dout[bt,i]
 *     a   = (1/C) sum_i g_i,   c = (1/C) sum_i g_i n_i
 *     dinp[bt,i] += rstd[bt] * (g_i - a - n_i c)
 *     dweight[i] += sum over bt of n_i dout[bt,i]
 *     dbias[i]   += sum over bt of dout[bt,i]
 *
 * All three gradients accumulate, as in the CPU reference. In GPT-2 the
 * `dout` of a LayerNorm is the `dinp` that the linear layer after it (the
 * attention qkv or the MLP fc) produced with mmbwd_run.
 *
 * Element types: the MMBWD_F32 / MMBWD_BF16 codes of mmbwd.h, one type for
 * dinp, dweight, dbias, dout, inp and weight. mean and rstd are fp32 in both
 * cases: the row statistics the forward cached (the CPU reference's type).
 * Sums are formed in fp32; each output element is rounded once to its storage
 * type after its old value is added.
 *
 * Determinism: the sums over rows run in an order fixed by the device's SM
 * count and the problem size (per-block partial sums in fixed row order, then
 * a fixed-order reduction of the blocks), never by timing: repeated calls on
 * one device give bitwise identical results.
 */
#ifndef LAYERNORM_BACKWARD_H
#define LAYERNORM_BACKWARD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#include "mmbwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest C accepted. Rows up to 4096 (bf16) / 2048 (fp32) wide are staged
 * whole in shared memory by one fused kernel; wider rows take two passes over
 * global memory (the row sums, then column tiles), with the same result
 * contract. */
#define LNBWD_MAX_C_BF16 (1 << 20)
#define LNBWD_MAX_C_F32 (1 << 20)

/*
 * lnbwd_run -- enqueue the LayerNorm backward of B*T rows of width C on `stream`.
 *
 *   dinp     device, (B*T, C), read and written (+=)
 *   dweight  device, (C),      read and written (+=)
 *   dbias    device, (C),      read and written (+=)
 *   dout     device, (B*T, C), read only
 *   inp      device, (B*T, C), read only
 *   weight   device, (C),      read only
 *   mean     device, (B*T),    fp32, read only
 *   rstd     device, (B*T),    fp32, read only
 *   B, T, C  sizes, each >= 0; C <= LNBWD_MAX_C_BF16 (bf16) or LNBWD_MAX_C_F32 (fp32)
 *   dtype    MMBWD_F32 or MMBWD_BF16
 *   stream   the CUDA stream to enqueue on
 *
 * Argument order follows layernorm_backward_cpu (dinp, dweight, dbias, dout,
 * inp, weight, mean, rstd, B, T, C).
 *
 * Returns MMBWD_OK or a negative MMBWD_ERR_* code; on an error nothing is
 * enqueued. MMBWD_ERR_NULL: a pointer that a non-empty tensor needs is NULL.
 * MMBWD_ERR_SHAPE: a negative size, an overflowing product, or C above the
 * limit. MMBWD_ERR_ALIGN: a tensor pointer not 16-byte aligned, mean or rstd
 * not 4-byte aligned, or C times the element size not a multiple of 16 bytes.
 * MMBWD_ERR_ALIAS: an output overlaps an input or another output.
 * MMBWD_ERR_MEMORY: a non-empty tensor is not device memory of the current
 * device. MMBWD_ERR_ALLOC / MMBWD_ERR_CAPTURE: the shared workspace (per-block fp32
 * partial sums, lnbwd_workspace_bytes) could not grow, or would have to grow
 * during stream capture. B*T == 0 or C == 0 enqueue nothing (empty sums).
 *
 * Ownership and synchronisation as for mmbwd_run: the caller owns every buffer;
 * the call returns after enqueueing; the library's workspace is per device and
 * shared with mmbwd_run, so calls on one device must be ordered (one stream).
 * Every wait inside the kernels is bounded; one that gives up is reported as
 * MMBWD_ERR_DEVICE_TIMEOUT by mmbwd_device_status().
 */
int lnbwd_run(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
              const float* mean, const float* rstd, int64_t B, int64_t T, int64_t C, int dtype,
              cudaStream_t stream);

/* Workspace bytes lnbwd_run needs on the current device for this problem
 * (0 for invalid arguments or an empty problem). */
size_t lnbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* LAYERNORM_BACKWARD_H */

/*
 * encoder_backward.h -- C ABI of the GPT-2 encoder backward in the same library
 * (libmmbwd.so) as the linear-layer backward.
 *
 * The operation is the backward of the encoder of llm.c's llmc/encoder.cuh,
 * whose forward adds token row inp[b,t] of wte and position row t of wpe:
 *
 *     dwte[ix, c] += sum over (b, t) with inp[b, t] == ix of dout[b, t, c]
 *     dwpe[t, c]  += sum over b of dout[b, t, c]
 *
 * Deterministic: the positions of each token are gathered on the device (a
 * stable sort of (token, position) keys), summed in position order in chunks
 * of up to 32, and the chunks of a token added in order; dwpe is summed in
 * batch order. No atomics on the data: repeated calls give bitwise identical
 * results. Each output element is rounded
 * once (round-to-nearest-even for bf16; stochastically with encbwd_run_sr)
 * after its old value is added.
 *
 * Element types: MMBWD_F32 or MMBWD_BF16 (mmbwd.h) for dwte, dwpe and dout;
 * inp is int32.
 */
#ifndef ENCODER_BACKWARD_H
#define ENCODER_BACKWARD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#include "mmbwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Limits of the device sort (B*T positions, V token ids) and of the channel
 * count C. Up to 16384 positions are sorted by one cluster of eight CTAs; more by a
 * multi-block radix sort (a few more launches). */
#define ENCBWD_MAX_POSITIONS (1 << 24)
#define ENCBWD_MAX_VOCAB 131071
#define ENCBWD_MAX_CHANNELS 65536

/*
 * encbwd_run -- enqueue the encoder backward on `stream`.
 *
 *   dwte   device, (V, C), read and written (+=)
 *   dwpe   device, (T, C), read and written (+=)
 *   dout   device, (B*T, C), read only
 *   inp    device, (B*T) int32 token ids, read only
 *   B, T, C, V   sizes >= 0; B*T <= ENCBWD_MAX_POSITIONS, V <= ENCBWD_MAX_VOCAB,
 *                C <= ENCBWD_MAX_CHANNELS
 *   dtype  MMBWD_F32 or MMBWD_BF16
 *
 * Argument order follows the page's encoder_backward (dwte, dwpe, dout, inp,
 * B, T, C) with the vocabulary size added; no host copy of inp is needed.
 *
 * Returns MMBWD_OK or a negative MMBWD_ERR_* code (nothing enqueued on an
 * error): ERR_NULL, ERR_DTYPE, ERR_SHAPE (a size out of range), ERR_ALIGN
 * (dwte, dwpe, dout not 16-byte aligned or C times the element size not a
 * multiple of 16 bytes; inp not 4-byte aligned), ERR_ALIAS, ERR_MEMORY (a
 * non-empty tensor not in device memory of the current device), ERR_ALLOC /
 * ERR_CAPTURE (the shared workspace). A token id outside [0, V) is skipped by
 * the kernels and reported as MMBWD_ERR_SHAPE by mmbwd_device_status().
 * B*T == 0, C == 0 enqueue nothing.
 */
int encbwd_run(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
               int64_t V, int dtype, cudaStream_t stream);

/*
 * encbwd_run_sr -- encbwd_run with the bf16 outputs rounded stochastically, as
 * the page's wte and wpe kernels round theirs (a deterministic seed per
 * element). Everything else as encbwd_run; dtype must be MMBWD_BF16
 * (otherwise MMBWD_ERR_DTYPE, nothing enqueued).
 *
 * The rule is mmbwd_run_sr's (mmbwd.h): element e (row-major index) of dwte
 * (tensor 3) or dwpe (tensor 4) takes the 16-bit threshold r = bits
 * 16*(e mod 4) .. 16*(e mod 4)+15 of splitmix64 output number
 * (tensor << 58) | (e / 4) from `seed`, and the bf16 result is the high half
 * of (bits(old + sum) + r). The same seed repeats the same bits.
 */
int encbwd_run_sr(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                  int64_t V, int dtype, uint64_t seed, cudaStream_t stream);

/*
 * The same computation in two calls, so that the bucketing (which depends only
 * on the token ids, known at the start of a training step) can run early --
 * beside the forward pass, on another stream -- and leave the backward's
 * critical path:
 *
 * encbwd_plan_bytes -- bytes of a plan for this problem (0 for invalid
 *   arguments or an empty problem).
 *
 * encbwd_prepare -- enqueue the device sort of the token ids into `plan`.
 *   plan       device, caller-owned, >= encbwd_plan_bytes bytes, 256-byte aligned;
 *              written. A plan holds the sorted (token, position) keys, per-window
 *              run tables and counters, and records B*T, V and C.
 *   plan_bytes its size (MMBWD_ERR_SHAPE if too small)
 *   inp        device, (B*T) int32 token ids, read only; ids outside [0, V) are
 *              left out and reported by mmbwd_device_status()
 *   B, T, C, V, dtype   as encbwd_run (C and dtype fix the plan's counters and
 *              the alignment rule)
 *   Errors as encbwd_run (ERR_NULL, ERR_ALIGN, ERR_ALIAS, ERR_SHAPE, ERR_MEMORY, ...).
 *
 * encbwd_run_planned -- enqueue dwte += ..., dwpe += ... from a plan.
 *   dwte, dwpe, dout, B, T, C, V, dtype   as encbwd_run
 *   plan       a plan from encbwd_prepare for the same B*T, V and C, ordered
 *              before this call (same stream, or an event); read, and its
 *              counters are returned to zero, so one plan serves any number of
 *              runs (not at the same time). A plan of another problem is
 *              detected on the device: nothing is written and
 *              mmbwd_device_status() reports MMBWD_ERR_SHAPE (info[0] = -1).
 *   sr_seed    NULL: round to nearest; else bf16 outputs rounded stochastically
 *              with *sr_seed (as encbwd_run_sr; MMBWD_ERR_DTYPE for fp32)
 *   Results are bitwise those of encbwd_run / encbwd_run_sr. Uses the shared
 *   library workspace for its scratch (as encbwd_run). One launch.
 */
size_t encbwd_plan_bytes(int64_t B, int64_t T, int64_t C, int64_t V, int dtype);
int encbwd_prepare(void* plan, size_t plan_bytes, const int32_t* inp, int64_t B, int64_t T, int64_t C, int64_t V,
                   int dtype, cudaStream_t stream);
int encbwd_run_planned(void* dwte, void* dwpe, const void* dout, void* plan, int64_t B, int64_t T, int64_t C,
                       int64_t V, int dtype, const uint64_t* sr_seed, cudaStream_t stream);

/* Workspace bytes encbwd_run needs for this problem (0 for invalid arguments). */
size_t encbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int64_t V, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* ENCODER_BACKWARD_H */

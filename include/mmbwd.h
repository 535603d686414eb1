/*
 * mmbwd.h -- C ABI of the GB300 (sm_103a) linear-layer backward library.
 *
 * The operation is the backward pass of a GPT-2 linear layer, as computed by
 * `matmul_backward_cpu` and launched by `matmul_backward1` in llm.c's
 * dev/cuda/matmul_backward.cu. With BT = B*T and every tensor row-major and
 * contiguous,
 *
 *     dout (B,T,OC)   inp (B,T,C)   weight (OC,C)
 *     dinp    (B,T,C) += dout . weight          (the "backward into inp" loop;
 *                                                 cuBLAS beta = 1 there: "gradients add")
 *     dweight (OC,C)  += dout^T . inp           (the "backward into weight" loop,
 *                                                 contracting over BT)
 *     dbias   (OC)     = sum over (b,t) of dout (the bias sum: `dbias[o] = sum`,
 *                                                 an overwrite, skipped when dbias is NULL)
 *
 * Element types (one type for all six tensors, like the pages' floatX switch):
 *   MMBWD_BF16: bf16 storage, products accumulated in fp32, each output element
 *               rounded once to bf16 (round-to-nearest-even) after the old value
 *               (converted to fp32) and the fp32 sum are added.
 *   MMBWD_F32:  fp32 storage and fp32-accurate products. Shapes whose two
 *               reduction lengths (OC and B*T) are at most 8192 run on the
 *               tensor
 *               cores: the kernel splits each staged operand, in shared memory,
 *               into its tf32 value and the exact fp32 remainder (no copy in
 *               device memory, no workspace), and each product is formed from three tf32
 *               products, hi.hi in one fp32 accumulator and hi.lo + lo.hi in a
 *               second, added once at the end. The tensor core rounds each
 *               accumulation toward zero, so this path's error grows with the
 *               reduction length (hence the 8192 limit). Other shapes use fp32
 *               fused multiply-adds on the CUDA cores. MMBWD_F32_PATH = "ffma" or
 *               "x3" in the environment forces one where the shape allows it.
 *
 * Every entry point is plain C: device pointers, sizes, a CUDA stream.
 * Nothing here takes or returns a framework type.
 */
#ifndef MMBWD_H
#define MMBWD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
#define MMBWD_F32 0
#define MMBWD_BF16 1

/* Status codes. MMBWD_OK is 0; every error is negative. */
#define MMBWD_OK 0
#define MMBWD_ERR_NULL (-1)           /* a required pointer is NULL */
#define MMBWD_ERR_DTYPE (-2)          /* dtype is neither MMBWD_F32 nor MMBWD_BF16 */
#define MMBWD_ERR_SHAPE (-3)          /* a size is negative, or a product overflows */
#define MMBWD_ERR_ALIGN (-4)          /* a pointer is not 16-byte aligned, or C or OC
                                         times the element size is not a multiple of 16 */
#define MMBWD_ERR_ALIAS (-5)          /* an output overlaps an input or another output */
#define MMBWD_ERR_ALLOC (-6)          /* the library could not allocate its workspace */
#define MMBWD_ERR_CUDA (-7)           /* a CUDA runtime call or a launch failed */
#define MMBWD_ERR_DEVICE_TIMEOUT (-8) /* a kernel gave up a bounded wait (device status) */
#define MMBWD_ERR_ARCH (-9)           /* the current device is not sm_103 */
#define MMBWD_ERR_CAPTURE (-10)       /* the workspace would have to grow while the
                                         stream is being captured into a CUDA graph */
#define MMBWD_ERR_MEMORY (-12)        /* a non-empty tensor does not lie in device memory
                                         of the current device (host memory, pinned or
                                         mapped host memory, managed memory, or memory
                                         of another GPU) */

/*
 * mmbwd_run -- enqueue the whole backward pass of one linear layer on `stream`.
 *
 *   dinp           device, (B*T, C), read and written (+=)
 *   dweight        device, (OC, C),  read and written (+=)
 *   dbias_or_null  device, (OC),     written (=); NULL skips the bias sum and
 *                  nothing else changes
 *   dout           device, (B*T, OC), read only
 *   inp            device, (B*T, C),  read only
 *   weight         device, (OC, C),   read only
 *   B, T, C, OC    sizes, each >= 0
 *   dtype          MMBWD_F32 or MMBWD_BF16 (the type of all six tensors)
 *   stream         the CUDA stream to enqueue on (0 = legacy default stream)
 *
 * Argument order follows matmul_backward_cpu (dinp, dweight, dbias, dout, inp,
 * weight, B, T, C, OC); the all-ones vector that matmul_backward1 takes is not
 * needed. Layout: row-major, contiguous, no strides.
 *
 * Ownership: the caller owns every buffer; the library never frees them.
 * Every non-empty tensor must be device memory of the current device: its
 * first and last bytes are checked with cudaPointerGetAttributes, and host,
 * managed or another GPU's memory gives MMBWD_ERR_MEMORY with nothing
 * enqueued. Outputs must not overlap inputs or each other (MMBWD_ERR_ALIAS);
 * inputs may overlap each other. Pointers must be 16-byte aligned, and C and
 * OC times the element size must be multiples of 16 bytes (MMBWD_ERR_ALIGN).
 * A pointer may be NULL only when its tensor has no elements.
 *
 * Workspace: the bf16 path may need a library-owned fp32 workspace for its
 * split reduction (mmbwd_workspace_bytes); fp32 needs none. It is allocated per device on
 * first need and reused; growing it synchronises the device, so the first
 * call of a new, larger shape should not be made during stream capture
 * (MMBWD_ERR_CAPTURE). Calls that share a device share this workspace:
 * calls on different streams of one device must not overlap in time.
 *
 * Synchronisation: asynchronous. The call validates, enqueues and returns; the
 * caller synchronises the stream before reading results. Invalid arguments
 * enqueue nothing and return a negative code. A kernel that gives up a bounded
 * wait records MMBWD_ERR_DEVICE_TIMEOUT in the device status word, read by
 * mmbwd_device_status(); nothing in the library calls exit() or traps.
 *
 * Degenerate sizes: B*T == 0 sets dbias to 0 (the empty sum) and leaves dinp
 * and dweight untouched; OC == 0 changes nothing; C == 0 still computes dbias.
 *
 * Determinism: for a given shape the work split is a pure function of the
 * shape, every reduction runs in a fixed order and no float atomics are used,
 * so repeated calls on identical inputs give bitwise identical results.
 */
int mmbwd_run(void* dinp, void* dweight, void* dbias_or_null, const void* dout, const void* inp,
              const void* weight, int64_t B, int64_t T, int64_t C, int64_t OC, int dtype,
              cudaStream_t stream);

/*
 * mmbwd_run_sr -- mmbwd_run with stochastic rounding of the bf16 outputs.
 *
 * The encoder page's kernels round their fp32 sums to bf16 stochastically,
 * with a deterministic per-element seed (wte_backward_kernel and
 * wpe_backward_kernel); this is that option for the linear layer's outputs.
 * Arguments, layout, ownership, workspace, errors and degenerate sizes are
 * those of mmbwd_run; dtype must be MMBWD_BF16 (anything else:
 * MMBWD_ERR_DTYPE, nothing enqueued).
 *
 * Each output value v = old + sum (fp32; dbias: the sum) is rounded to bf16
 * as follows. Element e (row-major index) of output tensor k (0 dinp,
 * 1 dweight, 2 dbias; the encoder's dwte and dwpe are 3 and 4) takes the
 * 16-bit threshold r = bits 16*(e mod 4) ..
 * 16*(e mod 4)+15 of output number n = (k << 58) | (e / 4) of the splitmix64
 * generator seeded with `seed` (z = seed + (n+1)*0x9E3779B97F4A7C15;
 * z = (z ^ z>>30)*0xBF58476D1CE4E5B9; z = (z ^ z>>27)*0x94D049BB133111EB;
 * z ^ z>>31); the result is the high 16 bits of (bits(v) + r), so the
 * magnitude rounds up with probability (low 16 bits of v) / 65536 and the
 * rounding is unbiased. Infinities and NaNs are truncated (NaNs stay NaN).
 * The same seed and inputs give bitwise identical results; a new seed per
 * step gives fresh rounding noise.
 */
int mmbwd_run_sr(void* dinp, void* dweight, void* dbias_or_null, const void* dout, const void* inp,
                 const void* weight, int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, uint64_t seed,
                 cudaStream_t stream);

/* Bytes of workspace mmbwd_run needs for this shape on the current device
 * (0 when it needs none, and for invalid arguments). The work split depends
 * on the device's SM count, which this queries (152, a full GB300, when no
 * usable device is present). Enqueues nothing. */
size_t mmbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype);

/* Free the current device's workspace (synchronises the device). Returns a status. */
int mmbwd_release(void);

/* Static description of a status code. Never NULL. */
const char* mmbwd_strerror(int code);

/* Read the current device's status word, written by kernels that gave up a
 * bounded wait: MMBWD_OK or MMBWD_ERR_DEVICE_TIMEOUT. Synchronises the device.
 * reset != 0 clears the word after reading. `info` (may be NULL) receives 3
 * integers: the block, the wait site and the work item of the first failure. */
int mmbwd_device_status(int reset, int* info);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int mmbwd_version(void);

/* Describe the work split mmbwd_run would use (a pure function of the shape
 * and the number of co-resident CTAs; num_sms <= 0 takes the current device's
 * value, or 152 without a usable device). out[0..n) receives, in order: path (0 = fp32 SIMT,
 * 1 = bf16 tensor-core, 2 = fp32 from three tf32 products), grid size (CTAs), work items, dweight splits, k-blocks
 * per split, dinp tiles, dweight tiles, schedule kind (1 = per-pair tables),
 * tile M (rows per CTA pair), tile N of dinp, tile N of dweight, tile K,
 * pipeline stages, kernel launches per call, CTA pairs per cluster (always 1:
 * a cluster is one CTA pair). num_sms stands for the resident CTAs. Returns
 * the number of values written (at most 15), or a negative status. */
int mmbwd_plan_info(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, int num_sms,
                    int* out, int n);

/* Self-test of the bounded-wait machinery: launches one tiny kernel whose
 * thread waits on a barrier that nothing completes, giving up after
 * `timeout_ns`. Synchronises, reads and clears the status word, and returns
 * what the kernel recorded (MMBWD_ERR_DEVICE_TIMEOUT when the mechanism works). */
int mmbwd_selftest_wait_timeout(uint64_t timeout_ns);

/*
 * mmbwd_forward -- the forward of the same linear layer, enqueued on `stream`:
 *
 *     out (B,T,OC) = inp (B,T,C) . weight^T + bias          (overwritten)
 *
 * the product that matmul_backward1's comment recalls ("the forward pass was
 * calculated with alpha = 1.0f, beta = 0.0f": cuBLAS SGEMM of weight^T and
 * inp into out), plus the optional bias of a GPT-2 linear layer.
 *
 *   out            device, (B*T, OC), written
 *   inp            device, (B*T, C),  read only
 *   weight         device, (OC, C),   read only
 *   bias_or_null   device, (OC),      read only; NULL: no bias term
 *   dtype          MMBWD_F32 or MMBWD_BF16 (all four tensors)
 *
 * bf16: fp32 accumulation on the tensor cores, out rounded once (RNE) after
 * adding the bias in fp32. fp32: as for mmbwd_run, three tf32 products on the
 * tensor cores where C is at most 8192 (out is set to the
 * bias, then the product is added), FFMA otherwise. Same alignment, aliasing (out
 * must not overlap an input), status codes, asynchrony and determinism as
 * mmbwd_run; no workspace. C == 0 gives out = bias (or 0).
 */
int mmbwd_forward(void* out, const void* inp, const void* weight, const void* bias_or_null, int64_t B,
                  int64_t T, int64_t C, int64_t OC, int dtype, cudaStream_t stream);

/* The path mmbwd_forward takes for this shape and type (0 = fp32 FMA kernel,
 * 1 = bf16 tensor cores, 2 = fp32 from three tf32 products), or a negative
 * status for invalid arguments. Reads MMBWD_F32_PATH like the call itself. */
int mmbwd_forward_path(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype);

/* Test hook: make the next `n` workspace allocations fail (MMBWD_ERR_ALLOC). */
void mmbwd_debug_fail_next_alloc(int n);

/* Test hook: the next `n` launch steps of any entry point fail as the CUDA
 * runtime does when it refuses a launch, before anything is enqueued; the
 * entry point returns MMBWD_ERR_CUDA and the outputs are untouched. */
void mmbwd_debug_fail_next_launch(int n);

/* Size of the library's fixed scratch buffer used by mmbwd_run_static_scratch. */
#define MMBWD_STATIC_SCRATCH_BYTES (32u << 20)
#define MMBWD_ERR_SCRATCH (-11) /* the problem needs more scratch than that buffer holds */

/*
 * mmbwd_run_static_scratch -- the operation of mmbwd_run, with its arguments,
 * layout and errors, for callers that must not allocate device memory.
 * The paper has no counterpart: this entry point exists only for such callers.
 *
 * Who needs it: code that runs where device allocation is unavailable or not
 * allowed -- inside a custom allocator or memory-pool callback (allocating
 * there re-enters the allocator), under a hard device-memory budget that was
 * fixed up front, or in a runtime that forbids cudaMalloc after start-up
 * because it synchronises the device. mmbwd_run may grow a workspace with
 * cudaMalloc; this entry point never calls cudaMalloc, cudaFree or any other
 * allocating routine.
 *
 * bf16: the plan, the kernels and so the results are those of mmbwd_run; the
 * split reduction uses one fixed buffer of MMBWD_STATIC_SCRATCH_BYTES compiled
 * into the library (a file-scope device array, so every GPU that loads the
 * library holds it until the process exits) instead of the grown workspace.
 * A problem whose work split needs more than that returns MMBWD_ERR_SCRATCH
 * and enqueues nothing; for bf16, mmbwd_workspace_bytes() gives the need in
 * advance. Nothing in the buffer has to start at zero: every value a call
 * reads there is written earlier by the same call.
 *
 * fp32: the path mmbwd_run takes (three tf32 products on the tensor cores
 * where the shape allows, the fused-multiply-add kernel otherwise), so the results are
 * those of mmbwd_run; neither path uses any scratch.
 *
 * All calls on a device share the one buffer, which keeps whatever the last
 * call left in it: calls that overlap on the GPU (for example on two streams
 * with nothing ordering them) race on it and give wrong results.
 *
 * The first call on each device looks up the buffer's device address (with
 * that device current); make that first call before any stream capture.
 */
int mmbwd_run_static_scratch(void* dinp, void* dweight, void* dbias_or_null, const void* dout,
                             const void* inp, const void* weight, int64_t B, int64_t T, int64_t C,
                             int64_t OC, int dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MMBWD_H */

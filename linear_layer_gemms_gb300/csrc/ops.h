// Internal declarations of the kernels other than the tensor-core kernel (the
// fp32 FFMA path, the fp32 tensor-core path's passes, the encoder and
// LayerNorm backwards), shared with the C-ABI layer. Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mmbwd {

// Test hook (mmbwd_debug_fail_next_launch): true for the next n calls, set by
// the test; every launch function checks it before it enqueues anything and
// then fails as the runtime does when it refuses a launch, so the error path
// of each entry point can be exercised without a GPU fault.
bool take_injected_launch_failure();

// ------------------------------------------------------------ fp32 SIMT path
constexpr int SIMT_BM = 128;
constexpr int SIMT_BN = 128;
constexpr int SIMT_BK = 8;
constexpr int SIMT_THREADS = 256;

cudaError_t simt_launch(float* dinp, float* dweight, float* dbias, const float* dout,
                        const float* inp, const float* weight, int64_t BT, int64_t C, int64_t OC,
                        cudaStream_t stream);

// out (BT x OC) = inp (BT x C) . weight^T + bias (bias may be null), fp32 FFMA.
cudaError_t simt_forward_launch(float* out, const float* inp, const float* weight, const float* bias,
                                int64_t BT, int64_t C, int64_t OC, cudaStream_t stream);

// out[r, o] = bias[o], or 0 without a bias (the forward when C == 0).
cudaError_t fill_rows_launch(void* out, const void* bias, int64_t rows, int64_t cols, int dtype,
                             cudaStream_t stream);

// dbias = column sums of dout (used when C == 0, where no GEMM tile exists).
cudaError_t colsum_launch(void* dbias, const void* dout, int64_t BT, int64_t OC, int dtype, bool sr, uint64_t sr_seed,
                          cudaStream_t stream);

// ---------------------------------------------------------------- fp32 on the tensor cores (3xTF32)

// (no workspace: the kernel splits the raw fp32 operands in shared memory)
bool x3_shape_ok(int64_t BT, int64_t C, int64_t OC);
cudaError_t x3_launch(float* dinp, float* dweight, float* dbias, const float* dout, const float* inp,
                      const float* weight, int64_t BT, int64_t C, int64_t OC, int num_sms, cudaStream_t stream);
bool x3_forward_shape_ok(int64_t BT, int64_t C, int64_t OC);
cudaError_t x3_forward_launch(float* out, const float* inp, const float* weight, const float* bias, int64_t BT,
                              int64_t C, int64_t OC, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- encoder backward

size_t enc_workspace_bytes(int64_t BT, int64_t C);
size_t enc_plan_bytes(int64_t BT, int64_t C);           // the tables encbwd_prepare writes
size_t enc_run_workspace_bytes(int64_t BT, int64_t C);  // scratch of a planned run
cudaError_t enc_prepare_launch(void* plan, const int32_t* inp, int64_t B, int64_t T, int64_t C, int64_t V,
                               cudaStream_t stream);
cudaError_t enc_run_planned_launch(void* dwte, void* dwpe, const void* dout, void* plan, int64_t B, int64_t T,
                                   int64_t C, int64_t V, int dtype, void* ws, int num_sms, cudaStream_t stream,
                                   bool sr, uint64_t seed);
cudaError_t enc_launch(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                       int64_t V, int dtype, void* ws, int num_sms, cudaStream_t stream, bool sr = false,
                       uint64_t seed = 0);
cudaError_t enc_read_status(int* code, int* info3, bool reset);

// ---------------------------------------------------------------- LayerNorm backward

struct LnPlan {
    int wide = 0;            // 1: rows too wide for the fused kernel (row sums, then column tiles)
    int vpl = 0;             // 16-byte column vectors per thread and row
    int team_warps = 0;      // warps that share one row
    int warps = 0;           // warps per block
    int grid = 0;            // blocks (one per SM), each a contiguous range of rows
    int64_t rows_per_block = 0;
    size_t off_ring = 0;     // start of the teams' row buffers in shared memory
    size_t smem = 0;         // weight (fp32) + row-sum exchange + barriers + row buffers
    size_t ws_bytes = 0;     // per-block partial sums, fp32 [grid][2][C] (+ the row sums when wide)
    int col_tiles = 0;       // wide: column tiles of 256 vectors
};

int ln_vec_elems(int dtype);
cudaError_t ln_make_plan(int64_t BT, int C, int dtype, int num_sms, LnPlan* plan);
cudaError_t ln_launch(const LnPlan& plan, void* dinp, void* dweight, void* dbias, const void* dout,
                      const void* inp, const void* weight, const float* mean, const float* rstd, int64_t BT,
                      int C, int dtype, void* ws, cudaStream_t stream);
cudaError_t ln_read_status(int* code, int* info3, bool reset);

}  // namespace mmbwd

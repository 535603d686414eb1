// fp32 linear-layer backward and forward on the CUDA cores (FFMA), and the
// stand-alone column sum used when C == 0.
//
// fp32 storage needs fp32-accurate products: the page's harness turns TF32
// off ("use fp32 to get accurate results for checking w.r.t. CPU", llm.c
// dev/cuda/matmul_backward.cu, main) because one TF32 rounding per operand
// would miss an fp32 tolerance. These kernels accumulate with fp32 fused
// multiply-adds.
//
// Two launches, both classic 128 x 128 register-tiled GEMMs (256 threads,
// 8 x 8 outputs per thread, K-tiles of 8 double-buffered through shared memory):
//   dinp    (BT x C) += dout (BT x OC) . weight (OC x C)          A row-major (M x K)
//   dweight (OC x C) += dout^T . inp, dout stored (BT x OC) = (K x M)
// and the bias: in the dweight launch, the CTAs of the first column tile sum
// the dout tile they stage in shared memory over its K (= BT) rows, in K order,
// and overwrite dbias. No split of K, so each output has one writer.
#include "../../include/mmbwd.h"
#include "ops.h"
#include "sr.cuh"

#include <algorithm>

namespace mmbwd {
namespace {

constexpr int BM = SIMT_BM, BN = SIMT_BN, BK = SIMT_BK;
constexpr int PAD = 4;  // keeps 16-byte alignment of smem rows

// D (M x N, row-major) += A . B, with A either (M x K) row-major (A_KM = false)
// or stored as (K x M) row-major (A_KM = true); B is (K x N) row-major, or
// stored as (N x K) row-major (B_NK = true). With OVERWRITE, D = A . B + bias
// (bias per column, may be null) instead of the accumulation.
template <bool A_KM, bool B_NK = false, bool OVERWRITE = false>
__global__ void __launch_bounds__(SIMT_THREADS, 2)
    simt_gemm_acc(float* __restrict__ D, const float* __restrict__ A, const float* __restrict__ Bm,
                  int64_t M, int64_t N, int64_t K, float* __restrict__ dbias,
                  const float* __restrict__ col_bias = nullptr) {
    __shared__ __align__(16) float As[2][BK][BM + PAD];
    __shared__ __align__(16) float Bs[2][BK][BN + PAD];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * BN;
    const bool do_bias = A_KM && dbias != nullptr && blockIdx.y == 0;

    // Global -> register staging of one K-tile (one float4 of A, one of B per thread).
    // A row-major (M x K): thread covers row tid/2, k-offset (tid%2)*4.
    // A stored (K x M):    thread covers k = tid/32, m-offset (tid%32)*4.
    // B (K x N):           thread covers k = tid/32, n-offset (tid%32)*4.
    float4 ra, rb;
    auto load_tile = [&](int64_t k0) {
        if (!A_KM) {
            const int64_t m = m0 + tid / 2;
            const int64_t k = k0 + (tid % 2) * 4;
            ra = (m < M && k < K) ? *reinterpret_cast<const float4*>(A + m * K + k)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int64_t k = k0 + tid / 32;
            const int64_t m = m0 + (tid % 32) * 4;
            ra = (k < K && m < M) ? *reinterpret_cast<const float4*>(A + k * M + m)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!B_NK) {
            const int64_t k = k0 + tid / 32;
            const int64_t n = n0 + (tid % 32) * 4;
            rb = (k < K && n < N) ? *reinterpret_cast<const float4*>(Bm + k * N + n)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int64_t n = n0 + tid / 2;
            const int64_t k = k0 + (tid % 2) * 4;
            rb = (n < N && k < K) ? *reinterpret_cast<const float4*>(Bm + n * K + k)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto store_tile = [&](int buf) {
        if (!A_KM) {
            const int m = tid / 2, k = (tid % 2) * 4;
            As[buf][k + 0][m] = ra.x;
            As[buf][k + 1][m] = ra.y;
            As[buf][k + 2][m] = ra.z;
            As[buf][k + 3][m] = ra.w;
        } else {
            *reinterpret_cast<float4*>(&As[buf][tid / 32][(tid % 32) * 4]) = ra;
        }
        if (!B_NK) {
            *reinterpret_cast<float4*>(&Bs[buf][tid / 32][(tid % 32) * 4]) = rb;
        } else {
            const int n = tid / 2, k = (tid % 2) * 4;
            Bs[buf][k + 0][n] = rb.x;
            Bs[buf][k + 1][n] = rb.y;
            Bs[buf][k + 2][n] = rb.z;
            Bs[buf][k + 3][n] = rb.w;
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float bsum = 0.f;

    const int64_t nkt = (K + BK - 1) / BK;
    if (nkt > 0) {
        load_tile(0);
        store_tile(0);
    }
    __syncthreads();
    for (int64_t kt = 0; kt < nkt; ++kt) {
        const int buf = static_cast<int>(kt & 1);
        if (kt + 1 < nkt) load_tile((kt + 1) * BK);
        if (do_bias && tid < BM) {
#pragma unroll
            for (int k = 0; k < BK; ++k) bsum += As[buf][k][tid];
        }
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4 + 64]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kt + 1 < nkt) store_tile(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (m >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + tx * 4 + h * 64;
            if (n >= N) continue;  // N is a multiple of 4: a float4 is all in or all out
            float4* p = reinterpret_cast<float4*>(D + m * N + n);
            float4 o;
            if (OVERWRITE) {
                o = col_bias ? *reinterpret_cast<const float4*>(col_bias + n) : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                o = *p;
            }
            o.x += acc[i][h * 4 + 0];
            o.y += acc[i][h * 4 + 1];
            o.z += acc[i][h * 4 + 2];
            o.w += acc[i][h * 4 + 3];
            *p = o;
        }
    }
    if (do_bias && tid < BM && m0 + tid < M) dbias[m0 + tid] = bsum;
}

// dbias[o] = sum over rows of dout[row, o], one thread per column, rows in order.
template <typename T>
__global__ void colsum_kernel(T* __restrict__ dbias, const T* __restrict__ dout, int64_t BT, int64_t OC, int sr,
                              uint64_t sr_seed) {
    const int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (o >= OC) return;
    float s = 0.f;
    for (int64_t r = 0; r < BT; ++r) s += static_cast<float>(dout[r * OC + o]);
    if constexpr (sizeof(T) == 2) {
        if (sr) {
            dbias[o] = sr::round(s, sr_seed, sr::DBIAS, static_cast<uint64_t>(o));
            return;
        }
    }
    dbias[o] = static_cast<T>(s);
}

}  // namespace

cudaError_t simt_launch(float* dinp, float* dweight, float* dbias, const float* dout, const float* inp,
                        const float* weight, int64_t BT, int64_t C, int64_t OC, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    // dinp: M = BT, N = C, K = OC
    {
        dim3 grid(static_cast<unsigned>((BT + BM - 1) / BM), static_cast<unsigned>((C + BN - 1) / BN));
        if (grid.x && grid.y) simt_gemm_acc<false><<<grid, SIMT_THREADS, 0, stream>>>(dinp, dout, weight, BT, C, OC, nullptr);
    }
    // dweight: M = OC, N = C, K = BT (+ bias on the first column tile)
    {
        dim3 grid(static_cast<unsigned>((OC + BM - 1) / BM), static_cast<unsigned>((C + BN - 1) / BN));
        if (grid.x && grid.y) simt_gemm_acc<true><<<grid, SIMT_THREADS, 0, stream>>>(dweight, dout, inp, OC, C, BT, dbias);
    }
    return cudaGetLastError();
}

cudaError_t simt_forward_launch(float* out, const float* inp, const float* weight, const float* bias,
                                int64_t BT, int64_t C, int64_t OC, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    // out: M = BT, N = OC, K = C; A = inp (BT x C), B = weight stored (OC x C)
    dim3 grid(static_cast<unsigned>((BT + BM - 1) / BM), static_cast<unsigned>((OC + BN - 1) / BN));
    if (grid.x && grid.y)
        simt_gemm_acc<false, true, true><<<grid, SIMT_THREADS, 0, stream>>>(out, inp, weight, BT, OC, C, nullptr, bias);
    return cudaGetLastError();
}

// out[r, o] = bias[o] (or 0 without a bias): the forward when C == 0.
template <typename T>
__global__ void fill_rows_kernel(T* __restrict__ out, const T* __restrict__ bias, int64_t rows, int64_t cols) {
    const int64_t n = rows * cols;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = bias ? bias[i % cols] : static_cast<T>(0.f);
}

cudaError_t fill_rows_launch(void* out, const void* bias, int64_t rows, int64_t cols, int dtype,
                             cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const int64_t n = rows * cols;
    if (n == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 4096));
    if (dtype == MMBWD_F32)
        fill_rows_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<float*>(out), static_cast<const float*>(bias),
                                                            rows, cols);
    else
        fill_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(bias), rows, cols);
    return cudaGetLastError();
}

cudaError_t colsum_launch(void* dbias, const void* dout, int64_t BT, int64_t OC, int dtype, bool sr, uint64_t sr_seed,
                          cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const unsigned blocks = static_cast<unsigned>((OC + 255) / 256);
    if (blocks == 0) return cudaSuccess;
    if (dtype == MMBWD_F32)
        colsum_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<float*>(dbias), static_cast<const float*>(dout), BT, OC,
                                                         0, 0);
    else
        colsum_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(dbias),
                                                                 static_cast<const __nv_bfloat16*>(dout), BT, OC,
                                                                 sr ? 1 : 0, sr_seed);
    return cudaGetLastError();
}

}  // namespace mmbwd

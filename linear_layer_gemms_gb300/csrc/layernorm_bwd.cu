// LayerNorm backward (llm.c dev/cuda/layernorm_backward.cu, layernorm_backward_cpu):
// per row, two row means of g = weight * dout, then dinp += rstd (g - a - n c);
// dweight and dbias are sums over all rows of n * dout and dout.
//
// The work is bound by HBM: each row's dout and inp are read once and its dinp
// read and written once (4 row-lengths of traffic per row); the weight row and
// the parameter-gradient partial sums stay on chip.
//
// Rows kernel: persistent blocks of W warps, each block a contiguous range of
// rows, each warp one row at a time. A lane owns the 16-byte column vectors
// lane, lane + 32, ... of every row, so it keeps its share of dout and inp in
// registers across the two passes (one HBM read per element). The two row
// sums are reduced with an xor butterfly, which leaves the same bits in every
// lane. Each warp adds n*dout and dout of its rows into its own fp32 rows in
// shared memory (no two lanes touch the same column, no atomics); at the end
// the block sums its warps in warp order and writes one fp32 partial row pair
// to the workspace.
//
// Params kernel: for each group of 32 columns, 32 warps each sum a fixed
// contiguous range of the block partials in block order, then one warp adds
// the 32 warp sums in warp order, adds the old dweight / dbias and rounds once.
//
// Both kernels are launched with programmatic stream serialization: their
// set-up may overlap the previous kernel on the stream, and they touch global
// memory only after `griddepcontrol.wait`.
#include "../../include/layernorm_backward.h"
#include "../../include/mmbwd.h"
#include "internal.h"

namespace mmbwd {
namespace {

constexpr int LN_MAX_WARPS = 8;
constexpr size_t LN_SMEM_LIMIT = 227 * 1024;
constexpr int LN_PARAM_WARPS = 32;

__device__ __forceinline__ void ln_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void ln_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T>
struct LnElem;
template <>
struct LnElem<float> {
    static constexpr int N = 4;  // elements per 16-byte vector
    __device__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static float load1(const void* p, int i) { return static_cast<const float*>(p)[i]; }
    __device__ static void store1(void* p, int i, float v) { static_cast<float*>(p)[i] = v; }
};
template <>
struct LnElem<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    __device__ static void unpack(const uint4& v, float (&f)[8]) {
        f[0] = lo(v.x), f[1] = hi(v.x), f[2] = lo(v.y), f[3] = hi(v.y);
        f[4] = lo(v.z), f[5] = hi(v.z), f[6] = lo(v.w), f[7] = hi(v.w);
    }
    __device__ static uint32_t pack2(float a, float b) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // RNE, .x = a (low half)
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
    }
    __device__ static float load1(const void* p, int i) {
        return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    }
    __device__ static void store1(void* p, int i, float v) {
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
};

struct LnParams {
    void* dinp;
    const void* dout;
    const void* inp;
    const void* weight;
    const float* mean;
    const float* rstd;
    float* partials;  // [grid][2][C]: n*dout sums, then dout sums
    int64_t BT;
    int64_t rows_per_block;
    int C;
    int nvec;  // C / N
};

template <typename T, int VPL>
__global__ void __launch_bounds__(LN_MAX_WARPS * 32) ln_bwd_rows_kernel(const LnParams p) {
    using E = LnElem<T>;
    constexpr int N = E::N;
    extern __shared__ __align__(16) float ln_smem[];
    const int C = p.C;
    const int W = static_cast<int>(blockDim.x >> 5);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    float* w_s = ln_smem;                      // weight as fp32, C
    float* part = ln_smem + C + warp * 2 * C;  // this warp's [dweight | dbias] sums, 2C

    for (int i = lane * 4; i < 2 * C; i += 32 * 4)
        *reinterpret_cast<float4*>(part + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    ln_grid_wait();  // global memory only from here on
    for (int i = threadIdx.x; i < C; i += blockDim.x) w_s[i] = E::load1(p.weight, i);
    __syncthreads();

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_block;
    const int64_t r1 = r0 + p.rows_per_block < p.BT ? r0 + p.rows_per_block : p.BT;
    for (int64_t r = r0 + warp; r < r1; r += W) {
        const uint4* drow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + r * C);
        const uint4* xrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.inp) + r * C);
        uint4* orow = reinterpret_cast<uint4*>(static_cast<T*>(p.dinp) + r * C);
        uint4 vd[VPL], vx[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            if (v < p.nvec) {
                vd[j] = __ldcs(drow + v);  // read once: stream past the caches
                vx[j] = __ldcs(xrow + v);
            }
        }
        const float m = __ldg(p.mean + r), s = __ldg(p.rstd + r);

        // first pass: the two row sums
        float sa = 0.f, sc = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            if (v < p.nvec) {
                float d[N], x[N];
                E::unpack(vd[j], d);
                E::unpack(vx[j], x);
#pragma unroll
                for (int e = 0; e < N; ++e) {
                    const float n = (x[e] - m) * s;
                    const float g = w_s[v * N + e] * d[e];
                    sa += g;
                    sc += g * n;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, off);
            sc += __shfl_xor_sync(0xffffffffu, sc, off);
        }
        const float a = sa / static_cast<float>(C), c = sc / static_cast<float>(C);

        // second pass: dinp, and this warp's parameter-gradient sums
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            if (v < p.nvec) {
                float d[N], x[N], o[N];
                E::unpack(vd[j], d);
                E::unpack(vx[j], x);
                E::unpack(__ldcg(orow + v), o);
                float* pw = part + v * N;
                float* pb = part + C + v * N;
#pragma unroll
                for (int q = 0; q < N; q += 4) {
                    float4 w4 = *reinterpret_cast<float4*>(pw + q);
                    float4 b4 = *reinterpret_cast<float4*>(pb + q);
                    float nn[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        nn[e] = (x[q + e] - m) * s;
                        const float g = w_s[v * N + q + e] * d[q + e];
                        o[q + e] += (g - a - nn[e] * c) * s;
                    }
                    w4.x += nn[0] * d[q + 0], w4.y += nn[1] * d[q + 1];
                    w4.z += nn[2] * d[q + 2], w4.w += nn[3] * d[q + 3];
                    b4.x += d[q + 0], b4.y += d[q + 1], b4.z += d[q + 2], b4.w += d[q + 3];
                    *reinterpret_cast<float4*>(pw + q) = w4;
                    *reinterpret_cast<float4*>(pb + q) = b4;
                }
                __stcg(orow + v, E::pack(o));
            }
        }
    }
    __syncthreads();
    ln_launch_dependents();

    // the block's partial: its warps' sums in warp order
    const float* all = ln_smem + C;
    float* dst = p.partials + static_cast<size_t>(blockIdx.x) * 2 * C;
    for (int i = threadIdx.x * 4; i < 2 * C; i += blockDim.x * 4) {
        float4 acc = *reinterpret_cast<const float4*>(all + i);
        for (int w = 1; w < W; ++w) {
            const float4 t = *reinterpret_cast<const float4*>(all + static_cast<size_t>(w) * 2 * C + i);
            acc.x += t.x, acc.y += t.y, acc.z += t.z, acc.w += t.w;
        }
        __stcg(reinterpret_cast<float4*>(dst + i), acc);
    }
}

// 32 warps: 32 columns of [dweight | dbias] per block; warp w sums blocks
// [w*per, (w+1)*per) in order, then warp 0 adds the 32 warp sums in warp order.
template <typename T>
__global__ void __launch_bounds__(LN_PARAM_WARPS * 32)
    ln_bwd_params_kernel(void* dweight, void* dbias, const float* partials, int grid, int C) {
    using E = LnElem<T>;
    __shared__ float red[LN_PARAM_WARPS][32];
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int i = static_cast<int>(blockIdx.x) * 32 + lane;  // index into [0, 2C)
    const int per = (grid + LN_PARAM_WARPS - 1) / LN_PARAM_WARPS;
    const int g0 = warp * per, g1 = g0 + per < grid ? g0 + per : grid;
    ln_grid_wait();  // the partials of the rows kernel
    float acc = 0.f;
    if (i < 2 * C) {
#pragma unroll 8
        for (int g = g0; g < g1; ++g) acc += __ldcg(partials + static_cast<size_t>(g) * 2 * C + i);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && i < 2 * C) {
        float sum = red[0][lane];
        for (int w = 1; w < LN_PARAM_WARPS; ++w) sum += red[w][lane];
        if (i < C)
            E::store1(dweight, i, E::load1(dweight, i) + sum);
        else
            E::store1(dbias, i - C, E::load1(dbias, i - C) + sum);
    }
}

template <typename T, int VPL>
const void* rows_kernel_ptr() {
    return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPL>);
}

// Instantiated lane widths (16-byte vectors per lane); a row uses the smallest
// one that covers it.
constexpr int kVpl[] = {1, 2, 3, 4, 6, 7, 8, 12, 16};

template <typename T>
const void* rows_kernel_for(int vpl) {
    switch (vpl) {
        case 1: return rows_kernel_ptr<T, 1>();
        case 2: return rows_kernel_ptr<T, 2>();
        case 3: return rows_kernel_ptr<T, 3>();
        case 4: return rows_kernel_ptr<T, 4>();
        case 6: return rows_kernel_ptr<T, 6>();
        case 7: return rows_kernel_ptr<T, 7>();
        case 8: return rows_kernel_ptr<T, 8>();
        case 12: return rows_kernel_ptr<T, 12>();
        default: return rows_kernel_ptr<T, 16>();
    }
}

cudaError_t launch_pdl(const void* k, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void** args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace

int ln_vec_elems(int dtype) { return dtype == MMBWD_F32 ? 4 : 8; }

cudaError_t ln_make_plan(int64_t BT, int C, int dtype, int num_sms, LnPlan* plan) {
    *plan = LnPlan{};
    const int N = ln_vec_elems(dtype);
    const int nvec = C / N;
    int vpl = 16;
    for (int v : kVpl)
        if (32 * v >= nvec) {
            vpl = v;
            break;
        }
    int warps = LN_MAX_WARPS;
    auto smem_for = [C](int w) { return static_cast<size_t>(C) * 4 * (1 + 2 * static_cast<size_t>(w)); };
    while (warps > 1 && smem_for(warps) > LN_SMEM_LIMIT) warps /= 2;
    const size_t smem = smem_for(warps);
    const void* k = dtype == MMBWD_F32 ? rows_kernel_for<float>(vpl) : rows_kernel_for<__nv_bfloat16>(vpl);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, warps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
    const int64_t max_grid = (BT + warps - 1) / warps;  // at least one row per warp
    if (grid > max_grid) grid = max_grid;
    if (grid < 1) grid = 1;
    const int64_t rows = (BT + grid - 1) / grid;
    plan->vpl = vpl;
    plan->warps = warps;
    plan->rows_per_block = rows;
    plan->grid = static_cast<int>((BT + rows - 1) / rows);  // no empty block
    plan->smem = smem;
    plan->ws_bytes = static_cast<size_t>(plan->grid) * 2 * static_cast<size_t>(C) * 4;
    return cudaSuccess;
}

cudaError_t ln_launch(const LnPlan& plan, void* dinp, void* dweight, void* dbias, const void* dout,
                      const void* inp, const void* weight, const float* mean, const float* rstd, int64_t BT,
                      int C, int dtype, void* ws, cudaStream_t stream) {
    LnParams p{};
    p.dinp = dinp;
    p.dout = dout;
    p.inp = inp;
    p.weight = weight;
    p.mean = mean;
    p.rstd = rstd;
    p.partials = static_cast<float*>(ws);
    p.BT = BT;
    p.rows_per_block = plan.rows_per_block;
    p.C = C;
    p.nvec = C / ln_vec_elems(dtype);
    const void* k = dtype == MMBWD_F32 ? rows_kernel_for<float>(plan.vpl) : rows_kernel_for<__nv_bfloat16>(plan.vpl);
    void* args[] = {&p};
    cudaError_t e = launch_pdl(k, dim3(plan.grid), dim3(plan.warps * 32), plan.smem, stream, args);
    if (e != cudaSuccess) return e;
    const unsigned pblocks = static_cast<unsigned>((2 * C + 31) / 32);
    const void* pk = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&ln_bwd_params_kernel<float>)
                                        : reinterpret_cast<const void*>(&ln_bwd_params_kernel<__nv_bfloat16>);
    float* partials = p.partials;
    int grid = plan.grid;
    void* pargs[] = {&dweight, &dbias, &partials, &grid, &C};
    return launch_pdl(pk, dim3(pblocks), dim3(LN_PARAM_WARPS * 32), 0, stream, pargs);
}

}  // namespace mmbwd

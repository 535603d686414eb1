// LayerNorm backward (llm.c dev/cuda/layernorm_backward.cu, layernorm_backward_cpu):
// per row, two row means of g = weight * dout, then dinp += rstd (g - a - n c);
// dweight and dbias are sums over all rows of n * dout and dout.
//
// The work is bound by HBM: each row's dout and inp are read once and its dinp
// read and written once (4 row-lengths of traffic per row); the weight row and
// the parameter-gradient sums stay on chip.
//
// Rows kernel (one block of 16 warps per SM, a contiguous range of rows per
// block). Warps form teams of P warps (P a compile-time parameter); a team
// takes two rows at a time (rows k and k + teams, then k + 2 teams ...). A
// thread owns the 16-byte column vectors t, t + 32P (at most two) of every
// row of its team. It copies its share of dout, inp and the old dinp of the
// next two rows into its team's two-stage shared-memory buffer with cp.async
// while it computes the current two, and reads back only the bytes it copied
// itself, so its own cp.async.wait_group is the only wait the data needs. Its
// share of dweight and dbias stays in registers for the block's whole range
// of rows. The two row sums are reduced in the warp with an xor butterfly
// (the same bits in every lane) and across the team's warps through shared
// memory in warp order behind a named barrier of the team. At the end the
// teams' sums are added in team order and the block writes one fp32 partial
// row pair to the workspace. There is no spin wait anywhere: the only waits
// are cp.async group waits and hardware barriers that every warp of the
// block or team reaches.
//
// Params kernel: for each group of 32 columns, 32 warps each sum a fixed
// contiguous range of the block partials in block order, then one warp adds
// the warp sums in warp order, adds the old dweight / dbias and rounds once.
//
// Both kernels are launched with programmatic stream serialization and touch
// global memory only after `griddepcontrol.wait`.
#include "../../include/layernorm_backward.h"
#include "../../include/mmbwd.h"
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace mmbwd {

// Status word of the LayerNorm kernels (they have no bounded waits that could
// give up; kept so that the device status covers every kernel of the library).
__device__ unsigned int g_ln_status[4];

namespace {

constexpr int LN_WARPS = 16;
constexpr int LN_THREADS = LN_WARPS * 32;
constexpr int LN_MAX_VPT = 2;  // 16-byte vectors per thread and row
constexpr int LN_PARAM_WARPS = 32;

__device__ __forceinline__ void ln_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void ln_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// 16-byte asynchronous copy global -> shared (L2 only), and its group waits
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void team_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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
    int nvec;        // C / N
    int team_warps;  // P
};

template <typename T, int VPT, int P>
__global__ void __launch_bounds__(LN_THREADS, 1) ln_bwd_rows_kernel(const LnParams p) {
    using E = LnElem<T>;
    constexpr int N = E::N;
    extern __shared__ __align__(16) float ln_smem[];
    const int C = p.C;
    constexpr int teams = LN_WARPS / P;
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int team = warp / P, pw = warp % P;
    const int tt = pw * 32 + lane;  // thread index in the team
    float* w_s = ln_smem;                                    // weight as fp32, C
    float* red = ln_smem + C;                                // [teams][2][P][4] row sums
    // [teams][2C] team sums at the end; during the row loop the same region
    // (sized for both) holds each team's two-stage row buffer
    float* tsum = red + static_cast<size_t>(teams) * 2 * P * 4;

    ln_grid_wait();  // global memory only from here on
    for (int i = threadIdx.x; i < C; i += blockDim.x) w_s[i] = E::load1(p.weight, i);
    __syncthreads();

    // a vector's weights: 128-bit shared loads (a thread's 4 or 8 consecutive floats)
    auto weights = [&](int v, float (&w)[N]) {
#pragma unroll
        for (int q = 0; q < N; q += 4) {
            const float4 t = *reinterpret_cast<const float4*>(w_s + v * N + q);
            w[q] = t.x, w[q + 1] = t.y, w[q + 2] = t.z, w[q + 3] = t.w;
        }
    };

    float acc_w[VPT][N], acc_b[VPT][N];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < N; ++e) acc_w[j][e] = acc_b[j][e] = 0.f;

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_block;
    const int64_t r1 = r0 + p.rows_per_block < p.BT ? r0 + p.rows_per_block : p.BT;
    // Two-stage buffer of this team: [stage][row][dout | inp | dinp][C] in the
    // storage type. A thread copies its own vectors with cp.async and reads
    // back only those bytes, so its own wait_group is the only wait needed.
    const uint32_t row_bytes = static_cast<uint32_t>(C) * sizeof(T);
    const uint32_t stage_bytes = 6 * row_bytes;
    const uint32_t team_buf = ptx::smem_u32(tsum) + static_cast<uint32_t>(team) * 2 * stage_bytes;
    auto issue = [&](int64_t k, int stage) {  // copies of rows k and k + teams (those < r1)
        const uint32_t sb = team_buf + static_cast<uint32_t>(stage) * stage_bytes;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t r = k + q * teams;
            if (r < r1) {
#pragma unroll
                for (int t3 = 0; t3 < 3; ++t3) {
                    const void* src = t3 == 0 ? p.dout : (t3 == 1 ? p.inp : static_cast<const void*>(p.dinp));
                    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const T*>(src) + r * C);
                    const uint32_t dst = sb + static_cast<uint32_t>(q * 3 + t3) * row_bytes;
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const int v = tt + 32 * P * j;
                        if (v < p.nvec) cp_async16(dst + 16u * v, row + v);
                    }
                }
            }
        }
        cp_async_commit();
    };

    // row statistics travel one iteration ahead in registers
    float st[4] = {0.f, 0.f, 0.f, 0.f};  // mean, rstd of rows k and k + teams
    auto stats = [&](int64_t k, float (&o)[4]) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t r = k + q * teams < r1 ? k + q * teams : k;
            o[2 * q] = __ldg(p.mean + r);
            o[2 * q + 1] = __ldg(p.rstd + r);
        }
    };
    int par = 0, stage = 0;
    if (r0 + team < r1) {
        issue(r0 + team, 0);
        stats(r0 + team, st);
    }
    for (int64_t k = r0 + team; k < r1; k += 2 * teams, par ^= 1, stage ^= 1) {
        const int64_t rows[2] = {k, k + teams};
        const bool two = rows[1] < r1;
        // the next iteration's rows are in flight while this one is computed
        float st_next[4] = {0.f, 0.f, 0.f, 0.f};
        if (k + 2 * teams < r1) {
            issue(k + 2 * teams, stage ^ 1);
            stats(k + 2 * teams, st_next);
        } else {
            cp_async_commit();  // an empty group keeps the count of groups in step
        }
        cp_async_wait_one();    // this iteration's group has landed (for this thread)
        const uint32_t sb = team_buf + static_cast<uint32_t>(stage) * stage_bytes;
        uint4 vd[2][VPT], vx[2][VPT], vo[2][VPT];
        float m[2], sd[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            m[q] = st[2 * q];
            sd[q] = st[2 * q + 1];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = tt + 32 * P * j;
                if (v < p.nvec && (q == 0 || two)) {
                    vd[q][j] = ptx::lds128(sb + static_cast<uint32_t>(q * 3 + 0) * row_bytes + 16u * v);
                    vx[q][j] = ptx::lds128(sb + static_cast<uint32_t>(q * 3 + 1) * row_bytes + 16u * v);
                    vo[q][j] = ptx::lds128(sb + static_cast<uint32_t>(q * 3 + 2) * row_bytes + 16u * v);
                }
            }
        }

        // first pass: the two row sums of each row
        float su[4] = {0.f, 0.f, 0.f, 0.f};  // sa0, sc0, sa1, sc1
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (q == 1 && !two) break;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = tt + 32 * P * j;
                if (v < p.nvec) {
                    float d[N], x[N], w[N];
                    E::unpack(vd[q][j], d);
                    E::unpack(vx[q][j], x);
                    weights(v, w);
#pragma unroll
                    for (int e = 0; e < N; ++e) {
                        const float g = w[e] * d[e];
                        su[2 * q] += g;
                        su[2 * q + 1] += g * ((x[e] - m[q]) * sd[q]);
                    }
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int u = 0; u < 4; ++u) su[u] += __shfl_xor_sync(0xffffffffu, su[u], off);
        if (P > 1) {
            // across the team's warps, in warp order (buffer `par`: the previous
            // use of this buffer was read before every warp reached the last
            // barrier of the team)
            float* rb = red + (static_cast<size_t>(team) * 2 + par) * P * 4;
            if (lane == 0)
#pragma unroll
                for (int u = 0; u < 4; ++u) rb[pw * 4 + u] = su[u];
            team_sync(1 + team, 32 * P);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float t = rb[u];
                for (int w = 1; w < P; ++w) t += rb[w * 4 + u];
                su[u] = t;
            }
        }

        // second pass: dinp, and this thread's parameter sums (row k, then k + teams)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (q == 1 && !two) break;
            const float a = su[2 * q] / static_cast<float>(C), c = su[2 * q + 1] / static_cast<float>(C);
            const float sda = sd[q] * a, sdc = sd[q] * c;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<T*>(p.dinp) + rows[q] * C);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = tt + 32 * P * j;
                if (v < p.nvec) {
                    float d[N], x[N], o[N], w[N];
                    E::unpack(vd[q][j], d);
                    E::unpack(vx[q][j], x);
                    E::unpack(vo[q][j], o);
                    weights(v, w);
#pragma unroll
                    for (int e = 0; e < N; ++e) {
                        const float nrm = (x[e] - m[q]) * sd[q];
                        // rstd * (g - a - n c), as sd*g - sd*a - (sd*c)*n
                        o[e] += fmaf(sd[q], w[e] * d[e], -fmaf(sdc, nrm, sda));
                        acc_w[j][e] = fmaf(nrm, d[e], acc_w[j][e]);
                        acc_b[j][e] += d[e];
                    }
                    __stcg(orow + v, E::pack(o));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) st[u] = st_next[u];
    }

    // the teams' sums, added in team order (the row buffers are free once
    // every team has finished)
    cp_async_wait_all();
    __syncthreads();
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tt + 32 * P * j;
        if (v < p.nvec) {
            float* dw = tsum + static_cast<size_t>(team) * 2 * C + v * N;
            float* db = dw + C;
#pragma unroll
            for (int e = 0; e < N; ++e) {
                dw[e] = acc_w[j][e];
                db[e] = acc_b[j][e];
            }
        }
    }
    __syncthreads();
    ln_launch_dependents();
    float* dst = p.partials + static_cast<size_t>(blockIdx.x) * 2 * C;
    for (int i = threadIdx.x * 4; i < 2 * C; i += blockDim.x * 4) {
        float4 acc = *reinterpret_cast<const float4*>(tsum + i);
        for (int t = 1; t < teams; ++t) {
            const float4 v = *reinterpret_cast<const float4*>(tsum + static_cast<size_t>(t) * 2 * C + i);
            acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
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

template <typename T, int VPT>
const void* rows_kernel_p(int P) {
    switch (P) {
        case 1: return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPT, 1>);
        case 2: return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPT, 2>);
        case 4: return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPT, 4>);
        case 8: return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPT, 8>);
        default: return reinterpret_cast<const void*>(&ln_bwd_rows_kernel<T, VPT, 16>);
    }
}

template <typename T>
const void* rows_kernel_for(int vpt, int P) {
    return vpt == 1 ? rows_kernel_p<T, 1>(P) : rows_kernel_p<T, 2>(P);
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
    // team width: the fewest warps (a power of two) that cover a row with at
    // most two vectors per thread
    int P = 1;
    while (P < LN_WARPS && nvec > 32 * P * LN_MAX_VPT) P *= 2;
    const int vpt = (nvec + 32 * P - 1) / (32 * P);
    if (vpt > LN_MAX_VPT) return cudaErrorInvalidValue;
    const int teams = LN_WARPS / P;
    plan->vpl = vpt;
    plan->team_warps = P;
    plan->warps = LN_WARPS;
    const size_t es = dtype == MMBWD_F32 ? 4 : 2;
    const size_t rows_buf = static_cast<size_t>(teams) * 2 * 6 * C * es;  // two stages of two rows
    plan->smem = 4 * (static_cast<size_t>(C) + static_cast<size_t>(teams) * 2 * P * 4) +
                 std::max(rows_buf, static_cast<size_t>(teams) * 2 * C * 4);
    const void* k = dtype == MMBWD_F32 ? rows_kernel_for<float>(vpt, P) : rows_kernel_for<__nv_bfloat16>(vpt, P);
    cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(plan->smem));
    if (e != cudaSuccess) return e;
    int64_t grid = num_sms;  // one block per SM
    if (grid > BT) grid = BT;
    if (grid < 1) grid = 1;
    const int64_t rows = (BT + grid - 1) / grid;
    plan->rows_per_block = rows;
    plan->grid = static_cast<int>((BT + rows - 1) / rows);  // no empty block
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
    p.team_warps = plan.team_warps;
    const void* k = dtype == MMBWD_F32 ? rows_kernel_for<float>(plan.vpl, plan.team_warps)
                                       : rows_kernel_for<__nv_bfloat16>(plan.vpl, plan.team_warps);
    void* args[] = {&p};
    cudaError_t e = launch_pdl(k, dim3(plan.grid), dim3(LN_THREADS), plan.smem, stream, args);
    if (e != cudaSuccess) return e;
    const unsigned pblocks = static_cast<unsigned>((2 * C + 31) / 32);
    const void* pk = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&ln_bwd_params_kernel<float>)
                                        : reinterpret_cast<const void*>(&ln_bwd_params_kernel<__nv_bfloat16>);
    float* partials = p.partials;
    int grid = plan.grid;
    void* pargs[] = {&dweight, &dbias, &partials, &grid, &C};
    return launch_pdl(pk, dim3(pblocks), dim3(LN_PARAM_WARPS * 32), 0, stream, pargs);
}

cudaError_t ln_read_status(int* code, int* info3, bool reset) {
    unsigned int h[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(h, g_ln_status, sizeof(h));
    if (e != cudaSuccess) return e;
    *code = h[0] ? -static_cast<int>(h[0]) : MMBWD_OK;
    if (info3) {
        info3[0] = static_cast<int>(h[1]);
        info3[1] = static_cast<int>(h[2]);
        info3[2] = static_cast<int>(h[3]);
    }
    if (reset) {
        const unsigned int z[4] = {0, 0, 0, 0};
        e = cudaMemcpyToSymbol(g_ln_status, z, sizeof(z));
    }
    return e;
}

}  // namespace mmbwd

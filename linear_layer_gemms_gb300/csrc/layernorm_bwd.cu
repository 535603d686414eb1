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
// takes rows k, k + teams, k + 2 teams, ... One thread of the team streams its
// rows (dout, inp and the old dinp of one row per buffer) into the team's
// ring of four shared-memory buffers with 1-D TMA bulk copies completing on
// the buffer's mbarrier, three rows ahead of the row being computed; the team
// consumes its ring in order, so each barrier is waited on phase by phase.
// A thread owns the 16-byte column vectors t, t + 32P (at most two) of every
// row of its team; its share of dweight and dbias stays in registers for the
// block's whole range of rows. The two row sums are reduced in the warp with
// an xor butterfly (the same bits in every lane) and across the team's warps
// through shared memory in warp order behind a named barrier of the team;
// that barrier also tells the issuing thread that the team is done with the
// buffer it refills next (with an async-proxy fence before the copies).
// Every mbarrier wait is bounded (2 s): one that gives up records the failure
// in the device status word and the row is processed anyway, so that every
// warp still reaches every barrier. At the end the teams' sums are added in
// team order and the block writes one fp32 partial row pair to the workspace.
//
// Params kernel: for each group of 32 columns, 32 warps each sum a fixed
// contiguous range of the block partials in block order, then one warp adds
// the warp sums in warp order, adds the old dweight / dbias and rounds once.
//
// Both kernels are launched with programmatic stream serialization and touch
// global memory only after `griddepcontrol.wait`.
#include "../../include/layernorm_backward.h"
#include "../../include/mmbwd.h"
#include "ops.h"
#include "ptx.cuh"

#include <algorithm>

namespace mmbwd {

// Status word of the LayerNorm kernels: [0] error code (positive), [1] block,
// [2] wait site, [3] row.
__device__ unsigned int g_ln_status[4];

namespace {

constexpr int LN_WARPS = 16;
constexpr int LN_THREADS = LN_WARPS * 32;
constexpr int LN_MAX_VPT = 2;  // 16-byte vectors per thread and row
constexpr int LN_PARAM_WARPS = 32;
constexpr int LN_STAGES = 4;  // row buffers per team (three rows in flight)
constexpr unsigned long long LN_TIMEOUT_NS = 2000000000ull;
// Widest rows of the fused rows kernel (row ring and weights in shared memory,
// at most two 16-byte vectors per thread); wider rows take the two-pass path.
constexpr int LN_FUSED_MAX_C_BF16 = 4096;
constexpr int LN_FUSED_MAX_C_F32 = 2048;

enum LnSite { LN_SITE_FULL = 2, LN_SITE_TEARDOWN = 4 };

__device__ __forceinline__ void ln_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void ln_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`
// (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ void ln_record_failure(int site, int64_t row) {
    if (atomicCAS(&g_ln_status[0], 0u, static_cast<unsigned>(-MMBWD_ERR_DEVICE_TIMEOUT)) == 0u) {
        g_ln_status[1] = blockIdx.x;
        g_ln_status[2] = static_cast<unsigned>(site);
        g_ln_status[3] = static_cast<unsigned>(row);
        __threadfence();
    }
}

// Bounded wait on an mbarrier phase (2 s by the global timer); false on
// timeout (recorded, abort raised) or, unless `ignore_abort`, once the block
// has aborted.
__device__ bool ln_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort, int site, int64_t row,
                        bool ignore_abort = false) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (!ignore_abort && *abort) return false;
            if (ptx::globaltimer() - t0 > LN_TIMEOUT_NS) {
                *abort = 1u;
                ln_record_failure(site, row);
                return false;
            }
        }
    }
}

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
    uint32_t off_ring;  // bytes from the start of shared memory to the row buffers
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
    float* red = ln_smem + C;                                // [teams][2][P][2] row sums
    uint64_t* bars = reinterpret_cast<uint64_t*>(red + teams * 2 * P * 2);  // [teams][LN_STAGES]
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(bars + teams * LN_STAGES);
    // [teams][2C] team sums at the end; during the row loop the same region
    // (sized for both, 128-byte aligned) holds each team's ring of row buffers
    float* tsum = reinterpret_cast<float*>(ln_smem + p.off_ring / 4);

    if (threadIdx.x == 0) {
        for (int b = 0; b < teams * LN_STAGES; ++b) ptx::mbar_init(ptx::smem_u32(bars + b), 1);
        *abort = 0u;
        ptx::fence_mbar_init();
    }
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
    // this thread's weights are the same for every row: registers
    float wr[VPT][N];
#pragma unroll
    for (int jj = 0; jj < VPT; ++jj) {
        const int v = tt + 32 * P * jj;
        if (v < p.nvec) {
            weights(v, wr[jj]);
        } else {
#pragma unroll
            for (int e = 0; e < N; ++e) wr[jj][e] = 0.f;
        }
    }

    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_block;
    const int64_t r1 = r0 + p.rows_per_block < p.BT ? r0 + p.rows_per_block : p.BT;
    // This team's ring of LN_STAGES row buffers ([dout | inp | dinp] of one
    // row each, storage type) and its "full" barriers. One thread of the team
    // issues the bulk copies of the team's rows in order; the team consumes
    // them in order, so each barrier is waited on phase by phase.
    const uint32_t row_bytes = static_cast<uint32_t>(C) * sizeof(T);
    const uint32_t stage_bytes = 3 * row_bytes;
    const uint32_t team_buf = ptx::smem_u32(tsum) + static_cast<uint32_t>(team) * LN_STAGES * stage_bytes;
    const uint32_t full0 = ptx::smem_u32(bars) + static_cast<uint32_t>(team) * LN_STAGES * 8u;
    const bool issuer = pw == 0 && lane == 0;
    const int64_t first = r0 + team;  // the team's rows: first + j * teams
    const int nj = first < r1 ? static_cast<int>((r1 - first + teams - 1) / teams) : 0;
    auto issue = [&](int j) {
        const int64_t off = (first + static_cast<int64_t>(j) * teams) * C;
        const uint32_t st = static_cast<uint32_t>(j % LN_STAGES);
        const uint32_t bar = full0 + 8u * st, dst = team_buf + st * stage_bytes;
        // the team's earlier reads of this buffer come before the copies' writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ptx::mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_load(dst, static_cast<const T*>(p.dout) + off, row_bytes, bar);
        bulk_load(dst + row_bytes, static_cast<const T*>(p.inp) + off, row_bytes, bar);
        bulk_load(dst + 2 * row_bytes, static_cast<const T*>(p.dinp) + off, row_bytes, bar);
    };
    if (issuer)
        for (int j = 0; j < LN_STAGES - 1 && j < nj; ++j) issue(j);

    // the row statistics one row ahead: the next row's load overlaps this row
    float m_next = 0.f, sd_next = 0.f;
    if (nj > 0) m_next = __ldg(p.mean + first), sd_next = __ldg(p.rstd + first);
    int par = 0;
    for (int j = 0; j < nj; ++j, par ^= 1) {
        const int64_t r = first + static_cast<int64_t>(j) * teams;
        const float m = m_next, sd = sd_next;
        if (j + 1 < nj) m_next = __ldg(p.mean + r + teams), sd_next = __ldg(p.rstd + r + teams);
        // A wait that gives up is recorded (device status) and the row is
        // processed anyway, so that every warp still reaches every barrier.
        ln_wait(full0 + 8u * (j % LN_STAGES), static_cast<uint32_t>((j / LN_STAGES) & 1), abort, LN_SITE_FULL, r);
        const uint32_t sb = team_buf + static_cast<uint32_t>(j % LN_STAGES) * stage_bytes;

        // first pass: the two row sums; dout and the normalised input stay in
        // registers for the second pass
        float sa = 0.f, sc = 0.f;
        float d[VPT][N], nrm[VPT][N];
#pragma unroll
        for (int jj = 0; jj < VPT; ++jj) {
            const int v = tt + 32 * P * jj;
            if (v < p.nvec) {
                float x[N];
                E::unpack(ptx::lds128(sb + 16u * v), d[jj]);
                E::unpack(ptx::lds128(sb + row_bytes + 16u * v), x);
#pragma unroll
                for (int e = 0; e < N; ++e) {
                    nrm[jj][e] = (x[e] - m) * sd;
                    const float g = wr[jj][e] * d[jj][e];
                    sa += g;
                    sc += g * nrm[jj][e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < N; ++e) d[jj][e] = nrm[jj][e] = 0.f;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, off);
            sc += __shfl_xor_sync(0xffffffffu, sc, off);
        }
        if (P > 1) {
            // across the team's warps, in warp order (buffer `par`: its previous
            // use was read before every warp reached the team's last barrier)
            float* rb = red + (static_cast<size_t>(team) * 2 + par) * P * 2;
            if (lane == 0) rb[pw * 2] = sa, rb[pw * 2 + 1] = sc;
            team_sync(1 + team, 32 * P);
            sa = rb[0];
            sc = rb[1];
            for (int w = 1; w < P; ++w) sa += rb[2 * w], sc += rb[2 * w + 1];
        } else {
            __syncwarp();
        }
        // Every warp of the team is past its second pass of row j - 1 (it came
        // before the barrier above): that row's buffer takes row j + LN_STAGES - 1.
        if (issuer && j + LN_STAGES - 1 < nj) issue(j + LN_STAGES - 1);

        // second pass: dinp, and this thread's parameter sums
        const float a = sa / static_cast<float>(C), c = sc / static_cast<float>(C);
        const float sda = sd * a, sdc = sd * c;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<T*>(p.dinp) + r * C);
#pragma unroll
        for (int jj = 0; jj < VPT; ++jj) {
            const int v = tt + 32 * P * jj;
            if (v < p.nvec) {
                float o[N];
                E::unpack(ptx::lds128(sb + 2 * row_bytes + 16u * v), o);
#pragma unroll
                for (int e = 0; e < N; ++e) {
                    // rstd * (g - a - n c), as sd*g - sd*a - (sd*c)*n
                    o[e] += fmaf(sd, wr[jj][e] * d[jj][e], -fmaf(sdc, nrm[jj][e], sda));
                    acc_w[jj][e] = fmaf(nrm[jj][e], d[jj][e], acc_w[jj][e]);
                    acc_b[jj][e] += d[jj][e];
                }
                __stcg(orow + v, E::pack(o));
            }
        }
    }
    // copies in flight land before the buffers are reused (normally all have
    // been waited for already)
    if (issuer)
        for (int j = nj - LN_STAGES > 0 ? nj - LN_STAGES : 0; j < nj; ++j)
            ln_wait(full0 + 8u * (j % LN_STAGES), static_cast<uint32_t>((j / LN_STAGES) & 1), abort,
                    LN_SITE_TEARDOWN, first + static_cast<int64_t>(j) * teams, true);

    // the teams' sums, added in team order (the row buffers are free once
    // every team has finished)
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
    // the old value, requested beside the partials rather than after their sum
    float old = 0.f;
    if (warp == 0 && i < 2 * C) old = i < C ? E::load1(dweight, i) : E::load1(dbias, i - C);
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
            E::store1(dweight, i, old + sum);
        else
            E::store1(dbias, i - C, old + sum);
    }
}

// ---------------------------------------------------------------------------
// Rows too wide for the fused kernel (its row buffers and weights in shared
// memory): two passes over global memory, any C.
//   ln_wide_sums_kernel: one warp per row (grid-stride) forms the row's two
//     sums, sum of g = w*dout and of g*n, lanes over 16-byte vectors in order
//     and an xor butterfly, and stores them as a float pair;
//   ln_wide_cols_kernel: block (column tile of 256 vectors, range of rows);
//     each thread owns one vector of the tile, walks the block's rows in order
//     (four rows' loads in flight) applying dinp += rstd (g - a - n c), and
//     keeps its columns' n*dout and dout sums in registers; one fp32 partial
//     row pair per block, which the params kernel adds in block order.
constexpr int LN_WIDE_TILE = 256;  // vectors per column tile (one per thread)

template <typename T>
__global__ void __launch_bounds__(256) ln_wide_sums_kernel(const T* __restrict__ dout, const T* __restrict__ inp,
                                                           const T* __restrict__ weight, const float* __restrict__ mean,
                                                           const float* __restrict__ rstd, float2* __restrict__ sums,
                                                           int64_t BT, int C) {
    using E = LnElem<T>;
    constexpr int N = E::N;
    ln_grid_wait();
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int nvec = C / N;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < BT; r += warps) {
        const float m = mean[r], sd = rstd[r];
        const uint4* dr = reinterpret_cast<const uint4*>(dout + r * C);
        const uint4* xr = reinterpret_cast<const uint4*>(inp + r * C);
        float sa = 0.f, sc = 0.f;
        for (int v = lane; v < nvec; v += 32) {
            float d[N], x[N], w[N];
            E::unpack(__ldg(dr + v), d);
            E::unpack(__ldg(xr + v), x);
            E::unpack(__ldg(reinterpret_cast<const uint4*>(weight) + v), w);
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const float g = w[e] * d[e];
                sa += g;
                sc += g * ((x[e] - m) * sd);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, off);
            sc += __shfl_xor_sync(0xffffffffu, sc, off);
        }
        if (lane == 0) sums[r] = make_float2(sa, sc);
    }
    ln_launch_dependents();
}

template <typename T>
__global__ void __launch_bounds__(LN_WIDE_TILE) ln_wide_cols_kernel(const LnParams p, const float2* __restrict__ sums) {
    using E = LnElem<T>;
    constexpr int N = E::N;
    ln_grid_wait();
    const int v = static_cast<int>(blockIdx.x) * LN_WIDE_TILE + static_cast<int>(threadIdx.x);
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * p.rows_per_block;
    const int64_t r1 = r0 + p.rows_per_block < p.BT ? r0 + p.rows_per_block : p.BT;
    const int C = p.C;
    float acc_w[N], acc_b[N], w[N];
#pragma unroll
    for (int e = 0; e < N; ++e) acc_w[e] = acc_b[e] = w[e] = 0.f;
    const bool on = v < p.nvec;
    if (on) E::unpack(__ldg(reinterpret_cast<const uint4*>(p.weight) + v), w);
    const float inv_c = 1.f / static_cast<float>(C);
    constexpr int RU = 4;  // rows in flight
    for (int64_t rb = r0; rb < r1 && on; rb += RU) {
        uint4 dv[RU], xv[RU], ov[RU];
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            const int64_t r = rb + u < r1 ? rb + u : r1 - 1;
            dv[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + r * C) + v);
            xv[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.inp) + r * C) + v);
            ov[u] = *(reinterpret_cast<const uint4*>(static_cast<const T*>(p.dinp) + r * C) + v);
        }
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            const int64_t r = rb + u;
            if (r >= r1) break;
            const float m = __ldg(p.mean + r), sd = __ldg(p.rstd + r);
            const float2 sm = sums[r];
            const float a = sm.x * inv_c, c = sm.y * inv_c;
            const float sda = sd * a, sdc = sd * c;
            float d[N], x[N], o[N];
            E::unpack(dv[u], d);
            E::unpack(xv[u], x);
            E::unpack(ov[u], o);
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const float n = (x[e] - m) * sd;
                o[e] += fmaf(sd, w[e] * d[e], -fmaf(sdc, n, sda));
                acc_w[e] = fmaf(n, d[e], acc_w[e]);
                acc_b[e] += d[e];
            }
            __stcg(reinterpret_cast<uint4*>(static_cast<T*>(p.dinp) + r * C) + v, E::pack(o));
        }
    }
    ln_launch_dependents();
    if (on) {
        float* dst = p.partials + static_cast<size_t>(blockIdx.y) * 2 * C + static_cast<size_t>(v) * N;
#pragma unroll
        for (int e = 0; e < N; e += 4) {
            __stcg(reinterpret_cast<float4*>(dst + e), make_float4(acc_w[e], acc_w[e + 1], acc_w[e + 2], acc_w[e + 3]));
            __stcg(reinterpret_cast<float4*>(dst + C + e),
                   make_float4(acc_b[e], acc_b[e + 1], acc_b[e + 2], acc_b[e + 3]));
        }
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
    if (C > (dtype == MMBWD_F32 ? LN_FUSED_MAX_C_F32 : LN_FUSED_MAX_C_BF16)) {
        // wide rows: column tiles x row blocks, about four blocks per SM
        plan->wide = 1;
        plan->col_tiles = (nvec + LN_WIDE_TILE - 1) / LN_WIDE_TILE;
        int64_t row_blocks = std::max<int64_t>(1, (4 * static_cast<int64_t>(std::max(num_sms, 1)) + plan->col_tiles - 1) /
                                                      plan->col_tiles);
        row_blocks = std::min<int64_t>(row_blocks, std::min<int64_t>(BT, 65535));
        const int64_t rows = (BT + row_blocks - 1) / row_blocks;
        plan->rows_per_block = rows;
        plan->grid = static_cast<int>((BT + rows - 1) / rows);  // row blocks, none empty
        plan->ws_bytes = static_cast<size_t>(plan->grid) * 2 * static_cast<size_t>(C) * 4 + static_cast<size_t>(BT) * 8;
        return cudaSuccess;
    }
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
    const size_t rows_buf = static_cast<size_t>(teams) * LN_STAGES * 3 * C * es;  // each team's ring
    const size_t head = 4 * (static_cast<size_t>(C) + static_cast<size_t>(teams) * 2 * P * 2) +
                        8 * static_cast<size_t>(teams) * LN_STAGES + 8;  // weight, row sums, barriers, flag
    plan->off_ring = (head + 127) / 128 * 128;
    plan->smem = plan->off_ring + std::max(rows_buf, static_cast<size_t>(teams) * 2 * C * 4);
    if (plan->smem > 227 * 1024) return cudaErrorInvalidValue;
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
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
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
    p.off_ring = static_cast<uint32_t>(plan.off_ring);
    cudaError_t e = cudaSuccess;
    if (plan.wide) {
        // row sums after the partials (the workspace holds [grid][2][C] fp32, then the pairs)
        float2* sums = reinterpret_cast<float2*>(p.partials + static_cast<size_t>(plan.grid) * 2 * C);
        const void* sk = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&ln_wide_sums_kernel<float>)
                                            : reinterpret_cast<const void*>(&ln_wide_sums_kernel<__nv_bfloat16>);
        int64_t bt = BT;
        int c = C;
        void* sargs[] = {const_cast<void**>(&dout), const_cast<void**>(&inp), const_cast<void**>(&weight),
                         const_cast<float**>(&mean), const_cast<float**>(&rstd), &sums, &bt, &c};
        const unsigned sblocks = static_cast<unsigned>(std::min<int64_t>((BT + 7) / 8, 65535));
        e = launch_pdl(sk, dim3(sblocks), dim3(256), 0, stream, sargs);
        if (e != cudaSuccess) return e;
        const void* ck = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&ln_wide_cols_kernel<float>)
                                            : reinterpret_cast<const void*>(&ln_wide_cols_kernel<__nv_bfloat16>);
        void* cargs[] = {&p, &sums};
        e = launch_pdl(ck, dim3(static_cast<unsigned>(plan.col_tiles), static_cast<unsigned>(plan.grid)),
                       dim3(LN_WIDE_TILE), 0, stream, cargs);
    } else {
        const void* k = dtype == MMBWD_F32 ? rows_kernel_for<float>(plan.vpl, plan.team_warps)
                                           : rows_kernel_for<__nv_bfloat16>(plan.vpl, plan.team_warps);
        void* args[] = {&p};
        e = launch_pdl(k, dim3(plan.grid), dim3(LN_THREADS), plan.smem, stream, args);
    }
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

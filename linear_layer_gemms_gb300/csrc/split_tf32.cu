// fp32 operands of the linear-layer backward split into tf32 halves, laid out
// K-major for the three-product tensor-core path (MODE 2 of tc_mmbwd_kernel).
//
// The fp32 path needs fp32-accurate products (llm.c dev/cuda/matmul_backward.cu
// turns TF32 off in its main for exactly that reason). A value x is split into
//   hi = x with its 13 low mantissa bits cleared   (a tf32 value, exactly)
//   lo = x - hi                                     (exact in fp32, |lo| < 2^-10 |x|)
// and x*y is formed as hi_x*hi_y + hi_x*lo_y + lo_x*hi_y: the dropped lo_x*lo_y
// and the tf32 reading of lo leave a relative error near 2^-20 per product,
// below fp32 accumulation error over the long reductions.
//
// Layouts (every product becomes D += A . B^T with both operands K-major):
//   dinp    (BT x C) += dout (BT x OC) . (weight^T) (C x OC)^T   A = dout,    B = weight^T
//   dweight (OC x C) += (dout^T) (OC x BT) . (inp^T) (C x BT)^T  A = dout^T,  B = inp^T
// so dout's low parts are written with its own layout and both parts
// transposed, weight and inp transposed. The tensor core reads an fp32
// operand of a tf32 product as its tf32 truncation (the low 13 mantissa bits
// ignored: measured bit for bit on GB300, the raw dout in place of its cleared
// copy gave identical results), so a tensor in its own layout serves as its
// own high part and only its low part is copied. The transposing pass over
// dout also sums each 32-row tile of every column, and a second small kernel
// adds those tile sums in tile order: dbias.
#include "../../include/mmbwd.h"
#include "internal.h"
#include "ops.h"

namespace mmbwd {
namespace {

constexpr int TILE = 32;

__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    lo = x - hi;
}

// src (R x Cc, row-major, Cc a multiple of 4) in 64 x 64 tiles, 256 threads,
// 16-byte accesses throughout:
//   COPY:   lo with the layout of src (src itself is the high part)
//   TRANS:  thi / tlo = the transpose (Cc x R), row pitch ldT (a multiple of 4,
//           >= R; the pitch's padding columns may be written)
//   COLSUM: part[32-row tile][c] = the sum of the tile's rows of column c, in
//           row order (two 32-row tiles per block)
constexpr int ST = 64;        // tile side
constexpr int ST_PAD = ST + 1;  // shared row pitch: the transposed reads fall in distinct banks
template <bool COPY, bool TRANS, bool COLSUM>
__global__ void __launch_bounds__(256) split_kernel(const float* __restrict__ src, int64_t R, int64_t Cc,
                                                    float* __restrict__ lo, float* __restrict__ thi,
                                                    float* __restrict__ tlo, int64_t ldT, float* __restrict__ part) {
    __shared__ float t[ST][ST_PAD];
    const int tid = static_cast<int>(threadIdx.x);
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * ST, c0 = static_cast<int64_t>(blockIdx.x) * ST;
    // load: 64 rows x 16 float4; thread tid takes float4 q = tid % 16 of rows tid / 16 + 16 i
    const int q = tid & 15;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int lr = (tid >> 4) + 16 * i;
        const int64_t r = r0 + lr, c = c0 + 4 * q;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < R && c < Cc) {
            x = __ldcs(reinterpret_cast<const float4*>(src + r * Cc + c));
            if (COPY) {
                float h, l0, l1, l2, l3;
                split_tf32(x.x, h, l0);
                split_tf32(x.y, h, l1);
                split_tf32(x.z, h, l2);
                split_tf32(x.w, h, l3);
                *reinterpret_cast<float4*>(lo + r * Cc + c) = make_float4(l0, l1, l2, l3);
            }
        }
        t[lr][4 * q] = x.x;
        t[lr][4 * q + 1] = x.y;
        t[lr][4 * q + 2] = x.z;
        t[lr][4 * q + 3] = x.w;
    }
    if (!TRANS && !COLSUM) return;
    __syncthreads();
    if (TRANS) {
        // transposed row c0 + oc holds source rows r0 .. r0 + 63: thread tid
        // writes float4 q (source rows 4q .. 4q + 3) of rows oc = tid / 16 + 16 i
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int oc = (tid >> 4) + 16 * i;
            const int64_t c = c0 + oc, r = r0 + 4 * q;
            if (c < Cc && r < R) {
                float h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_tf32(t[4 * q + e][oc], h[e], l[e]);
                *reinterpret_cast<float4*>(thi + c * ldT + r) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4*>(tlo + c * ldT + r) = make_float4(l[0], l[1], l[2], l[3]);
            }
        }
    }
    if (COLSUM && tid < 2 * ST) {
        // column tid % 64 of 32-row half tid / 64 (rows past R hold 0)
        const int col = tid & (ST - 1), half = tid >> 6;
        const int64_t tile = static_cast<int64_t>(blockIdx.y) * 2 + half;
        if (c0 + col < Cc && r0 + 32 * half < R) {
            float s = 0.f;
            for (int i = 0; i < 32; ++i) s += t[32 * half + i][col];
            part[tile * Cc + c0 + col] = s;
        }
    }
}

// dbias[c] = sum over tile rows of part[.][c] (overwrite), in a fixed order:
// 32 columns per block, 8 slices of the tile rows; slice j sums its rows in
// order (eight loads in flight), then the slices are added in slice order.
constexpr int TS_SLICES = 8;
__global__ void __launch_bounds__(32 * TS_SLICES) tile_sum_kernel(float* __restrict__ dbias,
                                                                  const float* __restrict__ part, int64_t tiles,
                                                                  int64_t Cc) {
    __shared__ float red[TS_SLICES][32];
    const int lane = static_cast<int>(threadIdx.x & 31), j = static_cast<int>(threadIdx.x >> 5);
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
    const int64_t per = (tiles + TS_SLICES - 1) / TS_SLICES;
    const int64_t k0 = j * per, k1 = k0 + per < tiles ? k0 + per : tiles;
    float s = 0.f;
    if (c < Cc) {
#pragma unroll 8
        for (int64_t k = k0; k < k1; ++k) s += part[k * Cc + c];
    }
    red[j][lane] = s;
    __syncthreads();
    if (j == 0 && c < Cc) {
        float t = red[0][lane];
        for (int q = 1; q < TS_SLICES; ++q) t += red[q][lane];
        dbias[c] = t;
    }
}

template <bool COPY, bool TRANS, bool COLSUM>
cudaError_t launch_split(const float* src, int64_t R, int64_t Cc, float* lo, float* thi, float* tlo, int64_t ldT,
                         float* part, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((Cc + ST - 1) / ST), static_cast<unsigned>((R + ST - 1) / ST));
    split_kernel<COPY, TRANS, COLSUM><<<grid, 256, 0, stream>>>(src, R, Cc, lo, thi, tlo, ldT, part);
    return cudaGetLastError();
}

}  // namespace

int64_t x3_ld(int64_t n) { return (n + 3) / 4 * 4; }

size_t x3_workspace_bytes(int64_t BT, int64_t C, int64_t OC, bool bias) {
    auto a = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t f = 4;
    const size_t ldbt = static_cast<size_t>(x3_ld(BT));
    size_t n = 0;
    n += a(static_cast<size_t>(BT) * OC * f);      // dout lo (dout itself is the high part)
    n += 2 * a(static_cast<size_t>(OC) * ldbt * f);  // dout^T hi, lo
    n += 2 * a(static_cast<size_t>(C) * OC * f);     // weight^T hi, lo
    n += 2 * a(static_cast<size_t>(C) * ldbt * f);   // inp^T hi, lo
    if (bias) n += a(static_cast<size_t>((BT + TILE - 1) / TILE) * OC * f);
    return n;
}

bool x3_shape_ok(int64_t BT, int64_t C, int64_t OC) {
    // K-major rows of 16-byte multiples, 8-column epilogue groups, tile grids
    // within the launch limits
    return BT > 0 && C > 0 && OC > 0 && C % 8 == 0 && OC % 4 == 0 && (BT + TILE - 1) / TILE <= 65535 &&
           (OC + TILE - 1) / TILE <= 65535;
}

cudaError_t x3_launch(float* dinp, float* dweight, float* dbias, const float* dout, const float* inp,
                      const float* weight, int64_t BT, int64_t C, int64_t OC, void* ws, int num_sms,
                      cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    auto a = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const int64_t ldbt = x3_ld(BT);
    uint8_t* w = static_cast<uint8_t*>(ws);
    auto take = [&](size_t bytes) {
        float* p = reinterpret_cast<float*>(w);
        w += a(bytes);
        return p;
    };
    float* dout_lo = take(static_cast<size_t>(BT) * OC * 4);
    float* doutT_hi = take(static_cast<size_t>(OC) * ldbt * 4);
    float* doutT_lo = take(static_cast<size_t>(OC) * ldbt * 4);
    float* wT_hi = take(static_cast<size_t>(C) * OC * 4);
    float* wT_lo = take(static_cast<size_t>(C) * OC * 4);
    float* inpT_hi = take(static_cast<size_t>(C) * ldbt * 4);
    float* inpT_lo = take(static_cast<size_t>(C) * ldbt * 4);
    float* part = dbias ? take(static_cast<size_t>((BT + TILE - 1) / TILE) * OC * 4) : nullptr;

    cudaError_t e = dbias ? launch_split<true, true, true>(dout, BT, OC, dout_lo, doutT_hi, doutT_lo, ldbt,
                                                           part, stream)
                          : launch_split<true, true, false>(dout, BT, OC, dout_lo, doutT_hi, doutT_lo, ldbt,
                                                            nullptr, stream);
    if (e != cudaSuccess) return e;
    e = launch_split<false, true, false>(weight, OC, C, nullptr, wT_hi, wT_lo, OC, nullptr, stream);
    if (e != cudaSuccess) return e;
    e = launch_split<false, true, false>(inp, BT, C, nullptr, inpT_hi, inpT_lo, ldbt, nullptr, stream);
    if (e != cudaSuccess) return e;
    if (dbias) {
        tile_sum_kernel<<<static_cast<unsigned>((OC + 31) / 32), 32 * TS_SLICES, 0, stream>>>(
            dbias, part, (BT + TILE - 1) / TILE, OC);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // Both products in one launch where it fits (their tiles share the CTA
    // pairs, longest first, instead of each launch ending on a partial wave):
    // dinp (BT x C) += dout . (weight^T)^T, K = OC, and
    // dweight (OC x C) += (dout^T) . (inp^T)^T, K = BT
    static thread_local TcPlan pp;
    pp = tc_make_plan_x3_pair(BT, C, OC, num_sms);
    if (pp.n_items > 0)
        return tc_launch_x3_pair(pp, dinp, dweight, dout, dout_lo, OC, wT_hi, wT_lo, OC, doutT_hi, doutT_lo, ldbt,
                                 inpT_hi, inpT_lo, ldbt, BT, C, OC, stream);
    // dinp (BT x C) += dout . (weight^T)^T, K = OC
    const TcPlan p1 = tc_make_plan_x3(BT, C, OC, num_sms);
    e = tc_launch_x3(p1, dinp, dout, dout_lo, OC, wT_hi, wT_lo, OC, BT, C, OC, stream);
    if (e != cudaSuccess) return e;
    // dweight (OC x C) += (dout^T) . (inp^T)^T, K = BT
    const TcPlan p2 = tc_make_plan_x3(OC, C, BT, num_sms);
    return tc_launch_x3(p2, dweight, doutT_hi, doutT_lo, ldbt, inpT_hi, inpT_lo, ldbt, OC, C, BT, stream);
}

// The forward out = inp . weight^T + bias on the same path: both operands are
// already K-major, so they are only split; out is first set to the bias (or
// zero) and the product is then added to it.
bool x3_forward_shape_ok(int64_t BT, int64_t C, int64_t OC) {
    return BT > 0 && C > 0 && OC > 0 && OC % 8 == 0 && C % 4 == 0 && (BT + TILE - 1) / TILE <= 65535 &&
           (OC + TILE - 1) / TILE <= 65535;
}

size_t x3_forward_workspace_bytes(int64_t BT, int64_t C, int64_t OC) {
    auto a = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    return a(static_cast<size_t>(BT) * C * 4) + a(static_cast<size_t>(OC) * C * 4);  // the low parts
}

cudaError_t x3_forward_launch(float* out, const float* inp, const float* weight, const float* bias, int64_t BT,
                              int64_t C, int64_t OC, void* ws, int num_sms, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    auto a = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    uint8_t* w = static_cast<uint8_t*>(ws);
    // inp and weight are already K-major and serve as their own high parts
    float* inp_lo = reinterpret_cast<float*>(w);
    float* w_lo = reinterpret_cast<float*>(w + a(static_cast<size_t>(BT) * C * 4));
    cudaError_t e = fill_rows_launch(out, bias, BT, OC, MMBWD_F32, stream);
    if (e != cudaSuccess) return e;
    e = launch_split<true, false, false>(inp, BT, C, inp_lo, nullptr, nullptr, 0, nullptr, stream);
    if (e != cudaSuccess) return e;
    e = launch_split<true, false, false>(weight, OC, C, w_lo, nullptr, nullptr, 0, nullptr, stream);
    if (e != cudaSuccess) return e;
    const TcPlan p = tc_make_plan_x3(BT, OC, C, num_sms);
    return tc_launch_x3(p, out, inp, inp_lo, C, weight, w_lo, C, BT, OC, C, stream);
}

}  // namespace mmbwd

// bf16 linear-layer backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent kernel computes both products of matmul_backward (llm.c
// dev/cuda/matmul_backward.cu, matmul_backward_cpu / matmul_backward1):
//
//   dinp    (BT x C) += dout (BT x OC) . weight (OC x C)     "NN": A K-major, B MN-major
//   dweight (OC x C) += dout^T (OC x BT) . inp (BT x C)      "TN": A MN-major, B MN-major
//   dbias   (OC)      = column sums of dout                  fused into the dweight pass
//
// Work list: every 128 x 256 output tile of dinp is one item; every 128 x 256
// tile of dweight is cut into `splits` items along its long BT reduction.
// Each CTA (one per SM) walks a static, shape-determined sequence of items.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: fills a 4-stage ring of (A 16 KB, B 32 KB) tiles
//               in 128-byte-swizzled shared memory.
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma (M128 N256 K16) per
//               stage into one of two 128 x 256 fp32 accumulators in tensor
//               memory (512 columns), so the epilogue of tile i overlaps the
//               main loop of tile i+1.
//   warps 2-3   bias: on dweight items of the first column tile, sum the dout
//               tile of every stage over its BT rows (the A operand already in
//               shared memory), reduce across lanes with shuffles.
//   warps 4-7   epilogue: tcgen05.ld the accumulator (warp w owns TMEM lanes
//               32*(w%4)..+31, i.e. tile rows), then either
//                 - read-modify-write the bf16 output: old + acc, one rounding
//                   (dinp, and dweight when it is not split), or
//                 - store an fp32 partial tile, count arrivals, and let the last
//                   arriving split sum all partials in split order 0..S-1 and
//                   do the read-modify-write (deterministic: the order of the
//                   sum never depends on which split finished last).
//
// Every wait is bounded (global timer); a wait that gives up records the
// failure in the device status word, raises a CTA abort flag, and all roles
// unwind; in-flight copies and MMAs are waited for before the tensor memory
// is released.
#include "../../include/mmbwd.h"
#include "internal.h"
#include "ptx.cuh"

#include <cstdio>
#include <cstdlib>
#include <mutex>

namespace mmbwd {

// Device status word: [0] error code (positive), [1] block, [2] wait site, [3] item.
__device__ unsigned int g_status[4];

namespace {

constexpr int A_BYTES = TC_BM * TC_BK * 2;      // 16 KB
constexpr int B_BYTES = TC_BN * TC_BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int BOX_BYTES = 64 * TC_BK * 2;       // 8 KB: 64 (MN) x 64 (K) bf16, MN-major
constexpr int ROW_BYTES = 128;                  // one swizzled 128-byte row
constexpr int NUM_BIAS_WARPS = 2;
constexpr int WARP_TMA = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_BIAS = 2;
constexpr int WARP_EPI = 4;
constexpr int NUM_EPI_THREADS = 128;
constexpr uint32_t TMEM_COLS = 2 * TC_BN;

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_BARS = TC_STAGES * STAGE_BYTES;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = TC_STAGES;
constexpr int BAR_TFULL = 2 * TC_STAGES;
constexpr int BAR_TEMPTY = 2 * TC_STAGES + 2;
constexpr int BAR_BIAS = 2 * TC_STAGES + 4;
constexpr int BAR_TEARDOWN = 2 * TC_STAGES + 6;
constexpr int N_BARS = 2 * TC_STAGES + 7;
constexpr int OFF_MISC = OFF_BARS + N_BARS * 8;  // [0] tmem base, [1] abort flag, [2] broadcast
constexpr int OFF_BIAS = (OFF_MISC + 16 + 127) & ~127;
constexpr int SMEM_USED = OFF_BIAS + 2 * TC_BM * 4;
constexpr int SMEM_TOTAL = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory budget");

constexpr uint32_t IDESC_DINP = ptx::idesc_bf16_f32(TC_BM, TC_BN, /*A MN*/ 0, /*B MN*/ 1);
constexpr uint32_t IDESC_DW = ptx::idesc_bf16_f32(TC_BM, TC_BN, /*A MN*/ 1, /*B MN*/ 1);

constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s per wait

__device__ void record_failure(int site, int item) {
    if (atomicCAS(&g_status[0], 0u, static_cast<unsigned>(-MMBWD_ERR_DEVICE_TIMEOUT)) == 0u) {
        g_status[1] = blockIdx.x;
        g_status[2] = static_cast<unsigned>(site);
        g_status[3] = static_cast<unsigned>(item);
        __threadfence();
    }
}

struct Waiter {
    volatile uint32_t* abort;
    unsigned long long timeout_ns;

    // Bounded wait for the phase of `bar` with parity `parity`. Returns false
    // on timeout (recorded) or when another warp of the CTA has aborted.
    __device__ bool wait(uint32_t bar, uint32_t parity, int site, int item) const {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer();
        for (uint32_t i = 1;; ++i) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if ((i & 31u) == 0) {
                if (*abort) return false;
                if (ptx::globaltimer() - t0 > timeout_ns) {
                    *abort = 1u;
                    record_failure(site, item);
                    return false;
                }
            }
        }
    }

    // Teardown wait: ignores the abort flag (copies and MMAs already in flight
    // must land before the CTA exits), still bounded.
    __device__ bool wait_teardown(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = ptx::globaltimer();
        for (uint32_t i = 0;; ++i) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if ((i & 31u) == 31u && ptx::globaltimer() - t0 > timeout_ns) {
                *abort = 1u;
                record_failure(SITE_TEARDOWN, -1);
                return false;
            }
        }
    }

    // All 32 lanes wait; the warp agrees on one outcome.
    __device__ bool wait_warp(uint32_t bar, uint32_t parity, int site, int item) const {
        const bool ok = wait(bar, parity, site, item);
        return __all_sync(0xffffffffu, ok);
    }
};

struct Item {
    int is_dw;
    int m_tile, n_tile;
    int split;
    int kb0, kb1;  // k-block range [kb0, kb1)
    int tile;      // dweight tile index (m_tile * tiles_n + n_tile)
};

__device__ __forceinline__ Item decode_item(const TcParams& p, int w) {
    Item it;
    const int first_n = p.dw_first ? p.n_dw_items : p.n_dinp_items;
    const bool in_first = w < first_n;
    const int local = in_first ? w : w - first_n;
    it.is_dw = (in_first == (p.dw_first != 0)) ? 1 : 0;
    it.n_tile = local % p.tiles_n;
    const int rest = local / p.tiles_n;
    if (it.is_dw) {
        it.m_tile = rest % p.dw_tiles_m;
        it.split = rest / p.dw_tiles_m;
        it.kb0 = it.split * p.kb_per_split;
        it.kb1 = min(it.kb0 + p.kb_per_split, p.dw_kb);
        it.tile = it.m_tile * p.tiles_n + it.n_tile;
    } else {
        it.m_tile = rest;
        it.split = 0;
        it.kb0 = 0;
        it.kb1 = p.dinp_kb;
        it.tile = 0;
    }
    return it;
}

// Item processed by this CTA in round `round` (>= n_items: none).
__device__ __forceinline__ int item_at(const TcParams& p, int round) {
    const int G = static_cast<int>(gridDim.x);
    const int b = (p.snake && (round & 1)) ? (G - 1 - static_cast<int>(blockIdx.x))
                                           : static_cast<int>(blockIdx.x);
    return round * G + b;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// (old bf16 pair) + (a, b) in fp32, rounded once to a bf16 pair (RNE).
__device__ __forceinline__ uint32_t add_round_pair(uint32_t old, float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(bf_lo(old) + a, bf_hi(old) + b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 add_round8(uint4 old, const float (&s)[8]) {
    uint4 r;
    r.x = add_round_pair(old.x, s[0], s[1]);
    r.y = add_round_pair(old.y, s[2], s[3]);
    r.z = add_round_pair(old.z, s[4], s[5]);
    r.w = add_round_pair(old.w, s[6], s[7]);
    return r;
}

// Old values of one tile row: 32 vectors of 8 bf16 (256 columns). Vectors
// outside the tensor are not read.
__device__ __forceinline__ void load_row(uint4 (&old)[TC_BN / 8], const __nv_bfloat16* drow,
                                         bool row_ok, int ncols) {
#pragma unroll
    for (int v = 0; v < TC_BN / 8; ++v) {
        old[v] = (row_ok && v * 8 < ncols) ? *reinterpret_cast<const uint4*>(drow + v * 8)
                                           : make_uint4(0u, 0u, 0u, 0u);
    }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_mmbwd_kernel(const __grid_constant__ CUtensorMap tm_dout_k,   // dout, A of dinp (K-major)
                    const __grid_constant__ CUtensorMap tm_weight,   // weight, B of dinp (MN-major)
                    const __grid_constant__ CUtensorMap tm_dout_mn,  // dout, A of dweight (MN-major)
                    const __grid_constant__ CUtensorMap tm_inp,      // inp, B of dweight (MN-major)
                    const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    const uint32_t bars = base + OFF_BARS;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
    float* bias_smem = reinterpret_cast<float*>(smem + OFF_BIAS);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const bool bias_on = p.dbias != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            ptx::mbar_init(bars + 8u * (BAR_FULL + s), 1);
            ptx::mbar_init(bars + 8u * (BAR_EMPTY + s), 1u + (bias_on ? NUM_BIAS_WARPS : 0));
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bars + 8u * (BAR_TFULL + a), 1);
            ptx::mbar_init(bars + 8u * (BAR_TEMPTY + a), NUM_EPI_THREADS / 32);
            ptx::mbar_init(bars + 8u * (BAR_BIAS + a), NUM_BIAS_WARPS);
        }
        ptx::mbar_init(bars + 8u * BAR_TEARDOWN, 1);
        misc[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(base + OFF_MISC, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = misc[0];
    const Waiter wt{misc + 1, p.timeout_ns};

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_dout_k);
            ptx::prefetch_tmap(&tm_weight);
            ptx::prefetch_tmap(&tm_dout_mn);
            ptx::prefetch_tmap(&tm_inp);
            uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = item_at(p, r);
                if (w >= p.n_items) break;
                const Item it = decode_item(p, w);
                // Boxes that start inside the tensor; boxes wholly outside would
                // only feed accumulator rows/columns that are never stored.
                int nb = 0;
                for (int j = 0; j < TC_BN / 64; ++j) nb += (it.n_tile * TC_BN + j * 64 < p.C) ? 1 : 0;
                int na = 1;
                if (it.is_dw) na = (it.m_tile * TC_BM + 64 < p.OC) ? 2 : 1;
                const uint32_t bytes =
                    static_cast<uint32_t>((it.is_dw ? na * BOX_BYTES : A_BYTES) + nb * BOX_BYTES);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!wt.wait(bars + 8u * (BAR_EMPTY + stage), phase ^ 1u, SITE_PRODUCER_EMPTY, w)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * STAGE_BYTES;
                    const uint32_t sB = sA + A_BYTES;
                    const uint32_t fb = bars + 8u * (BAR_FULL + stage);
                    ptx::mbar_arrive_expect_tx(fb, bytes);
                    if (it.is_dw) {
                        for (int j = 0; j < na; ++j)
                            ptx::tma_load_2d(sA + j * BOX_BYTES, &tm_dout_mn, fb,
                                             it.m_tile * TC_BM + j * 64, kb * TC_BK);
                        for (int j = 0; j < nb; ++j)
                            ptx::tma_load_2d(sB + j * BOX_BYTES, &tm_inp, fb,
                                             it.n_tile * TC_BN + j * 64, kb * TC_BK);
                    } else {
                        ptx::tma_load_2d(sA, &tm_dout_k, fb, kb * TC_BK, it.m_tile * TC_BM);
                        for (int j = 0; j < nb; ++j)
                            ptx::tma_load_2d(sB + j * BOX_BYTES, &tm_weight, fb,
                                             it.n_tile * TC_BN + j * 64, kb * TC_BK);
                    }
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == TC_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Copies still in flight must land before shared memory goes away.
            for (int s = 0; s < TC_STAGES; ++s)
                if ((issued >> s) & 1u) wt.wait_teardown(bars + 8u * (BAR_FULL + s), (last_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = item_at(p, r);
                if (w >= p.n_items) break;
                const Item it = decode_item(p, w);
                if (!wt.wait(bars + 8u * (BAR_TEMPTY + acc), acc_phase ^ 1u, SITE_MMA_TMEM_EMPTY, w)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TC_BN;
                const uint32_t idesc = it.is_dw ? IDESC_DW : IDESC_DINP;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!wt.wait(bars + 8u * (BAR_FULL + stage), phase, SITE_MMA_FULL, w)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sA = base + stage * STAGE_BYTES;
                    const uint32_t sB = sA + A_BYTES;
#pragma unroll
                    for (int k = 0; k < TC_BK / 16; ++k) {
                        // K-major A: the 16-element K slice starts 32 bytes further
                        // into each swizzled 128-byte row; rows in 8-row groups of
                        // 1024 bytes. MN-major operands: 16 K rows of 128 bytes per
                        // slice (2048 bytes); 64-wide MN boxes 8 KB apart (leading
                        // offset), 8-row K groups 1024 bytes apart (stride offset).
                        const uint64_t adesc =
                            it.is_dw ? ptx::smem_desc_sw128(sA + k * 2048, BOX_BYTES, 1024)
                                     : ptx::smem_desc_sw128(sA + k * 32, 16, 1024);
                        const uint64_t bdesc = ptx::smem_desc_sw128(sB + k * 2048, BOX_BYTES, 1024);
                        ptx::mma_bf16(d_tmem, adesc, bdesc, idesc, (kb > it.kb0 || k > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(bars + 8u * (BAR_EMPTY + stage));
                    if (++stage == TC_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bars + 8u * (BAR_TFULL + acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued completes before tensor memory is freed.
            ptx::mma_commit(bars + 8u * BAR_TEARDOWN);
            wt.wait_teardown(bars + 8u * BAR_TEARDOWN, 0);
        }
        __syncwarp();
    } else if (warp < WARP_EPI) {
        // ------------------------------------------------------------ bias warps
        if (bias_on) {
            const int bw = warp - WARP_BIAS;  // which 64-wide box of the A tile
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            for (int r = 0;; ++r) {
                const int w = item_at(p, r);
                if (w >= p.n_items) break;
                const Item it = decode_item(p, w);
                const bool has_bias = it.is_dw && it.n_tile == 0;
                // Lockstep with the MMA issuer: the epilogue has finished with this
                // accumulator slot (and its bias slot) from two items ago.
                if (!wt.wait_warp(bars + 8u * (BAR_TEMPTY + acc), acc_phase ^ 1u, SITE_BIAS_TMEM_EMPTY, w))
                    break;
                float s[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = 0.f;
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!wt.wait_warp(bars + 8u * (BAR_FULL + stage), phase, SITE_BIAS_FULL, w)) {
                        ok = false;
                        break;
                    }
                    if (has_bias) {
                        // A tile of dweight: 64 BT rows x 64 OC columns per box, each
                        // row 128 bytes with its 16-byte chunks swizzled by (row & 7).
                        const uint8_t* box = smem + stage * STAGE_BYTES + bw * BOX_BYTES;
                        const int chunk = lane & 7;
#pragma unroll
                        for (int j = 0; j < TC_BK / 4; ++j) {
                            const int row = (lane >> 3) + 4 * j;
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                box + row * ROW_BYTES + ((chunk ^ (row & 7)) << 4));
                            s[0] += bf_lo(v.x);
                            s[1] += bf_hi(v.x);
                            s[2] += bf_lo(v.y);
                            s[3] += bf_hi(v.y);
                            s[4] += bf_lo(v.z);
                            s[5] += bf_hi(v.z);
                            s[6] += bf_lo(v.w);
                            s[7] += bf_hi(v.w);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bars + 8u * (BAR_EMPTY + stage));
                    if (++stage == TC_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (has_bias) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        s[e] += __shfl_xor_sync(0xffffffffu, s[e], 8);
                        s[e] += __shfl_xor_sync(0xffffffffu, s[e], 16);
                    }
                    if (lane < 8) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) bias_smem[acc * TC_BM + bw * 64 + lane * 8 + e] = s[e];
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bars + 8u * (BAR_BIAS + acc));
                }
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;         // TMEM lane quadrant this warp may read
        const int rit = q * 32 + lane;  // tile row owned by this thread
        uint32_t acc = 0, acc_phase = 0;
        uint32_t bias_parity[2] = {0u, 0u};
        for (int r = 0;; ++r) {
            const int w = item_at(p, r);
            if (w >= p.n_items) break;
            const Item it = decode_item(p, w);
            const bool has_bias = bias_on && it.is_dw && it.n_tile == 0;
            const bool split_mode = it.is_dw && p.splits > 1;
            const int64_t rows_total = it.is_dw ? p.OC : p.BT;
            const int64_t row = static_cast<int64_t>(it.m_tile) * TC_BM + rit;
            const bool row_ok = row < rows_total;
            const int col0 = it.n_tile * TC_BN;
            const int ncols = static_cast<int>(min(static_cast<int64_t>(TC_BN), p.C - col0));
            __nv_bfloat16* D = it.is_dw ? p.dweight : p.dinp;
            __nv_bfloat16* drow = D + (row_ok ? row : 0) * p.C + col0;

            uint4 old[TC_BN / 8];
            if (!split_mode) load_row(old, drow, row_ok, ncols);  // in flight during the main loop

            bool ok = wt.wait_warp(bars + 8u * (BAR_TFULL + acc), acc_phase, SITE_EPI_TMEM_FULL, w);
            if (!ptx::named_bar_and(1, NUM_EPI_THREADS, ok)) break;
            ptx::tc_fence_after();
            float bias_val = 0.f;
            if (has_bias) {
                ok = wt.wait_warp(bars + 8u * (BAR_BIAS + acc), bias_parity[acc], SITE_EPI_BIAS_FULL, w);
                bias_parity[acc] ^= 1u;
                if (!ptx::named_bar_and(1, NUM_EPI_THREADS, ok)) break;
                bias_val = bias_smem[acc * TC_BM + rit];
            }
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TC_BN;

            if (!split_mode) {
#pragma unroll
                for (int c = 0; c < TC_BN / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c * 32, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int vi = c * 4 + j;
                        if (row_ok && vi * 8 < ncols) {
                            float s[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) s[e] = __uint_as_float(v[j * 8 + e]);
                            *reinterpret_cast<uint4*>(drow + vi * 8) = add_round8(old[vi], s);
                        }
                    }
                }
                if (has_bias && row_ok) p.dbias[row] = __float2bfloat16_rn(bias_val);
            } else {
                // Partial tile, laid out [column quad][row][4] so that a warp's
                // 16-byte stores are contiguous.
                float* part = p.partials +
                              (static_cast<size_t>(it.tile) * p.splits + it.split) * (TC_BM * TC_BN);
#pragma unroll
                for (int c = 0; c < TC_BN / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c * 32, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int qd = c * 8 + j;
                        *reinterpret_cast<float4*>(part + (static_cast<size_t>(qd) * TC_BM + rit) * 4) =
                            make_float4(__uint_as_float(v[j * 4 + 0]), __uint_as_float(v[j * 4 + 1]),
                                        __uint_as_float(v[j * 4 + 2]), __uint_as_float(v[j * 4 + 3]));
                    }
                }
                if (has_bias)
                    p.bias_partials[(static_cast<size_t>(it.m_tile) * p.splits + it.split) * TC_BM + rit] =
                        bias_val;
                __threadfence();
                ptx::named_bar_sync(1, NUM_EPI_THREADS);
                if (threadIdx.x == WARP_EPI * 32) misc[2] = static_cast<uint32_t>(atomicAdd(&p.counters[it.tile], 1));
                ptx::named_bar_sync(1, NUM_EPI_THREADS);
                const bool last = misc[2] == static_cast<uint32_t>(p.splits - 1);
                if (last) {
                    __threadfence();
#pragma unroll 1
                    for (int c = 0; c < TC_BN / 32; ++c) {
                        uint4 oldc[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int vi = c * 4 + j;
                            oldc[j] = (row_ok && vi * 8 < ncols) ? *reinterpret_cast<const uint4*>(drow + vi * 8)
                                                                 : make_uint4(0u, 0u, 0u, 0u);
                        }
                        uint32_t v[32];
                        ptx::tmem_ld32(tbase + c * 32, v);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int vi = c * 4 + j;
                            float s[8];
                            for (int sp = 0; sp < p.splits; ++sp) {
                                float f[8];
                                if (sp == it.split) {
#pragma unroll
                                    for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[j * 8 + e]);
                                } else {
                                    const float* ps = p.partials +
                                                      (static_cast<size_t>(it.tile) * p.splits + sp) * (TC_BM * TC_BN);
                                    const float4 a = __ldcg(reinterpret_cast<const float4*>(
                                        ps + (static_cast<size_t>(2 * vi) * TC_BM + rit) * 4));
                                    const float4 b = __ldcg(reinterpret_cast<const float4*>(
                                        ps + (static_cast<size_t>(2 * vi + 1) * TC_BM + rit) * 4));
                                    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                                    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
                                }
#pragma unroll
                                for (int e = 0; e < 8; ++e) s[e] = (sp == 0) ? f[e] : s[e] + f[e];
                            }
                            if (row_ok && vi * 8 < ncols)
                                *reinterpret_cast<uint4*>(drow + vi * 8) = add_round8(oldc[j], s);
                        }
                    }
                    if (has_bias) {
                        float b = 0.f;
                        for (int sp = 0; sp < p.splits; ++sp) {
                            const float f = (sp == it.split)
                                                ? bias_val
                                                : __ldcg(p.bias_partials +
                                                         (static_cast<size_t>(it.m_tile) * p.splits + sp) * TC_BM + rit);
                            b = (sp == 0) ? f : b + f;
                        }
                        if (row_ok) p.dbias[row] = __float2bfloat16_rn(b);
                    }
                    // Every split has arrived: reset the counter for the next call.
                    if (threadIdx.x == WARP_EPI * 32) p.counters[it.tile] = 0;
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + 8u * (BAR_TEMPTY + acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must give up and report.
        const Waiter wt{&abort_flag, timeout_ns};
        wt.wait(ptx::smem_u32(&bar), 0u, SITE_SELFTEST, 0);
    }
}

int ceil_div_i(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

long env_long(const char* name, long dflt) {
    const char* s = std::getenv(name);
    if (!s || !*s) return dflt;
    char* end = nullptr;
    const long v = std::strtol(s, &end, 10);
    return (end && *end == '\0') ? v : dflt;
}

// Makespan of the static schedule, in units of one k-block of MMA work.
double schedule_cost(const TcPlan& pl, int grid) {
    const double item_overhead = 2.0;   // prologue/epilogue not hidden by the pipeline
    const double split_overhead = 2.0;  // partial-tile store and the fixed-order sum
    static thread_local double load[4096];
    for (int b = 0; b < grid; ++b) load[b] = 0.0;
    for (int r = 0;; ++r) {
        bool any = false;
        for (int b = 0; b < grid; ++b) {
            const int bb = (pl.snake && (r & 1)) ? grid - 1 - b : b;
            const int w = r * grid + bb;
            if (w >= pl.n_items) continue;
            any = true;
            const int first_n = pl.dw_first ? pl.n_dw_items : pl.n_dinp_items;
            const bool in_first = w < first_n;
            const bool is_dw = in_first == (pl.dw_first != 0);
            double c;
            if (is_dw) {
                const int local = in_first ? w : w - first_n;
                const int split = local / pl.tiles_n / pl.dw_tiles_m;
                const int kb0 = split * pl.kb_per_split;
                const int kb1 = std::min(kb0 + pl.kb_per_split, pl.dw_kb);
                c = (kb1 - kb0) + item_overhead + (pl.splits > 1 ? split_overhead : 0.0);
            } else {
                c = pl.dinp_kb + item_overhead;
            }
            load[b] += c;
        }
        if (!any) break;
    }
    double m = 0.0;
    for (int b = 0; b < grid; ++b) m = std::max(m, load[b]);
    return m;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

std::mutex g_attr_mutex;
bool g_attr_set[64];

}  // namespace

size_t tc_smem_bytes() { return SMEM_TOTAL; }

TcPlan tc_make_plan(int64_t BT, int64_t C, int64_t OC, int num_sms) {
    TcPlan pl{};
    pl.tiles_n = ceil_div_i(C, TC_BN);
    pl.dinp_tiles_m = ceil_div_i(BT, TC_BM);
    pl.dw_tiles_m = ceil_div_i(OC, TC_BM);
    pl.dinp_kb = ceil_div_i(OC, TC_BK);
    pl.dw_kb = ceil_div_i(BT, TC_BK);
    pl.n_dinp_items = pl.dinp_tiles_m * pl.tiles_n;
    const int dw_tiles = pl.dw_tiles_m * pl.tiles_n;
    num_sms = std::max(1, std::min(num_sms, 4096));

    const long force_splits = env_long("MMBWD_SPLITK", 0);
    const long force_grid = env_long("MMBWD_GRID", 0);
    const int max_splits = std::max(1, std::min(pl.dw_kb, 16));
    double best = 1e300;
    TcPlan best_pl = pl;
    for (int S = 1; S <= max_splits; ++S) {
        if (force_splits > 0 && S != std::min<long>(force_splits, max_splits)) continue;
        const int kps = ceil_div_i(pl.dw_kb, S);
        if (ceil_div_i(pl.dw_kb, kps) != S) continue;  // would leave an empty split
        for (int dw_first = 1; dw_first >= 0; --dw_first) {
            for (int snake = 0; snake <= 1; ++snake) {
                TcPlan c = pl;
                c.splits = S;
                c.kb_per_split = kps;
                c.n_dw_items = dw_tiles * S;
                c.n_items = c.n_dw_items + c.n_dinp_items;
                c.dw_first = dw_first;
                c.snake = snake;
                c.grid = std::max(1, std::min(c.n_items, num_sms));
                if (force_grid > 0) c.grid = static_cast<int>(std::min<long>(force_grid, c.grid));
                const double cost = schedule_cost(c, c.grid) * (1.0 + 0.01 * (S - 1));
                if (cost < best - 1e-9) {
                    best = cost;
                    best_pl = c;
                }
            }
        }
    }
    pl = best_pl;
    if (pl.splits > 1) {
        pl.ws_partials_bytes = align256(static_cast<size_t>(dw_tiles) * pl.splits * TC_BM * TC_BN * 4);
        pl.ws_bias_bytes = align256(static_cast<size_t>(pl.dw_tiles_m) * pl.splits * TC_BM * 4);
        pl.ws_counter_bytes = align256(static_cast<size_t>(dw_tiles) * 4);
    }
    return pl;
}

cudaError_t tc_launch(const TcPlan& plan, void* dinp, void* dweight, void* dbias, const void* dout,
                      const void* inp, const void* weight, int64_t BT, int64_t C, int64_t OC, void* ws,
                      cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> g(g_attr_mutex);
        if (dev < 0 || dev >= 64 || !g_attr_set[dev]) {
            e = cudaFuncSetAttribute(tc_mmbwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) g_attr_set[dev] = true;
        }
    }
    EncodeTiledFn encode = get_encode_tiled();
    if (!encode) return cudaErrorNotSupported;

    CUtensorMap maps[4];
    struct MapSpec {
        const void* base;
        uint64_t inner, outer;
        uint32_t box_inner, box_outer;
    } specs[4] = {
        {dout, static_cast<uint64_t>(OC), static_cast<uint64_t>(BT), TC_BK, TC_BM},  // dout, K-major A
        {weight, static_cast<uint64_t>(C), static_cast<uint64_t>(OC), 64, TC_BK},    // weight, MN-major B
        {dout, static_cast<uint64_t>(OC), static_cast<uint64_t>(BT), 64, TC_BK},     // dout, MN-major A
        {inp, static_cast<uint64_t>(C), static_cast<uint64_t>(BT), 64, TC_BK},       // inp, MN-major B
    };
    for (int i = 0; i < 4; ++i) {
        const cuuint64_t dims[2] = {specs[i].inner, specs[i].outer};
        const cuuint64_t strides[1] = {specs[i].inner * 2};
        const cuuint32_t box[2] = {specs[i].box_inner, specs[i].box_outer};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = encode(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(specs[i].base),
                                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    TcParams p{};
    p.BT = BT;
    p.C = C;
    p.OC = OC;
    p.dinp = static_cast<__nv_bfloat16*>(dinp);
    p.dweight = static_cast<__nv_bfloat16*>(dweight);
    p.dbias = static_cast<__nv_bfloat16*>(dbias);
    p.tiles_n = plan.tiles_n;
    p.dinp_tiles_m = plan.dinp_tiles_m;
    p.dw_tiles_m = plan.dw_tiles_m;
    p.dinp_kb = plan.dinp_kb;
    p.dw_kb = plan.dw_kb;
    p.splits = plan.splits;
    p.kb_per_split = plan.kb_per_split;
    p.n_dw_items = plan.n_dw_items;
    p.n_dinp_items = plan.n_dinp_items;
    p.n_items = plan.n_items;
    p.dw_first = plan.dw_first;
    p.snake = plan.snake;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.partials = plan.splits > 1 ? reinterpret_cast<float*>(w) : nullptr;
    p.bias_partials = plan.splits > 1 ? reinterpret_cast<float*>(w + plan.ws_partials_bytes) : nullptr;
    p.counters = plan.splits > 1 ? reinterpret_cast<int*>(w + plan.ws_partials_bytes + plan.ws_bias_bytes) : nullptr;
    p.timeout_ns = static_cast<unsigned long long>(env_long("MMBWD_WAIT_TIMEOUT_NS", static_cast<long>(DEFAULT_TIMEOUT_NS)));

    tc_mmbwd_kernel<<<plan.grid, TC_THREADS, SMEM_TOTAL, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
    return cudaGetLastError();
}

cudaError_t tc_read_status(int* code, int* info3, bool reset) {
    unsigned int h[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(h, g_status, sizeof(h));
    if (e != cudaSuccess) return e;
    *code = h[0] ? -static_cast<int>(h[0]) : MMBWD_OK;
    if (info3) {
        info3[0] = static_cast<int>(h[1]);
        info3[1] = static_cast<int>(h[2]);
        info3[2] = static_cast<int>(h[3]);
    }
    if (reset) {
        const unsigned int z[4] = {0, 0, 0, 0};
        e = cudaMemcpyToSymbol(g_status, z, sizeof(z));
    }
    return e;
}

cudaError_t tc_selftest_wait(unsigned long long timeout_ns) {
    selftest_wait_kernel<<<1, 32>>>(timeout_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaDeviceSynchronize();
}

}  // namespace mmbwd

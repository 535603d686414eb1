// bf16 linear-layer backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent kernel computes both products of matmul_backward (llm.c
// dev/cuda/matmul_backward.cu, matmul_backward_cpu / matmul_backward1):
//
//   dinp    (BT x C) += dout (BT x OC) . weight (OC x C)     "NN": A K-major, B MN-major
//   dweight (OC x C) += dout^T (OC x BT) . inp (BT x C)      "TN": A MN-major, B MN-major
//   dbias   (OC)      = column sums of dout                  fused into the dweight pass
//
// CTA pairs. The grid is made of clusters of two CTAs on neighbouring SMs.
// A pair computes one 256 x 256 output tile with pair MMAs (tcgen05.mma
// cta_group::2, M = 256, N = 256, K = 16): CTA r of the pair stages rows
// [128 r, 128 r + 128) of A and columns [128 r, 128 r + 128) of B, and its
// tensor memory receives rows [128 r, 128 r + 128) of the accumulator. Each SM
// thus moves 32 KB per 64-deep K step instead of 48 KB for a single-CTA
// 128 x 256 tile, which is what lets the load pipeline keep the tensor core fed.
//
// Work list: every 256 x 256 tile of dinp is one item; every 256 x 256 tile of
// dweight is cut into `splits` items along its long BT reduction. Each pair
// walks a static, shape-determined sequence of items.
//
// Warp roles (384 threads per CTA; 256 in MODE 2):
//   warp 0      TMA producer (both CTAs): a 6-stage ring of (A 16 KB, B 16 KB)
//               tiles in 128-byte-swizzled shared memory; completion lands on
//               the CTA's own "full" barrier.
//   warp 1      even CTA: MMA issuer (one thread) into one of two 128 x 256 fp32
//               accumulators per CTA (512 tensor-memory columns), so the epilogue
//               of one item overlaps the main loop of the next; each commit
//               arrives on both CTAs' barriers.
//               odd CTA: forwards each stage's "full" to the even CTA's barrier.
//   warps 2-3   bias: on dweight items of the first column tile, sum the CTA's
//               dout tile of every stage over its BT rows (the A operand already
//               in shared memory) and reduce across lanes with shuffles.
//   warps 4-11  epilogue (both CTAs; warps 4-7 in MODE 2): tcgen05.ld the
//               accumulator (warp w reads tensor-memory lanes 32*(w%4)..+31, i.e.
//               tile rows; the two warps of a lane quadrant take every other
//               32-column chunk) in 32 x 32 chunks that travel between global and
//               shared memory by TMA, then either
//                 - read-modify-write the bf16 output: old + acc, one rounding
//                   (dinp, and dweight when it is not split), each warp's old
//                   values loaded two of its chunks ahead, or
//                 - store the fp32 partial tile of this split (dweight split
//                   along BT); a second kernel then sums the partials of every
//                   tile in split order 0..S-1 and does the read-modify-write, so
//                   the sum never depends on which split finished first.
//
// Every wait is bounded (global timer); a wait that gives up records the
// failure in the device status word, raises a CTA abort flag, and all roles
// unwind; copies and MMAs in flight are waited for before tensor memory is
// released.
#include "../../include/mmbwd.h"
#include "internal.h"
#include "ptx.cuh"
#include "sr.cuh"

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace mmbwd {

// Device status word: [0] error code (positive), [1] block, [2] wait site, [3] item.
__device__ unsigned int g_status[4];

namespace {

constexpr int A_BYTES = TC_BM * TC_BK * 2;            // 16 KB: this CTA's 128 rows of A
constexpr int B_BYTES = (TC_BN / 2) * TC_BK * 2;      // 16 KB: room for this CTA's (up to) 128 columns of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // 32 KB
constexpr int BOX_BYTES = 64 * TC_BK * 2;             // 8 KB: 64 (MN) x 64 (K) bf16, MN-major
constexpr int ROW_BYTES = 128;                        // one swizzled 128-byte row
constexpr int NUM_BIAS_WARPS = 2;
constexpr int WARP_TMA = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_BIAS = 2;
constexpr int WARP_EPI = 4;
constexpr uint32_t TMEM_COLS = 2 * TC_BN;

constexpr int STG_STRIDE = 36;  // floats per staged row: 16-byte aligned, conflict-free
constexpr int STG_WARP_BYTES = 32 * STG_STRIDE * 4;
// Epilogue chunks: 32 rows x 32 columns of the output, one row per thread.
// bf16: 2 KB, rows of 64 bytes, 64-byte swizzle (read-modify-write and forward
// stores). fp32 split partials: 4 KB, rows of 128 bytes, 128-byte swizzle.
constexpr int OLD_CHUNK_BYTES = 32 * 32 * 2;
constexpr int PART_CHUNK_BYTES = 32 * 32 * 4;

// Shared memory map (offsets from a 1024-byte aligned base), per kernel mode:
// the TMA stage ring, the barriers, then one region per epilogue warp. The
// bf16 modes keep six 32 KB stages and give each of their eight epilogue warps
// two chunk buffers (4 KB): its first two chunks of old values are requested at
// the start of an item, each later one as soon as the store of the chunk two
// before has read its buffer. A sixth stage (a stage's round trip is about
// 2 us, five covered it only just) is worth more than a whole tile of old values
// in flight: with five stages and eight buffers a quadrant every bf16 backward
// plan ran 1-4 % slower. MODE 2 keeps three 64 KB stages
// and the fp32 staging rows, and a second barrier per stage: the raw fp32
// operands land on the first (TMA), the split planes are signalled on the
// second (the split warps of both CTAs, on the even CTA's copy).
template <int MODE>
struct Smem {
    static constexpr bool X3 = MODE == 2;
    static constexpr int STAGES = X3 ? TC_STAGES_X3 : TC_STAGES;
    static constexpr int STG_BYTES = X3 ? 2 * STAGE_BYTES : STAGE_BYTES;
    // Epilogue warps: in the bf16 modes two per tensor-memory lane quadrant, each
    // taking every other 32-column chunk of the quadrant's rows with two chunk
    // buffers of its own; MODE 2 keeps one per quadrant (its staging rows fill
    // the region of one warp of four).
    static constexpr int EPI_WARPS = X3 ? 4 : 8;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int THREADS = 32 * WARP_EPI + EPI_THREADS;
    static constexpr int OLD_SLOTS = X3 ? 4 : 2;  // bf16 chunk buffers per epilogue warp
    static constexpr int PART_SLOTS = 1;  // fp32 partial chunk buffers (same memory)
    static constexpr int OFF_BARS = STAGES * STG_BYTES;
    static constexpr int BAR_FULL = 0;                   // [stages] TMA landed (even CTA: and the peer's too)
    static constexpr int BAR_EMPTY = STAGES;             // [stages] stage may be refilled
    static constexpr int BAR_TFULL = 2 * STAGES;         // [2] accumulator ready
    static constexpr int BAR_TEMPTY = 2 * STAGES + 2;    // [2] accumulator drained by both CTAs (even CTA)
    static constexpr int BAR_TEARDOWN = 2 * STAGES + 4;
    static constexpr int BAR_OLD = 2 * STAGES + 5;       // [epilogue warp][slot] old chunk landed
    static constexpr int BAR_CONV = BAR_OLD + EPI_WARPS * OLD_SLOTS;  // MODE 2: [stages] split planes ready
    static constexpr int N_BARS = BAR_CONV + (X3 ? STAGES : 0);
    static constexpr int OFF_MISC = OFF_BARS + N_BARS * 8;  // [0] tmem base, [1] abort flag
    static constexpr int OFF_STAGE = (OFF_MISC + 16 + 1023) & ~1023;
    static constexpr int OLD_WARP_BYTES = OLD_SLOTS * OLD_CHUNK_BYTES;
    static constexpr int WARP_REGION =
        X3 ? (STG_WARP_BYTES > OLD_WARP_BYTES ? STG_WARP_BYTES : OLD_WARP_BYTES) : OLD_WARP_BYTES;
    // ones tile of the dbias-by-MMA variant: 8 rows (this CTA's half of N = 16)
    // of 64 bf16 ones, one 128-byte-swizzled 1 KB atom
    static constexpr int OFF_ONES = OFF_STAGE + EPI_WARPS * WARP_REGION;
    static constexpr int SMEM_TOTAL = OFF_ONES + 1024 + 1024;  // + slack for aligning the base
    static_assert(X3 || PART_SLOTS * PART_CHUNK_BYTES <= WARP_REGION, "partial chunks fit the warp region");
    static_assert(EPI_WARPS % 4 == 0 && (!X3 || EPI_WARPS == 4), "whole quadrants; MODE 2 one warp each");
    static_assert(WARP_REGION % 1024 == 0, "chunk buffers stay 1024-byte aligned (128-byte swizzle)");
    static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory budget");
};
constexpr int SMEM_TOTAL = Smem<0>::SMEM_TOTAL > Smem<2>::SMEM_TOTAL ? Smem<0>::SMEM_TOTAL : Smem<2>::SMEM_TOTAL;

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
    // CLUSTER: acquire at cluster scope (a barrier the other CTA of the pair
    // arrives on).
    template <bool CLUSTER = false>
    __device__ bool wait(uint32_t bar, uint32_t parity, int site, int item) const {
        auto probe = [&]() { return CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
        if (probe()) return true;
        const uint64_t t0 = ptx::globaltimer();
        for (uint32_t i = 1;; ++i) {
            if (probe()) return true;
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
    int pm;      // row tile of the pair (256 rows)
    int n_tile;  // column tile (bn columns)
    int bn;      // tile width: 128 or 256
    int split;
    int kb0, kb1;  // k-block range [kb0, kb1)
};

__device__ __forceinline__ Item decode_item(const TcParams& p, int w) {
    Item it;
    it.is_dw = w < p.n_dw_items ? 1 : 0;
    const int local = it.is_dw ? w : w - p.n_dw_items;
    const int tiles_n = it.is_dw ? p.dw_tiles_n : p.dinp_tiles_n;
    it.bn = it.is_dw ? p.dw_bn : p.dinp_bn;
    it.n_tile = local % tiles_n;
    const int rest = local / tiles_n;
    if (it.is_dw) {
        it.pm = rest % p.dw_tiles_m;
        it.split = rest / p.dw_tiles_m;
        it.kb0 = it.split * p.kb_per_split;
        it.kb1 = min(it.kb0 + p.kb_per_split, p.dw_kb);
    } else {
        it.pm = rest;
        it.split = 0;
        it.kb0 = 0;
        it.kb1 = p.dinp_kb;
    }
    return it;
}

// Item processed by this CTA pair in round `round` (>= n_items: none).
__device__ __forceinline__ int item_at(const TcParams& p, const TcSchedule& sch, int round) {
    const int c = static_cast<int>(blockIdx.x) / 2;
    if (p.table) {
        const int idx = sch.start[c] + round;
        return idx < sch.start[c + 1] ? static_cast<int>(sch.items[idx]) : p.n_items;
    }
    return round * (static_cast<int>(gridDim.x) / 2) + c;
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

// Two elements (old bf16 pair) + (a, b), stochastically rounded (sr.cuh) with
// the 16-bit thresholds in the low and high halves of r2. Branch-free: an
// infinity plus any threshold stays an infinity after the low half is
// dropped, and a NaN takes threshold 0 (it is truncated, as sr.cuh states).
__device__ __forceinline__ uint32_t add_sr_pair(uint32_t old2, float a, float b, uint32_t r2) {
    const float x0 = bf_lo(old2) + a, x1 = bf_hi(old2) + b;
    const uint32_t r0 = (x0 == x0) ? (r2 & 0xFFFFu) : 0u, r1 = (x1 == x1) ? (r2 >> 16) : 0u;
    return __byte_perm(__float_as_uint(x0) + r0, __float_as_uint(x1) + r1, 0x7632);
}

// (old bf16 x 8) + s, stochastically rounded; w0 and w1 are the generator
// words of elements e0..e0+3 and e0+4..e0+7 (e0 a multiple of 4).
__device__ __forceinline__ uint4 add_sr8(uint4 old, const float (&s)[8], uint64_t w0, uint64_t w1) {
    return make_uint4(add_sr_pair(old.x, s[0], s[1], static_cast<uint32_t>(w0)),
                      add_sr_pair(old.y, s[2], s[3], static_cast<uint32_t>(w0 >> 32)),
                      add_sr_pair(old.z, s[4], s[5], static_cast<uint32_t>(w1)),
                      add_sr_pair(old.w, s[6], s[7], static_cast<uint32_t>(w1 >> 32)));
}

// fp32 x = hi + lo with hi its tf32 truncation (13 low mantissa bits cleared)
// and lo the exact remainder; the tensor core reads an fp32 operand as hi.
__device__ __forceinline__ float tf32_lo(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Split warp, K-major raw operand: the tile in `hi` (n16 granules of 16
// bytes, 128-byte swizzled rows; n16 a multiple of 256) is its own high
// plane; its low plane goes to the same offsets in `lo`. Eight granules a
// lane in flight (a warp reads 512 contiguous bytes per instruction).
__device__ __forceinline__ void x3_split_k(uint32_t hi, uint32_t lo, int n16, int lane) {
#pragma unroll 1
    for (int i0 = 0; i0 < n16; i0 += 256) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = ptx::lds128f(hi + 16u * static_cast<uint32_t>(i0 + 32 * u + lane));
#pragma unroll
        for (int u = 0; u < 8; ++u)
            ptx::sts128(lo + 16u * static_cast<uint32_t>(i0 + 32 * u + lane), tf32_lo(x[u].x), tf32_lo(x[u].y),
                        tf32_lo(x[u].z), tf32_lo(x[u].w));
    }
}

// Split warp, MN-major raw operand: nbox (1 or 2) boxes of 32 K rows x 64
// fp32 (256-byte rows, box j at j * 8 KB) in `lo`, transposed into both
// K-major planes: row j * 64 + m holds the 32 K values of column m of box j in
// 128 bytes, 16-byte granule g at g ^ (row & 7). Box j's raw bytes are exactly
// where its 64 rows of the low plane go, so a box is read whole (lane l takes
// columns l and l + 32: a warp reads 128 contiguous bytes per K row), the
// warp synchronises, and its rows are written (a quarter warp's eight rows
// hit eight distinct granule positions). With `sums`, sum[2 j + h] += the sum
// of row j * 64 + 32 h + lane's 32 K values (pairwise, in a fixed order).
__device__ __forceinline__ void x3_split_mn(uint32_t hi, uint32_t lo, int nbox, int lane, bool sums,
                                            float (&sum)[4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (j >= nbox) break;
        float v[2][32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                v[h][k] = ptx::lds32f(lo + static_cast<uint32_t>(j * BOX_BYTES + k * 256 + (32 * h + lane) * 4));
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t row = static_cast<uint32_t>(j * 64 + 32 * h + lane);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t off = row * 128u + ((static_cast<uint32_t>(g) ^ (row & 7u)) << 4);
                const float* x = &v[h][4 * g];
                ptx::sts128(hi + off, x[0], x[1], x[2], x[3]);
                ptx::sts128(lo + off, tf32_lo(x[0]), tf32_lo(x[1]), tf32_lo(x[2]), tf32_lo(x[3]));
            }
            if (sums) {
                float t[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) t[i] = v[h][2 * i] + v[h][2 * i + 1];
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int i = 0; i < w; ++i) t[i] = t[2 * i] + t[2 * i + 1];
                sum[2 * j + h] += t[0];
            }
        }
        __syncwarp();
    }
}

// MODE 0: the backward (dinp and dweight items). MODE 1: the forward
// (dinp-type items with a K-major B and an overwrite epilogue). MODE 2: fp32
// products D (M x N) += A (M x K) . B (N x K)^T from tf32 halves: the raw
// fp32 operands arrive by TMA (K-major into the high plane, or MN-major into
// the low plane as scratch), the two split warps of each CTA write both planes
// K-major -- the high part (the value itself: the tensor core reads an fp32
// operand as its tf32 truncation) and the low part (the exact remainder) --
// and each K step issues three tf32 MMAs, hi.hi + hi.lo + lo.hi; fp32
// read-modify-write epilogue. MODE 3: the backward with stochastic rounding of the bf16 outputs
// (seeded; sr.cuh). Four instantiations, so that none pays for the
// others' branches.
template <int MODE>
__global__ void __launch_bounds__(Smem<MODE>::THREADS, 1)
    tc_mmbwd_kernel(const __grid_constant__ CUtensorMap tm_dout_k,   // dout, A of dinp (K-major)
                    const __grid_constant__ CUtensorMap tm_weight,   // weight, B of dinp (MN-major)
                    const __grid_constant__ CUtensorMap tm_dout_mn,  // dout, A of dweight (MN-major)
                    const __grid_constant__ CUtensorMap tm_inp,      // inp, B of dweight (MN-major)
                    const __grid_constant__ CUtensorMap tm_dinp_out, // dinp, for L2 prefetch of old values
                    const __grid_constant__ CUtensorMap tm_dw_out,   // dweight, likewise
                    // Both 64-column halves of a B (or dweight A) operand in one request:
                    // backward, three-dimensional maps {64, rows, extent / 64} whose
                    // boxes {64, 64, 2} land as two consecutive 64 x 64 boxes; forward,
                    // weight rows in boxes of 128. Used where p.wide_maps has the bit.
                    const __grid_constant__ CUtensorMap tm_weight_w,
                    const __grid_constant__ CUtensorMap tm_dout_mn_w,
                    const __grid_constant__ CUtensorMap tm_inp_w,
                    // dinp and dweight in 32 x 32 boxes, 64-byte swizzle: the bf16
                    // read-modify-write of the backward (MODE 0 and 3)
                    const __grid_constant__ CUtensorMap tm_dinp_rmw,
                    const __grid_constant__ CUtensorMap tm_dw_rmw,
                    // fp32 partial tiles of a split dweight reduction, 32 x 32
                    // boxes, 128-byte swizzle (MODE 0 and 3 with splits > 1)
                    const __grid_constant__ CUtensorMap tm_part,
                    const TcParams p, const __grid_constant__ TcSchedule sch) {
    constexpr bool FWD = MODE == 1 || MODE == 2;  // dinp-type items only, K-major B
    constexpr bool X3 = MODE == 2;                // fp32 from three tf32 products
    constexpr bool SR = MODE == 3;                // stochastic rounding of the outputs
    // MODE 2 stages hold A hi | A lo | B hi | B lo (twice the bytes, half the
    // stages: the same shared memory) and 32 fp32 of K per k-block (128 bytes).
    using L = Smem<MODE>;
    constexpr int STAGES = L::STAGES;
    constexpr int STG_BYTES = L::STG_BYTES;
    constexpr int OLD_SLOTS = L::OLD_SLOTS;
    constexpr int BAR_FULL = L::BAR_FULL, BAR_EMPTY = L::BAR_EMPTY, BAR_TFULL = L::BAR_TFULL;
    constexpr int BAR_TEMPTY = L::BAR_TEMPTY, BAR_TEARDOWN = L::BAR_TEARDOWN, BAR_OLD = L::BAR_OLD;
    constexpr int KBLK = X3 ? TC_BK / 2 : TC_BK;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    const uint32_t bars = base + L::OFF_BARS;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_MISC);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const uint32_t rank = ptx::cluster_ctarank();  // within the CTA pair: 0 issues the pair MMAs
    const bool leader = rank == 0;
    const bool bias_on = p.dbias != nullptr;
    // Accumulator sets in tensor memory. For long reductions MODE 2 keeps two
    // accumulators per item side by side -- the hi.hi product, and the two
    // small correction products -- so a set is 2 x bn columns: two sets when
    // bn <= 128, else one (the epilogue then does not overlap the next item's
    // main loop).
    const bool corr = X3 && p.x3_corr;
    const uint32_t acc_cols = corr ? 2u * static_cast<uint32_t>(p.dinp_bn) : static_cast<uint32_t>(TC_BN);
    const int acc_sets = (corr && p.dinp_bn > 128) ? 1 : 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // MODE 2: this CTA's raw copies only (the split warps signal the MMA)
            ptx::mbar_init(bars + 8u * (BAR_FULL + s), leader && !X3 ? 2u : 1u);
            // refilled once the pair MMAs reading it have completed (one commit)
            // and this CTA's bias warps are done with it
            ptx::mbar_init(bars + 8u * (BAR_EMPTY + s), 1u + (!X3 && bias_on && !p.bias_mma ? NUM_BIAS_WARPS : 0));
            // MODE 2, even CTA: both split warps of both CTAs
            if constexpr (X3) ptx::mbar_init(bars + 8u * (L::BAR_CONV + s), 2u * NUM_BIAS_WARPS);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bars + 8u * (BAR_TFULL + a), 1);
            ptx::mbar_init(bars + 8u * (BAR_TEMPTY + a), 2 * L::EPI_WARPS);
        }
        ptx::mbar_init(bars + 8u * BAR_TEARDOWN, 1);
        for (int b = 0; b < L::EPI_WARPS * OLD_SLOTS; ++b) ptx::mbar_init(bars + 8u * (BAR_OLD + b), 1);
        misc[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        ptx::tmem_alloc_pair(base + L::OFF_MISC, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    if constexpr (!FWD && !X3) {
        if (p.bias_mma) {  // the ones tile (bf16 1.0 in every element, so any layout reads ones)
            reinterpret_cast<uint32_t*>(smem + L::OFF_ONES)[threadIdx.x] = 0x3F803F80u;
            ptx::fence_proxy_async_smem();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // both CTAs' barriers exist before any remote arrive or commit
    ptx::tc_fence_after();
    // Everything above overlaps the previous launch on the stream. Threads that
    // touch global memory wait for it to complete first: the epilogue warps
    // here, the producer only just ahead of its first load, so that its first
    // item's schedule entry, geometry and barrier steps (first-touch latencies
    // of about 2 us in all) also overlap the previous launch. The MMA and bias
    // warps read only shared and tensor memory.
    const bool defer_wait = warp < WARP_EPI;
    if (!defer_wait) ptx::grid_dependency_wait();
    const uint32_t tmem_base = misc[0];
    const Waiter wt{misc + 1, p.timeout_ns};

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_dout_k);
            ptx::prefetch_tmap(&tm_weight);
            ptx::prefetch_tmap(&tm_dout_mn);
            ptx::prefetch_tmap(&tm_inp);
            if (p.wide_maps & TC_WIDE_WEIGHT) ptx::prefetch_tmap(&tm_weight_w);
            if (p.wide_maps & TC_WIDE_DOUT_MN) ptx::prefetch_tmap(&tm_dout_mn_w);
            if (p.wide_maps & TC_WIDE_INP) ptx::prefetch_tmap(&tm_inp_w);
            if (X3 && p.n_dw_items > 0) {  // the dweight product's maps of a paired fp32 launch
                ptx::prefetch_tmap(&tm_weight_w);
                ptx::prefetch_tmap(&tm_dout_mn_w);
            }
            ptx::prefetch_tmap(&tm_dinp_out);
            ptx::prefetch_tmap(&tm_dw_out);
            uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
            bool ok = true, waited = false;
            for (int r = 0; ok; ++r) {
                const int w = item_at(p, sch, r);
                if (w >= p.n_items) break;
                const Item it = decode_item(p, w);
                // This CTA's rows of A and columns of B. Boxes wholly outside the
                // tensor are skipped: they would only feed accumulator rows or
                // columns that are never stored.
                const int row0 = it.pm * TC_PAIR_BM + static_cast<int>(rank) * TC_BM;
                const int half = it.bn / 2;  // columns of B staged by this CTA
                const int col0 = it.n_tile * it.bn + static_cast<int>(rank) * half;
                const int64_t n_extent = FWD ? p.n_dinp : p.C;  // N of this item's product
                int nb = 0;
                for (int j = 0; j < half / 64; ++j) nb += (col0 + j * 64 < n_extent) ? 1 : 0;
                // Output tile of this CTA, prefetched into L2 a few k-blocks before the
                // main loop ends so that the epilogue's read of the old values hits L2.
                const bool direct = X3 || (!(it.is_dw && p.splits > 1) && !FWD);  // forward: nothing to read back
                const int64_t out_rows = it.is_dw ? p.OC : p.BT;
                const int pf_kb = max(it.kb0, it.kb1 - 8);
                // A of a bf16 dweight item, or an MN-major fp32 A: 64-row boxes
                // (8 KB either way); every other A: one K-major 128-row tile
                const int sh = it.is_dw ? 2 : 0;
                const bool a_mn = X3 ? ((p.x3_mn >> sh) & 1) != 0 : it.is_dw != 0;
                const bool b_mn = X3 && ((p.x3_mn >> (sh + 1)) & 1) != 0;
                const int na = a_mn ? (row0 < out_rows ? 1 : 0) + (row0 + 64 < out_rows ? 1 : 0)
                                    : (row0 < out_rows ? 1 : 0);
                const uint32_t bytes = static_cast<uint32_t>((a_mn ? na * BOX_BYTES : na * A_BYTES) + nb * BOX_BYTES);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!wt.wait(bars + 8u * (BAR_EMPTY + stage), phase ^ 1u, SITE_PRODUCER_EMPTY, w)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * STG_BYTES;
                    const uint32_t sB = sA + (X3 ? 2 : 1) * A_BYTES;
                    const uint32_t fb = bars + 8u * (BAR_FULL + stage);
                    ptx::mbar_arrive_expect_tx(fb, bytes);
                    if (!waited) {  // the previous launch has completed before any load
                        ptx::grid_dependency_wait();
                        waited = true;
                    }
                    if (direct && kb == pf_kb && row0 < out_rows) {
                        for (int j = 0; j < it.bn / 128; ++j)
                            if (it.n_tile * it.bn + j * 128 < n_extent)
                                ptx::tma_prefetch_l2_2d(it.is_dw ? &tm_dw_out : &tm_dinp_out,
                                                        it.n_tile * it.bn + j * 128, row0);
                    }
                    if (X3) {
                        // Raw fp32: a K-major operand into its high plane, an
                        // MN-major one (64-wide boxes of 32 K rows) into its low
                        // plane, which the split warps read before writing it.
                        // Maps: A and B of dinp-type items 0 and 1, of the
                        // dweight items of a paired launch 6 and 7.
                        const void* ta = it.is_dw ? static_cast<const void*>(&tm_weight_w) : &tm_dout_k;
                        const void* tb = it.is_dw ? static_cast<const void*>(&tm_dout_mn_w) : &tm_weight;
                        if (a_mn) {
                            for (int j = 0; j < na; ++j)
                                ptx::tma_load_2d(sA + A_BYTES + j * BOX_BYTES, ta, fb, row0 + j * 64, kb * KBLK);
                        } else if (na) {
                            ptx::tma_load_2d(sA, ta, fb, kb * KBLK, row0);
                        }
                        for (int j = 0; j < nb; ++j) {
                            if (b_mn)
                                ptx::tma_load_2d(sB + B_BYTES + j * BOX_BYTES, tb, fb, col0 + j * 64, kb * KBLK);
                            else
                                ptx::tma_load_2d(sB + j * BOX_BYTES, tb, fb, kb * KBLK, col0 + j * 64);
                        }
                    } else if (it.is_dw) {
                        if (na == 2 && (p.wide_maps & TC_WIDE_DOUT_MN))
                            ptx::tma_load_3d(sA, &tm_dout_mn_w, fb, 0, kb * KBLK, row0 / 64);
                        else
                            for (int j = 0; j < na; ++j)
                                ptx::tma_load_2d(sA + j * BOX_BYTES, &tm_dout_mn, fb, row0 + j * 64, kb * KBLK);
                    } else if (na) {
                        ptx::tma_load_2d(sA, &tm_dout_k, fb, kb * KBLK, row0);
                    }
                    const void* tmB = it.is_dw ? static_cast<const void*>(&tm_inp) : static_cast<const void*>(&tm_weight);
                    const void* tmBw =
                        it.is_dw ? static_cast<const void*>(&tm_inp_w) : static_cast<const void*>(&tm_weight_w);
                    const bool b_wide = nb == 2 && (p.wide_maps & (it.is_dw ? TC_WIDE_INP : TC_WIDE_WEIGHT));
                    // B boxes: 64 columns x 64 k, MN-major (backward) or K-major (forward)
                    if (X3) {
                        // loaded above
                    } else if (b_wide) {
                        if (FWD) ptx::tma_load_2d(sB, tmBw, fb, kb * KBLK, col0);
                        else ptx::tma_load_3d(sB, tmBw, fb, 0, kb * KBLK, col0 / 64);
                    } else {
                        for (int j = 0; j < nb; ++j) {
                            if (FWD) ptx::tma_load_2d(sB + j * BOX_BYTES, tmB, fb, kb * KBLK, col0 + j * 64);
                            else ptx::tma_load_2d(sB + j * BOX_BYTES, tmB, fb, col0 + j * 64, kb * KBLK);
                        }
                    }
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // This CTA's copies still in flight land before shared memory goes
            // away (its own full barrier counts its own bytes; in a normal run
            // every phase has already been consumed and these return at once).
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u) wt.wait_teardown(bars + 8u * (BAR_FULL + s), (last_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (leader) {
            // -------------------------------------------------------- MMA issuer
            if (lane == 0) {
                const uint16_t pair_mask = 0x3u;  // both CTAs of the pair
                uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
                bool ok = true;
                bool prev_bias = false;  // the previous item put its column sums in this set
                for (int r = 0; ok; ++r) {
                    const int w = item_at(p, sch, r);
                    if (w >= p.n_items) break;
                    const Item it = decode_item(p, w);
                    if (!wt.wait(bars + 8u * (BAR_TEMPTY + acc), acc_phase ^ 1u, SITE_MMA_TMEM_EMPTY, w)) break;
                    // dbias by MMA: a dweight item of the first column tile also
                    // accumulates doutT . ones (N = 16) into the first 16 columns of
                    // the other accumulator set, so the last item issued into that set
                    // must have been drained, and the item after this one must wait
                    // until this item's epilogue has read the sums.
                    const bool bias_item = !FWD && !X3 && p.bias_mma && it.is_dw && it.n_tile == 0;
                    if (bias_item || prev_bias) {
                        const uint32_t o = acc ^ 1u, ph_o = acc == 0 ? acc_phase ^ 1u : acc_phase;
                        if (!wt.wait(bars + 8u * (BAR_TEMPTY + o), ph_o, SITE_MMA_TMEM_EMPTY, w)) break;
                    }
                    prev_bias = bias_item;
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * acc_cols;
                    const uint32_t d_bias = tmem_base + (acc ^ 1u) * TC_BN;
                    const uint32_t ones = base + L::OFF_ONES;
                    const uint32_t idesc = X3 ? ptx::idesc_tf32_f32(TC_PAIR_BM, it.bn, 0, 0)
                                              : ptx::idesc_bf16_f32(TC_PAIR_BM, it.bn, /*A MN*/ it.is_dw,
                                                                    /*B MN*/ FWD ? 0 : 1);
                    for (int kb = it.kb0; kb < it.kb1; ++kb) {
                        // Both CTAs' copies of this stage have landed (own bytes +
                        // the odd CTA's forwarded arrival); MODE 2: both CTAs'
                        // split warps have written the planes.
                        const bool ready =
                            X3 ? wt.wait<true>(bars + 8u * (L::BAR_CONV + stage), phase, SITE_MMA_CONV, w)
                               : wt.wait(bars + 8u * (BAR_FULL + stage), phase, SITE_MMA_FULL, w);
                        if (!ready) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t sA = base + stage * STG_BYTES;
                        const uint32_t sB = sA + (X3 ? 2 : 1) * A_BYTES;
                        if constexpr (X3) {
                            // K-major tf32 slices of 8 elements: 32 bytes further into
                            // each swizzled 128-byte row, as for the bf16 K-major case.
                            const uint64_t ah0 = ptx::smem_desc_sw128(sA, 16, 1024);
                            const uint64_t al0 = ptx::smem_desc_sw128(sA + A_BYTES, 16, 1024);
                            const uint64_t bh0 = ptx::smem_desc_sw128(sB, 16, 1024);
                            const uint64_t bl0 = ptx::smem_desc_sw128(sB + B_BYTES, 16, 1024);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t ah = ah0 + 2u * k, al = al0 + 2u * k;  // +32 bytes per slice
                                const uint64_t bh = bh0 + 2u * k, bl = bl0 + 2u * k;
                                // The tensor core rounds each accumulation toward zero, so
                                // the error of an accumulator grows with the number of
                                // accumulations into it times its own magnitude. Long
                                // reductions: hi.hi alone in the main accumulator, hi.lo +
                                // lo.hi (about 2^-11 of it) in the correction accumulator
                                // beside it; short ones: all three in one.
                                const uint32_t acc0 = (kb > it.kb0 || k > 0) ? 1u : 0u;
                                const uint32_t d_corr = corr ? d_tmem + it.bn : d_tmem;
                                ptx::mma_tf32_pair(d_tmem, ah, bh, idesc, acc0);
                                ptx::mma_tf32_pair(d_corr, ah, bl, idesc, corr ? acc0 : 1u);
                                ptx::mma_tf32_pair(d_corr, al, bh, idesc, 1u);
                            }
                        } else {
                            // K-major A: the 16-element K slice starts 32 bytes further
                            // into each swizzled 128-byte row (descriptor address +2);
                            // rows in 8-row groups of 1024 bytes. MN-major operands: 16 K
                            // rows of 128 bytes per slice (2048 bytes: address +128);
                            // 64-wide MN boxes 8 KB apart (leading offset), 8-row K groups
                            // 1024 bytes apart (stride offset). The descriptors of a
                            // k-block are formed once and stepped by addition (the address
                            // field stays below 2^14), which keeps this single thread's
                            // issue loop short: the tensor pipe waits on it.
                            const uint64_t a0 = it.is_dw ? ptx::smem_desc_sw128(sA, BOX_BYTES, 1024)
                                                         : ptx::smem_desc_sw128(sA, 16, 1024);
                            const uint64_t a_step = it.is_dw ? 128u : 2u;
                            // Forward: B is K-major like A (weight rows of 128 bytes of K).
                            const uint64_t b0 = FWD ? ptx::smem_desc_sw128(sB, 16, 1024)
                                                    : ptx::smem_desc_sw128(sB, BOX_BYTES, 1024);
                            constexpr uint64_t b_step = FWD ? 2u : 128u;
                            const uint32_t first = kb > it.kb0 ? 1u : 0u;
                            if (!bias_item) {
#pragma unroll
                                for (int k = 0; k < TC_BK / 16; ++k)
                                    ptx::mma_bf16_pair(d_tmem, a0 + k * a_step, b0 + k * b_step, idesc,
                                                       k > 0 ? 1u : first);
                            } else {
                                // dbias by MMA: D_bias (256 x 16) += doutT (256 x 16 of K) .
                                // ones (16 x 16) beside each main MMA
                                const uint64_t o0 = ptx::smem_desc_sw128(ones, 16, 1024);
                                constexpr uint32_t idesc_b = ptx::idesc_bf16_f32(TC_PAIR_BM, 16, 1, 0);
#pragma unroll
                                for (int k = 0; k < TC_BK / 16; ++k) {
                                    ptx::mma_bf16_pair(d_tmem, a0 + k * a_step, b0 + k * b_step, idesc,
                                                       k > 0 ? 1u : first);
                                    ptx::mma_bf16_pair(d_bias, a0 + k * a_step, o0 + k * 2u, idesc_b,
                                                       k > 0 ? 1u : first);
                                }
                            }
                        }
                        ptx::mma_commit_pair_multicast(bars + 8u * (BAR_EMPTY + stage), pair_mask);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair_multicast(bars + 8u * (BAR_TFULL + acc), pair_mask);
                    if (++acc == acc_sets) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
                // Every MMA this thread issued completes (and with it every copy
                // they read) before shared and tensor memory are released.
                ptx::mma_commit_pair(bars + 8u * BAR_TEARDOWN);
                wt.wait_teardown(bars + 8u * BAR_TEARDOWN, 0);
            }
        } else {
            // ---------------------------------------------- forwarder (odd CTA)
            // (MODE 2: the split warps signal the even CTA themselves)
            if (lane == 0 && !X3) {
                const uint32_t leader_full = ptx::mapa(bars + 8u * BAR_FULL, 0);
                uint32_t stage = 0, phase = 0;
                bool ok = true;
                for (int r = 0; ok; ++r) {
                    const int w = item_at(p, sch, r);
                    if (w >= p.n_items) break;
                    const Item it = decode_item(p, w);
                    for (int kb = it.kb0; kb < it.kb1; ++kb) {
                        if (!wt.wait(bars + 8u * (BAR_FULL + stage), phase, SITE_FORWARD_FULL, w)) {
                            ok = false;
                            break;
                        }
                        ptx::mbar_arrive_cluster_relaxed(leader_full + 8u * stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI) {
        if constexpr (X3) {
            // ------------------------------------------------------ split warps
            // Warp 2 splits operand A of every stage, warp 3 operand B, each
            // into its K-major high and low planes (x3_split_k / x3_split_mn),
            // each on its own, then a proxy fence (the planes are read by the
            // tensor cores of both CTAs) and one arrival on the even CTA's
            // barrier of the stage. The fence completes only once the warp's
            // shared-memory writes are visible to the async proxy, and the
            // arrival is issued after it, so it is relaxed, as the forwarder's
            // is for TMA data: a releasing arrival at cluster scope also waits
            // for the SM's unrelated memory traffic in flight and cost this
            // path a third of its time (XL fc 662 -> 980 us). On the items of
            // column tile 0 whose A arrives MN-major (the dweight product: A =
            // dout^T), warp 2 also sums A's rows over all of K: dbias.
            const bool is_a = warp == WARP_BIAS;
            const uint32_t conv0 = ptx::mapa(bars + 8u * L::BAR_CONV, 0);
            uint32_t stage = 0, phase = 0;
            for (int r = 0;; ++r) {
                const int w = item_at(p, sch, r);
                if (w >= p.n_items) break;
                const Item it = decode_item(p, w);
                const int sh = (it.is_dw ? 2 : 0) + (is_a ? 0 : 1);
                const bool mn = ((p.x3_mn >> sh) & 1) != 0;
                const int64_t a_rows = it.is_dw ? p.OC : p.BT;
                const int row0 = it.pm * TC_PAIR_BM + static_cast<int>(rank) * TC_BM;
                const int half = it.bn / 2;
                const int col0 = it.n_tile * it.bn + static_cast<int>(rank) * half;
                // this CTA's boxes of the operand holding any row of the tensor
                int nbox = 0;
                if (is_a) {
                    nbox = mn ? (row0 < a_rows ? 1 : 0) + (row0 + 64 < a_rows ? 1 : 0) : (row0 < a_rows ? 1 : 0);
                } else {
                    for (int j = 0; j < half / 64; ++j) nbox += (col0 + j * 64 < p.n_dinp) ? 1 : 0;
                }
                const bool sums = is_a && mn && p.x3_dbias != nullptr && it.n_tile == 0;
                float bsum[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t plane = base + (is_a ? 0u : 2u * A_BYTES);  // high plane; the low one follows
                const uint32_t plane_bytes = is_a ? A_BYTES : B_BYTES;
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!wt.wait_warp(bars + 8u * (BAR_FULL + stage), phase, SITE_CONV_RAW, w)) {
                        ok = false;
                        break;
                    }
                    const uint32_t hi = plane + stage * STG_BYTES, lo = hi + plane_bytes;
                    if (mn) x3_split_mn(hi, lo, nbox, lane, sums, bsum);
                    else if (nbox) x3_split_k(hi, lo, is_a ? A_BYTES / 16 : nbox * (BOX_BYTES / 16), lane);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_cluster_relaxed(conv0 + 8u * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (sums) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t o = static_cast<int64_t>(row0) + 32 * q + lane;
                        if (q / 2 < nbox && o < a_rows) p.x3_dbias[o] = bsum[q];
                    }
                }
            }
        } else {
            // ------------------------------------------------------- bias warps
            // They read every stage (releasing it), sum the dout tiles of dweight
            // items of the first column tile, and store their 64 column sums
            // themselves: to dbias, rounded once, or as this split's fp32 partial
            // (the split reduction adds them in split order). They share no
            // buffer with the epilogue, so they never wait for it.
            if (bias_on && !p.bias_mma) {
                const int bw = warp - WARP_BIAS;  // which 64-wide box of the A tile
                uint32_t stage = 0, phase = 0;
                for (int r = 0;; ++r) {
                    const int w = item_at(p, sch, r);
                    if (w >= p.n_items) break;
                    const Item it = decode_item(p, w);
                    const bool has_bias = it.is_dw && it.n_tile == 0;
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
                            const uint8_t* box = smem + stage * STG_BYTES + bw * BOX_BYTES;
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
                        if (++stage == STAGES) {
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
                            const int m_tile = it.pm * 2 + static_cast<int>(rank);  // 128-row tile of dweight
                            const int row0 = bw * 64 + lane * 8;                    // first of this lane's 8 rows
                            if (p.splits > 1) {
                                float* bp = p.bias_partials + (static_cast<size_t>(m_tile) * p.splits + it.split) * TC_BM + row0;
                                *reinterpret_cast<float4*>(bp) = make_float4(s[0], s[1], s[2], s[3]);
                                *reinterpret_cast<float4*>(bp + 4) = make_float4(s[4], s[5], s[6], s[7]);
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const int64_t o = static_cast<int64_t>(m_tile) * TC_BM + row0 + e;
                                    if (o < p.OC) {
                                        if constexpr (SR)
                                            p.dbias[o] = sr::round(s[e], p.sr_seed, sr::DBIAS, o);
                                        else
                                            p.dbias[o] = __float2bfloat16_rn(s[e]);
                                    }
                                }
                            }
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;         // tensor-memory lane quadrant: tile rows 32q..32q+31
        const int ew = warp - WARP_EPI;  // this warp's buffers and barriers
        constexpr int NH = L::EPI_WARPS / 4;  // warps per quadrant: chunks h, h + NH, h + 2 NH, ...
        const int h = ew / 4;
        const int r8 = lane >> 2;       // coalesced phase: rows 8i + r8 of the quadrant,
        const int cg = (lane & 3) * 8;  //   columns cg..cg+7 of each 32-column chunk
        const uint32_t stg = base + L::OFF_STAGE + ew * L::WARP_REGION;
        // bf16 read-modify-write (MODE 0 and 3, unsplit items): this warp's
        // ring of old-value chunks, their barriers, parities and pending loads
        const uint32_t oldbuf = base + L::OFF_STAGE + ew * L::WARP_REGION;
        const uint32_t oldbar0 = bars + 8u * (BAR_OLD + ew * OLD_SLOTS);
        uint32_t oldpar = 0, oldpend = 0;
        uint32_t fwd_chunks = 0;  // forward: chunks this warp has stored (slot = count mod OLD_SLOTS)
        const uint32_t leader_tempty = ptx::mapa(bars + 8u * BAR_TEMPTY, 0);
        uint32_t acc = 0, acc_phase = 0;
        for (int r = 0;; ++r) {
            const int w = item_at(p, sch, r);
            if (w >= p.n_items) break;
            const Item it = decode_item(p, w);
            const int m_tile = it.pm * 2 + static_cast<int>(rank);  // 128-row tile
            const bool split_mode = it.is_dw && p.splits > 1;
            const int64_t rows_total = it.is_dw ? p.OC : p.BT;
            const int64_t qrow0 = static_cast<int64_t>(m_tile) * TC_BM + q * 32;  // first row of the quadrant
            const int col0 = it.n_tile * it.bn;
            const int64_t n_extent = FWD ? p.n_dinp : p.C;  // columns and row stride of D
            const int ncols = static_cast<int>(min(static_cast<int64_t>(it.bn), n_extent - col0));
            const int nchunks = it.bn / 32;
            float* Df = reinterpret_cast<float*>(it.is_dw ? p.dweight : p.dinp);  // MODE 2: fp32 output
            // fp32 read-modify-write (MODE 2): this thread's rows of the coalesced phase
            bool rok[4];
            float* drowf[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t row = qrow0 + 8 * i + r8;
                rok[i] = row < rows_total;
                drowf[i] = Df + (rok[i] ? row : 0) * n_extent + col0 + cg;
            }
            // The backward's bf16 read-modify-write goes through TMA: the old
            // values of this warp's 32 rows arrive in 32-column chunks (its first
            // two requested at the start of the item, before waiting for the
            // accumulator), each thread adds its own row in place, and the chunk
            // goes back out with one bulk store. Rows and columns outside the
            // tensor read as zero and are not stored.
            const bool tma_rmw = !FWD && !X3 && !split_mode;
            constexpr bool TMA_FWD = FWD && !X3;  // the forward's stores through TMA as well
            const void* tmo = it.is_dw ? static_cast<const void*>(&tm_dw_rmw) : static_cast<const void*>(&tm_dinp_rmw);
            const int nvc = (ncols + 31) / 32;  // chunks holding columns of the tensor
            const int nloc = nvc > h ? (nvc - h + NH - 1) / NH : 0;  // of them this warp's
            const int nloc_all = (nchunks - h + NH - 1) / NH;       // this warp's of the tile
            const bool qvalid = qrow0 < rows_total;
            if constexpr (!FWD && !X3) {
                // the previous item's stores have read the chunk buffers (also the
                // staging area of a split item)
                if (lane == 0) ptx::bulk_wait_read_all();
                __syncwarp();
            }
            if (tma_rmw && qvalid && lane == 0) {
                for (int k = 0; k < OLD_SLOTS && k < nloc; ++k) {
                    const uint32_t b = oldbar0 + 8u * k;
                    ptx::mbar_arrive_expect_tx(b, OLD_CHUNK_BYTES);
                    ptx::tma_load_2d(oldbuf + k * OLD_CHUNK_BYTES, tmo, b, col0 + (h + NH * k) * 32,
                                     static_cast<int32_t>(qrow0));
                    oldpend |= 1u << k;
                }
            }

            // MODE 2: this thread's old values of the first chunk (4 rows x 8
            // columns), requested before the accumulator is ready; each later
            // chunk's are requested while the chunk before is added and stored
            float4 olda[4], oldb[4];
            auto x3_load_old = [&](int cc, float4 (&A)[4], float4 (&Bv)[4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    A[i] = Bv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (rok[i] && cc * 32 + cg < ncols) {  // (the row width is a multiple of 4)
                        const float4* dp = reinterpret_cast<const float4*>(drowf[i] + cc * 32);
                        A[i] = dp[0];
                        if (cc * 32 + cg + 4 < ncols) Bv[i] = dp[1];
                    }
                }
            };
            if constexpr (X3) x3_load_old(0, olda, oldb);
            bool ok = wt.wait_warp(bars + 8u * (BAR_TFULL + acc), acc_phase, SITE_EPI_TMEM_FULL, w);
            if (!ptx::named_bar_and(1, L::EPI_THREADS, ok)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * acc_cols;
            if constexpr (!FWD && !X3) {
                if (p.bias_mma && it.is_dw && it.n_tile == 0 && qvalid && h == 0) {
                    // dbias by MMA: every column of the sums block holds the row's sum
                    const float bsum = __uint_as_float(
                        ptx::tmem_ld1(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + (acc ^ 1u) * TC_BN));
                    const int64_t o = qrow0 + lane;
                    if (split_mode)
                        p.bias_partials[(static_cast<size_t>(m_tile) * p.splits + it.split) * TC_BM + q * 32 + lane] = bsum;
                    else if (o < p.OC) {
                        if constexpr (SR)
                            p.dbias[o] = sr::round(bsum, p.sr_seed, sr::DBIAS, o);
                        else
                            p.dbias[o] = __float2bfloat16_rn(bsum);
                    }
                }
            }
            if constexpr (!FWD && !X3) {
                if (split_mode && qvalid) {
                    // This split's fp32 partial through TMA: row `lane` of each 32 x 32
                    // chunk into a 4 KB buffer (128-byte rows; 16-byte granule g at
                    // g ^ (lane & 7), the 128-byte swizzle, conflict-free), one bulk
                    // store per chunk into [128-row tile x column tile][split][128][bn];
                    // a buffer is rewritten once the store that used it PART_SLOTS
                    // chunks ago has read it.
                    const int32_t prow = static_cast<int32_t>(
                        ((static_cast<int64_t>(m_tile) * p.dw_tiles_n + it.n_tile) * p.splits + it.split) * TC_BM + q * 32);
                    const uint32_t swz = static_cast<uint32_t>(lane & 7);
#pragma unroll 1
                    for (int k = 0; k < nloc_all; ++k) {
                        const int c = h + NH * k;
                        uint32_t v[32];
                        ptx::tmem_ld32(tbase + c * 32, v);
                        const int slot = k & (L::PART_SLOTS - 1);
                        if (k >= L::PART_SLOTS && lane == 0) ptx::bulk_wait_read_but_n<L::PART_SLOTS - 1>();
                        __syncwarp();
                        const uint32_t rowaddr = oldbuf + slot * PART_CHUNK_BYTES + lane * 128;
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            ptx::sts128u(rowaddr + ((static_cast<uint32_t>(g) ^ swz) << 4),
                                         make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&tm_part, oldbuf + slot * PART_CHUNK_BYTES, c * 32, prow);
                            ptx::bulk_commit_group();
                        }
                    }
                }
            }
            if (tma_rmw && qvalid) {
                const uint64_t t_sr = it.is_dw ? sr::DWEIGHT : sr::DINP;
                // 16-byte granule g of row `lane` sits at granule g ^ ((lane >> 1) & 3)
                // (64-byte swizzle; conflict-free across each 8-thread phase)
                const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll 1
                for (int k = 0; k < nloc; ++k) {
                    const int c = h + NH * k;
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c * 32, v);
                    const int slot = k & (OLD_SLOTS - 1);
                    const uint32_t b = oldbar0 + 8u * slot;
                    if (!wt.wait_warp(b, (oldpar >> slot) & 1u, SITE_EPI_OLD, w)) {
                        ok = false;
                        break;
                    }
                    oldpar ^= 1u << slot;
                    oldpend &= ~(1u << slot);
                    const uint32_t rowaddr = oldbuf + slot * OLD_CHUNK_BYTES + lane * 64;
                    // the row's 32 columns start at element e_row (a multiple of 8:
                    // C is), so their eight words have consecutive counters
                    const uint64_t e_row = static_cast<uint64_t>(qrow0 + lane) * n_extent + col0 + c * 32;
                    const uint64_t z0 = SR ? sr::word_state(p.sr_seed, t_sr, e_row) : 0;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint32_t a = rowaddr + ((static_cast<uint32_t>(g) ^ swz) << 4);
                        const uint4 o = ptx::lds128(a);
                        float s8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) s8[e] = __uint_as_float(v[8 * g + e]);
                        uint4 res;
                        if constexpr (SR)
                            res = add_sr8(o, s8, sr::sm64_mix(z0 + (2 * g) * sr::SM64_GAMMA),
                                          sr::sm64_mix(z0 + (2 * g + 1) * sr::SM64_GAMMA));
                        else
                            res = add_round8(o, s8);
                        ptx::sts128u(a, res);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(tmo, oldbuf + slot * OLD_CHUNK_BYTES, col0 + c * 32, static_cast<int32_t>(qrow0));
                        ptx::bulk_commit_group();
                        // Refill this chunk's buffer with the warp's chunk OLD_SLOTS
                        // ahead once this chunk's store has read it.
                        const int kn = k + OLD_SLOTS;
                        if (kn < nloc) {
                            ptx::bulk_wait_read_all();
                            ptx::mbar_arrive_expect_tx(b, OLD_CHUNK_BYTES);
                            ptx::tma_load_2d(oldbuf + slot * OLD_CHUNK_BYTES, tmo, b, col0 + (h + NH * kn) * 32,
                                             static_cast<int32_t>(qrow0));
                            oldpend |= 1u << slot;
                        }
                    }
                    __syncwarp();
                }
            }
            if (TMA_FWD && qvalid) {
                // out = acc + bias, rounded once, row by row into a chunk buffer and
                // out with one bulk store; a buffer is rewritten once the store that
                // used it OLD_SLOTS chunks ago has read it.
                const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll 1
                for (int k = 0; k < nloc; ++k) {
                    const int c = h + NH * k;
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c * 32, v);
                    const uint32_t slot = fwd_chunks & (OLD_SLOTS - 1);
                    if (fwd_chunks >= OLD_SLOTS && lane == 0) ptx::bulk_wait_read_but_n<OLD_SLOTS - 1>();
                    __syncwarp();
                    const uint32_t rowaddr = oldbuf + slot * OLD_CHUNK_BYTES + lane * 64;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int cc = col0 + c * 32 + 8 * g;
                        const uint4 b8 = (p.fwd_bias && cc < n_extent)
                                             ? __ldg(reinterpret_cast<const uint4*>(p.fwd_bias + cc))
                                             : make_uint4(0u, 0u, 0u, 0u);
                        float s8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) s8[e] = __uint_as_float(v[8 * g + e]);
                        ptx::sts128u(rowaddr + ((static_cast<uint32_t>(g) ^ swz) << 4), add_round8(b8, s8));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(tmo, oldbuf + slot * OLD_CHUNK_BYTES, col0 + c * 32, static_cast<int32_t>(qrow0));
                        ptx::bulk_commit_group();
                    }
                    ++fwd_chunks;
                }
            }
            if (!ptx::named_bar_and(1, L::EPI_THREADS, ok)) break;
            if constexpr (X3) {  // MODE 2: fp32 read-modify-write through staging rows
#pragma unroll 1
                for (int c = 0; c < nchunks; ++c) {
                    float4 nxa[4], nxb[4];
                    if (c + 1 < nchunks) x3_load_old(c + 1, nxa, nxb);
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c * 32, v);
                    if (corr) {  // main + correction, one IEEE fp32 addition
                        uint32_t w2[32];
                        ptx::tmem_ld32(tbase + it.bn + c * 32, w2);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(w2[e]));
                    }
                    // Row `lane` of the quadrant into the staging buffer ...
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        ptx::sts128(stg + (lane * STG_STRIDE + 4 * k) * 4, __uint_as_float(v[4 * k]),
                                    __uint_as_float(v[4 * k + 1]), __uint_as_float(v[4 * k + 2]),
                                    __uint_as_float(v[4 * k + 3]));
                    __syncwarp();
                    // ... and back out as 8 rows x 32 columns per instruction.
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int lr = 8 * i + r8;
                        const float4 a4 = ptx::lds128f(stg + (lr * STG_STRIDE + cg) * 4);
                        const float4 b4 = ptx::lds128f(stg + (lr * STG_STRIDE + cg + 4) * 4);
                        if (rok[i] && c * 32 + cg < ncols) {
                            float4* dp = reinterpret_cast<float4*>(drowf[i] + c * 32);
                            float4 o0 = olda[i], o1 = oldb[i];
                            o0.x += a4.x, o0.y += a4.y, o0.z += a4.z, o0.w += a4.w;
                            o1.x += b4.x, o1.y += b4.y, o1.z += b4.z, o1.w += b4.w;
                            dp[0] = o0;
                            if (c * 32 + cg + 4 < ncols) dp[1] = o1;
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        olda[i] = nxa[i];
                        oldb[i] = nxb[i];
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_relaxed(leader_tempty + 8u * acc);
            if (++acc == acc_sets) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // Old-value loads still in flight (only after an abort) land, and every
        // bulk store has completed, before shared memory goes away.
        if (lane == 0) {
            for (int sl = 0; sl < OLD_SLOTS; ++sl)
                if ((oldpend >> sl) & 1u) wt.wait_teardown(oldbar0 + 8u * sl, (oldpar >> sl) & 1u);
            ptx::bulk_wait_all();
        }
        __syncwarp();
    }

    // Each thread is done with its role: the next launch on the stream may start
    // its prologue on SMs this grid frees (every thread signals; measured faster
    // than a single signalling thread).
    ptx::grid_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    // The even CTA's MMAs (which write this CTA's tensor memory and read its
    // shared memory) have completed before either CTA releases anything.
    ptx::cluster_sync();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Split reduction: dweight = dweight + (partial_0 + partial_1 + ... + partial_{S-1})
// with the partials summed in split order and one rounding to bf16 (to nearest,
// or stochastic as in the kernel's MODE 3), and
// dbias = bias_partial_0 + ... + bias_partial_{S-1} in the same order. One
// thread per 8-column vector of dweight; all loads are independent, so the
// pass runs at memory speed with the partials still in L2.
__global__ void __launch_bounds__(256) tc_splitk_fixup_kernel(const TcParams p) {
    // The next launch on the stream (the tensor-core kernel, as a rule) may
    // start its prologue beside this small pass; it still waits for this grid
    // to complete before touching global memory.
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();  // the partials of the GEMM launch before this one
    const int64_t vec_per_row = p.C / 8;
    const int64_t nvec = p.OC * vec_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const size_t tile_elems = static_cast<size_t>(TC_BM) * p.dw_bn;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        const int64_t row = v / vec_per_row;
        const int64_t col = (v - row * vec_per_row) * 8;
        const int m_tile = static_cast<int>(row / TC_BM), rl = static_cast<int>(row % TC_BM);
        const int n_tile = static_cast<int>(col / p.dw_bn), cl = static_cast<int>(col % p.dw_bn);
        const float* pp = p.partials + static_cast<size_t>(m_tile * p.dw_tiles_n + n_tile) * p.splits * tile_elems +
                          static_cast<size_t>(rl) * p.dw_bn + cl;
        uint4* dst = reinterpret_cast<uint4*>(p.dweight + row * p.C + col);
        const uint4 old = *dst;  // requested beside the partials, not after their sum
        float s8[8];
#pragma unroll 4
        for (int sp = 0; sp < p.splits; ++sp) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(pp + sp * tile_elems));
            const float4 b = __ldcg(reinterpret_cast<const float4*>(pp + sp * tile_elems + 4));
            const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) s8[e] = (sp == 0) ? f[e] : s8[e] + f[e];
        }
        if (p.sr) {
            const uint64_t e0 = static_cast<uint64_t>(row * p.C + col);
            *dst = add_sr8(old, s8, sr::word(p.sr_seed, sr::DWEIGHT, e0), sr::word(p.sr_seed, sr::DWEIGHT, e0 + 4));
        } else {
            *dst = add_round8(old, s8);
        }
    }
    if (p.dbias) {
        for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < p.OC; o += stride) {
            const int m_tile = static_cast<int>(o / TC_BM), rl = static_cast<int>(o % TC_BM);
            float b = 0.f;
            for (int sp = 0; sp < p.splits; ++sp) {
                const float f = __ldcg(p.bias_partials + (static_cast<size_t>(m_tile) * p.splits + sp) * TC_BM + rl);
                b = (sp == 0) ? f : b + f;
            }
            p.dbias[o] = p.sr ? sr::round(b, p.sr_seed, sr::DBIAS, o) : __float2bfloat16_rn(b);
        }
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

// Planner cost model (µs). An item costs its main loop (a 64-deep k-block of
// a 256 x bn pair tile) or its epilogue, whichever is longer, since the two
// overlap across the two accumulators, plus a per-item handoff; the last
// item's epilogue is not overlapped. Split dweight adds the fixup pass. The
// constants are fitted, through this planner's own schedule, to 60 plans
// forced on GB300 (six GPT-2 layer shapes, split counts 1 to 5, both tile
// widths; squared relative error 0.07, and the measured-best plan picked for
// every shape). A k-block costs the same at either width: the stage ring's
// round trip, not the MMA, sets a 128-wide k-block's time.
double t_kb(int /*bn*/) { return 0.32; }
double t_rmw(int bn) { return 0.9 + 3.5 * bn / 256.0; }      // bf16 read-modify-write of 128 x bn
double t_partial(int bn) { return 1.5 + 1.6 * bn / 256.0; }  // fp32 partial store of 128 x bn
constexpr double T_ITEM = 1.0;                                 // per-item handoff

struct ItemCost {
    double run, epi;
};

// fp32 from three tf32 products, both products in one launch: a k-block of
// 32 fp32 of K with three pair MMAs, its operands split in shared memory by
// the kernel, takes about 0.99 us at width 256 and 0.87 at 128 (the split of
// the A operand, the same at either width, and the stage ring's round trip
// keep a 128-wide k-block from halving); with a correction accumulator a
// 256-wide tile fills all 512 tensor-memory columns, so its fp32 epilogue is
// not overlapped (about 2 us exposed). Fitted, through this planner's own
// longest-first schedule, to the paired launches of the GPT-2 XL fc and qkv
// layers at both widths (658, 1031, 540, 722 us measured; 660, 1019, 540, 729
// modelled with 3 us per launch).
double x3_item_us(int kb, int bn, bool corr) { return kb * (bn == 256 ? 0.99 : 0.87) + (bn == 256 && corr ? 2.0 : 0.0); }

ItemCost item_cost(const TcPlan& pl, int w) {
    if (pl.x3) {
        const bool dw = w < pl.n_dw_items;
        return {x3_item_us(dw ? pl.dw_kb : pl.dinp_kb, dw ? pl.dw_bn : pl.dinp_bn, pl.x3_corr != 0), 0.0};
    }
    if (w < pl.n_dw_items) {
        const int split = w / pl.dw_tiles_n / pl.dw_tiles_m;
        const int kb0 = split * pl.kb_per_split;
        const int kb = std::min(kb0 + pl.kb_per_split, pl.dw_kb) - kb0;
        const double epi = pl.splits > 1 ? t_partial(pl.dw_bn) : t_rmw(pl.dw_bn);
        return {std::max(kb * t_kb(pl.dw_bn), epi) + T_ITEM, epi};
    }
    const double epi = t_rmw(pl.dinp_bn);
    return {std::max(pl.dinp_kb * t_kb(pl.dinp_bn), epi) + T_ITEM, epi};
}

double fixup_cost(const TcPlan& pl, int64_t C, int64_t OC) {
    if (pl.splits == 1) return 0.0;
    // a launch gap, about 1 us per split (each adds a wave of partial-store
    // epilogues), and the S fp32 partials read and dweight read and written
    // (L2-resident: 8 MB/us)
    const double bytes = static_cast<double>(OC) * C * (4.0 * pl.splits + 4.0);
    return 3.0 + 1.0 * pl.splits + bytes / 8e6;
}

// Longest-first greedy assignment of items to pairs; fills pl.sched and
// returns the estimated makespan (µs). Ties go to the lower pair index and to
// the earlier item, so the schedule is a pure function of the shape.
double assign_lpt(TcPlan& pl, int pairs) {
    static thread_local double load[TC_MAX_PAIRS], last_epi[TC_MAX_PAIRS];
    static thread_local int cnt[TC_MAX_PAIRS];
    static thread_local uint16_t owner[TC_MAX_SCHED_ITEMS];
    static thread_local int order[TC_MAX_SCHED_ITEMS];
    static thread_local ItemCost cost[TC_MAX_SCHED_ITEMS];
    const int n = pl.n_items;
    for (int w = 0; w < n; ++w) order[w] = w, cost[w] = item_cost(pl, w);
    std::stable_sort(order, order + n, [&](int a, int b) { return cost[a].run > cost[b].run; });
    for (int c = 0; c < pairs; ++c) load[c] = last_epi[c] = 0.0, cnt[c] = 0;
    for (int k = 0; k < n; ++k) {
        const int w = order[k];
        int best = 0;
        for (int c = 1; c < pairs; ++c)
            if (load[c] < load[best] - 1e-9) best = c;
        const ItemCost ic = cost[w];
        load[best] += ic.run;
        last_epi[best] = ic.epi;
        owner[k] = static_cast<uint16_t>(best);
        ++cnt[best];
    }
    pl.sched.start[0] = 0;
    for (int c = 0; c < pairs; ++c) pl.sched.start[c + 1] = static_cast<uint16_t>(pl.sched.start[c] + cnt[c]);
    for (int c = pairs; c < TC_MAX_PAIRS; ++c) pl.sched.start[c + 1] = pl.sched.start[pairs];
    int fill[TC_MAX_PAIRS];
    for (int c = 0; c < pairs; ++c) fill[c] = pl.sched.start[c];
    for (int k = 0; k < n; ++k) pl.sched.items[fill[owner[k]]++] = static_cast<uint16_t>(order[k]);
    double m = 0.0;
    for (int c = 0; c < pairs; ++c) m = std::max(m, load[c] + last_epi[c]);
    return m;
}

// Makespan (µs) of round-robin assignment (lists too long for the table).
double roundrobin_cost(const TcPlan& pl, int pairs) {
    double m = 0.0;
    for (int c = 0; c < pairs; ++c) {
        double l = 0.0, e = 0.0;
        for (int w = c; w < pl.n_items; w += pairs) {
            const ItemCost ic = item_cost(pl, w);
            l += ic.run;
            e = ic.epi;
        }
        m = std::max(m, l + e);
    }
    return m;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

std::mutex g_attr_mutex;
bool g_attr_set[64];

}  // namespace

size_t tc_smem_bytes() { return SMEM_TOTAL; }

int tc_max_active_clusters(int cluster_size) {
    if (cudaFuncSetAttribute(tc_mmbwd_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc_mmbwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc_mmbwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) !=
            cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster_size), 1, 1);
    cfg.blockDim = dim3(Smem<0>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_TOTAL;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_mmbwd_kernel<0>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// The planner for a launch whose dinp-type product is (BT x N) += (BT x K) . (K x N)
// with N = C and K = OC, plus, when `with_dw`, the dweight product.
static TcPlan make_plan_impl(int64_t BT, int64_t C, int64_t OC, int num_sms, bool with_dw) {
    TcPlan pl{};
    pl.dinp_kb = ceil_div_i(OC, TC_BK);
    pl.dw_kb = ceil_div_i(BT, TC_BK);

    // Overrides (tuning, tests): a forced split count that would leave an
    // empty split is lowered to the nearest count that does not; a forced grid
    // is rounded down to whole pairs; MMBWD_TILE_N = "<dinp>,<dweight>" widths;
    // MMBWD_SPLIT_KB = k-blocks per split (the last split takes the rest).
    const long force_splits = env_long("MMBWD_SPLITK", 0);
    const long force_split_kb = env_long("MMBWD_SPLIT_KB", 0);
    const long force_grid = env_long("MMBWD_GRID", 0);
    int force_dinp_bn = 0, force_dw_bn = 0;
    if (const char* t = std::getenv("MMBWD_TILE_N")) {
        int a = 0, b = 0;
        if (std::sscanf(t, "%d,%d", &a, &b) == 2 && (a == 128 || a == 256) && (b == 128 || b == 256)) {
            force_dinp_bn = a;
            force_dw_bn = b;
        }
    }
    const int max_splits = with_dw ? std::max(1, std::min(pl.dw_kb, 16)) : 1;
    // Split lengths tried: dw_kb / x k-blocks (rounded up), the last split
    // taking what is left, for x = 1 .. max_splits (equal splits) and, up to
    // eight splits, x in quarter steps: longer splits with a short last one,
    // which shorten the longest items and leave the short ones to fill pairs
    // that hold dinp items (GPT-2 small qkv: 103 + 25 k-blocks, 46.3 -> 44.8 us
    // against two equal splits; every uneven split of the attention
    // projection measured slower than its three equal ones).
    static thread_local int kps_list[64];
    int n_kps = 0;
    auto add_kps = [&](int kps) {
        kps = std::max(1, kps);
        for (int i = 0; i < n_kps; ++i)
            if (kps_list[i] == kps) return;
        if (n_kps < 64) kps_list[n_kps++] = kps;
    };
    if (force_split_kb > 0) {
        add_kps(static_cast<int>(std::min<long>(force_split_kb, pl.dw_kb)));
    } else {
        for (int x = 1; x <= max_splits; ++x) add_kps(ceil_div_i(pl.dw_kb, x));
        for (int q = 5; q <= 4 * std::min(max_splits, 8); ++q) add_kps((4 * pl.dw_kb + q - 1) / q);
    }
    double best = 1e300;
    static thread_local TcPlan best_pl, c;
    const int max_pairs = std::max(1, std::min(num_sms / 2, TC_MAX_PAIRS));
    for (int dinp_bn = 256; dinp_bn >= 128; dinp_bn -= 128) {
        if (force_dinp_bn && dinp_bn != force_dinp_bn) continue;
        for (int dw_bn = 256; dw_bn >= 128; dw_bn -= 128) {
            if (force_dw_bn && dw_bn != force_dw_bn) continue;
            for (int ki = 0; ki < n_kps; ++ki) {
                const int kps = kps_list[ki];
                const int S = ceil_div_i(pl.dw_kb, kps);  // every split non-empty
                // the partial tiles' rows are addressed by a 32-bit TMA coordinate
                if (S > 1 && static_cast<int64_t>(2 * ceil_div_i(OC, TC_PAIR_BM)) * ceil_div_i(C, dw_bn) * S * TC_BM >
                                 INT32_MAX)
                    continue;
                if (force_splits > 0) {  // equal splits of the forced count
                    const int fk = ceil_div_i(pl.dw_kb, static_cast<int>(std::min<long>(force_splits, max_splits)));
                    if (kps != fk) continue;
                }
                c = pl;
                c.dinp_tiles_m = ceil_div_i(BT, TC_PAIR_BM);
                c.dw_tiles_m = ceil_div_i(OC, TC_PAIR_BM);
                c.dinp_bn = dinp_bn;
                c.dw_bn = dw_bn;
                c.dinp_tiles_n = ceil_div_i(C, dinp_bn);
                c.dw_tiles_n = ceil_div_i(C, dw_bn);
                c.n_dinp_items = c.dinp_tiles_m * c.dinp_tiles_n;
                c.splits = S;
                c.kb_per_split = kps;
                c.n_dw_items = with_dw ? c.dw_tiles_m * c.dw_tiles_n * S : 0;
                c.n_items = c.n_dw_items + c.n_dinp_items;
                int pairs = std::max(1, std::min(c.n_items, max_pairs));
                if (force_grid > 0) pairs = static_cast<int>(std::max<long>(1, std::min<long>(force_grid / 2, pairs)));
                c.grid = 2 * pairs;
                c.table = (pairs <= TC_MAX_PAIRS && c.n_items <= TC_MAX_SCHED_ITEMS) ? 1 : 0;
                // No schedule beats the work per pair or the longest item: skip
                // the candidate when that bound is no better than the best so far.
                {
                    double work = 0.0, longest = 0.0;
                    if (c.n_dinp_items > 0) {
                        const ItemCost d = item_cost(c, c.n_dw_items);
                        work += d.run * c.n_dinp_items;
                        longest = d.run;
                    }
                    const int tiles = c.n_dw_items / std::max(1, S);
                    for (int sp = 0; sp < S && tiles > 0; ++sp) {
                        const ItemCost d = item_cost(c, sp * tiles);
                        work += d.run * tiles;
                        longest = std::max(longest, d.run);
                    }
                    if (std::max(work / pairs, longest) + fixup_cost(c, C, OC) >= best - 1e-9) continue;
                }
                const double cost = (c.table ? assign_lpt(c, pairs) : roundrobin_cost(c, pairs)) + fixup_cost(c, C, OC);
                c.est_us = cost;
                if (cost < best - 1e-9) {
                    best = cost;
                    best_pl = c;
                }
            }
        }
    }
    pl = best_pl;
    pl.fixup_grid = 0;
    if (pl.splits > 1) {
        const int64_t nvec = OC * (C / 8);
        pl.fixup_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((nvec + 255) / 256, 8 * std::max(2, num_sms))));
        const size_t row_tiles = static_cast<size_t>(2 * pl.dw_tiles_m);  // 128-row tiles
        const size_t half_tiles = row_tiles * pl.dw_tiles_n;
        pl.ws_partials_bytes = align256(half_tiles * pl.splits * TC_BM * pl.dw_bn * 4);
        pl.ws_bias_bytes = align256(row_tiles * pl.splits * TC_BM * 4);
    }
    return pl;
}

TcPlan tc_make_plan(int64_t BT, int64_t C, int64_t OC, int num_sms) {
    return make_plan_impl(BT, C, OC, num_sms, true);
}

TcPlan tc_make_plan_forward(int64_t BT, int64_t C, int64_t OC, int num_sms) {
    // forward: N = OC, K = C, no dweight product
    return make_plan_impl(BT, OC, C, num_sms, false);
}

// One fp32 product D (M x N) += A (M x K) . B (N x K)^T from tf32 halves: one
// pair per cluster, k-blocks of 32, the tile width (128 or 256) with the lower
// modelled time; items are equal in cost, so a round-robin assignment is
// balanced. Model (us, measured on the GPT-2 XL forward: 311 us at width 256,
// 429 at 128): a k-block of three pair MMAs with its operands split in shared
// memory takes about 1.0 us at width 256 and 0.8 at 128; with a separate
// correction accumulator (K > TC_X3_CORR_K) a 256-wide tile fills all 512
// tensor-memory columns, so its fp32 epilogue (about 2 us) is not overlapped.
TcPlan tc_make_plan_x3(int64_t M, int64_t N, int64_t K, int num_sms) {
    TcPlan pl{};
    pl.dinp_kb = ceil_div_i(K, TC_BK / 2);
    pl.dw_kb = 0;
    pl.dinp_tiles_m = ceil_div_i(M, TC_PAIR_BM);
    const int max_pairs = std::max(1, std::min(num_sms / 2, TC_MAX_PAIRS));
    double best = 1e300;
    const long force = env_long("MMBWD_TILE_N_X3", 0);
    for (int bn = 256; bn >= 128; bn -= 128) {
        if (force && bn != force) continue;
        const int tiles = pl.dinp_tiles_m * ceil_div_i(N, bn);
        const int pairs = std::max(1, std::min(tiles, max_pairs));
        const double item = pl.dinp_kb * (bn == 256 ? 1.0 : 0.8) + (bn == 256 && K > TC_X3_CORR_K ? 2.0 : 0.0);
        const double cost = std::ceil(static_cast<double>(tiles) / pairs) * item;
        if (cost < best) {
            best = cost;
            pl.dinp_bn = bn;
        }
    }
    pl.dw_bn = pl.dinp_bn;
    pl.dinp_tiles_n = ceil_div_i(N, pl.dinp_bn);
    pl.dw_tiles_n = pl.dinp_tiles_n;
    pl.n_dinp_items = pl.dinp_tiles_m * pl.dinp_tiles_n;
    pl.n_dw_items = 0;
    pl.n_items = pl.n_dinp_items;
    pl.splits = 1;
    pl.kb_per_split = pl.dinp_kb;
    const int pairs = std::max(1, std::min(pl.n_items, max_pairs));
    pl.grid = 2 * pairs;
    pl.table = 0;  // round robin
    pl.x3 = 1;
    pl.x3_corr = K > TC_X3_CORR_K ? 1 : 0;
    pl.est_us = best;
    pl.fixup_grid = 0;
    return pl;
}

namespace {

struct MapSpec {
    const void* base;
    uint64_t inner, outer;  // elements: contiguous dimension, rows
    uint32_t box_inner, box_outer;
    CUtensorMapSwizzle swz;
    uint64_t pitch = 0;     // bytes between rows (0: inner x element size)
};

// Encodes the six tensor maps, completes the parameters from the plan, and
// launches the kernel (and the split fixup when the plan splits dweight).
cudaError_t launch_common(const TcPlan& plan, const MapSpec (&specs)[6], TcParams& p, int mode, cudaStream_t stream,
                          const MapSpec* pair_specs = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> g(g_attr_mutex);
        if (dev < 0 || dev >= 64 || !g_attr_set[dev]) {
            e = cudaFuncSetAttribute(tc_mmbwd_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(tc_mmbwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(tc_mmbwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(tc_mmbwd_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) g_attr_set[dev] = true;
        }
    }
    EncodeTiledFn encode = get_encode_tiled();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap maps[12];
    for (int i = 0; i < 6; ++i) {
        const cuuint64_t dims[2] = {specs[i].inner, specs[i].outer};
        const uint64_t es = mode == 2 ? 4 : 2;
        const cuuint64_t strides[1] = {specs[i].pitch ? specs[i].pitch : specs[i].inner * es};
        const cuuint32_t box[2] = {specs[i].box_inner, specs[i].box_outer};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = encode(&maps[i], mode == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                  2, const_cast<void*>(specs[i].base),
                                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, specs[i].swz,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // Two-box maps of maps 1..3 (weight, dout MN-major, inp). Backward: the
    // MN-major operands as {64 columns, rows, column blocks} with strides
    // {row pitch, 128 bytes}, box {64, 64, 2}: the two 64-column boxes in the
    // order the shared-memory stage holds them. Only where the extent is a
    // multiple of 64, so that the last column block ends at the row's end.
    // Forward: weight rows in boxes of 128 (two 64-row boxes).
    p.wide_maps = 0;
    for (int i = 1; i <= 3; ++i) {
        maps[5 + i] = maps[i];  // placeholder where unused
        const MapSpec& m = specs[i];
        CUresult r = CUDA_SUCCESS;
        if ((mode == 0 || mode == 3) && m.box_inner == 64 && m.inner >= 64 && m.inner % 64 == 0) {
            const cuuint64_t dims[3] = {64, m.outer, m.inner / 64};
            const cuuint64_t strides[2] = {m.pitch ? m.pitch : m.inner * 2, 128};
            const cuuint32_t box[3] = {64, m.box_outer, 2};
            const cuuint32_t estr[3] = {1, 1, 1};
            r = encode(&maps[5 + i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(m.base), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, m.swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else if (mode == 1 && i == 1) {
            const cuuint64_t dims[2] = {m.inner, m.outer};
            const cuuint64_t strides[1] = {m.pitch ? m.pitch : m.inner * 2};
            const cuuint32_t box[2] = {m.box_inner, 2 * m.box_outer};
            const cuuint32_t estr[2] = {1, 1};
            r = encode(&maps[5 + i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(m.base), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, m.swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            continue;
        }
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        if (env_long("MMBWD_WIDE_MAPS", 1)) p.wide_maps |= 1 << (i - 1);
    }
    // Output maps of the bf16 epilogues (maps 4 and 5 give the tensors and
    // their extents): boxes of 32 columns x 32 rows.
    for (int i = 0; i < 2; ++i) {
        maps[9 + i] = maps[4 + i];  // placeholder where unused
        if (mode == 2 || (mode == 1 && i == 1)) continue;  // the forward writes through map 9
        const MapSpec& m = specs[4 + i];
        const cuuint64_t dims[2] = {m.inner, m.outer};
        const cuuint64_t strides[1] = {m.inner * 2};
        const cuuint32_t box[2] = {32, 32};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = encode(&maps[9 + i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(m.base), dims,
                                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // fp32 partial tiles of a split reduction: [half tile][split][128][dw_bn]
    // as rows of dw_bn floats, stored in 32 x 32 boxes (128-byte swizzle).
    // fp32 launches with the dweight product too: its raw A and B in maps 6
    // and 7 (slots the bf16 modes use for other maps)
    if (mode == 2 && pair_specs) {
        for (int i = 0; i < 2; ++i) {
            const MapSpec& m = pair_specs[i];
            const cuuint64_t dims[2] = {m.inner, m.outer};
            const cuuint64_t strides[1] = {m.pitch ? m.pitch : m.inner * 4};
            const cuuint32_t box[2] = {m.box_inner, m.box_outer};
            const cuuint32_t estr[2] = {1, 1};
            const CUresult r = encode(&maps[6 + i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(m.base), dims,
                                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, m.swz,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        }
    }
    maps[11] = maps[0];  // placeholder where unused
    if ((mode == 0 || mode == 3) && plan.splits > 1 && p.partials) {
        const uint64_t rows = static_cast<uint64_t>(2 * plan.dw_tiles_m) * plan.dw_tiles_n * plan.splits * TC_BM;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(plan.dw_bn), rows};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(plan.dw_bn) * 4};
        const cuuint32_t box[2] = {32, 32};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = encode(&maps[11], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.partials, dims, strides, box, estr,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    p.dinp_bn = plan.dinp_bn;
    p.dw_bn = plan.dw_bn;
    p.dinp_tiles_n = plan.dinp_tiles_n;
    p.dw_tiles_n = plan.dw_tiles_n;
    p.dinp_tiles_m = plan.dinp_tiles_m;
    p.dw_tiles_m = plan.dw_tiles_m;
    p.dinp_kb = plan.dinp_kb;
    p.dw_kb = plan.dw_kb;
    p.splits = plan.splits;
    p.kb_per_split = plan.kb_per_split;
    p.n_dw_items = plan.n_dw_items;
    p.n_dinp_items = plan.n_dinp_items;
    p.n_items = plan.n_items;
    p.table = plan.table;
    p.timeout_ns = static_cast<unsigned long long>(env_long("MMBWD_WAIT_TIMEOUT_NS", static_cast<long>(DEFAULT_TIMEOUT_NS)));

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid), 1, 1);
    cfg.blockDim = dim3(mode == 2 ? Smem<2>::THREADS : Smem<0>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_TOTAL;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;  // one CTA pair
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the prologue may start while the previous
    // kernel on the stream finishes; the kernel waits for it before any load.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (mode == 2)
        e = cudaLaunchKernelEx(&cfg, tc_mmbwd_kernel<2>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], p,
                               plan.sched);
    else if (mode == 1)
        e = cudaLaunchKernelEx(&cfg, tc_mmbwd_kernel<1>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], p,
                               plan.sched);
    else if (mode == 3)
        e = cudaLaunchKernelEx(&cfg, tc_mmbwd_kernel<3>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], p,
                               plan.sched);
    else
        e = cudaLaunchKernelEx(&cfg, tc_mmbwd_kernel<0>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], p,
                               plan.sched);
    if (e != cudaSuccess || plan.splits == 1) return e;
    cudaLaunchConfig_t fcfg{};
    fcfg.gridDim = dim3(static_cast<unsigned>(plan.fixup_grid), 1, 1);
    fcfg.blockDim = dim3(256, 1, 1);
    fcfg.stream = stream;
    fcfg.attrs = attr + 1;
    fcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&fcfg, tc_splitk_fixup_kernel, p);
}

}  // namespace

cudaError_t tc_launch(const TcPlan& plan, void* dinp, void* dweight, void* dbias, const void* dout,
                      const void* inp, const void* weight, int64_t BT, int64_t C, int64_t OC, void* ws,
                      cudaStream_t stream, bool sr, uint64_t sr_seed) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const uint64_t bt = static_cast<uint64_t>(BT), c = static_cast<uint64_t>(C), oc = static_cast<uint64_t>(OC);
    const MapSpec specs[6] = {
        {dout, oc, bt, TC_BK, TC_BM, CU_TENSOR_MAP_SWIZZLE_128B},        // dout, K-major A of dinp
        {weight, c, oc, 64, TC_BK, CU_TENSOR_MAP_SWIZZLE_128B},          // weight, MN-major B of dinp
        {dout, oc, bt, 64, TC_BK, CU_TENSOR_MAP_SWIZZLE_128B},           // dout, MN-major A of dweight
        {inp, c, bt, 64, TC_BK, CU_TENSOR_MAP_SWIZZLE_128B},             // inp, MN-major B of dweight
        {dinp, c, bt, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE},           // dinp, L2 prefetch
        {dweight, c, oc, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE},        // dweight, L2 prefetch
    };
    TcParams p{};
    p.BT = BT;
    p.C = C;
    p.OC = OC;
    p.n_dinp = C;
    p.dinp = static_cast<__nv_bfloat16*>(dinp);
    p.dweight = static_cast<__nv_bfloat16*>(dweight);
    p.dbias = static_cast<__nv_bfloat16*>(dbias);
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.partials = plan.splits > 1 ? reinterpret_cast<float*>(w) : nullptr;
    p.bias_partials = plan.splits > 1 ? reinterpret_cast<float*>(w + plan.ws_partials_bytes) : nullptr;
    p.sr = sr ? 1 : 0;
    p.sr_seed = sr_seed;
    // MMBWD_DBIAS=ones: dbias from an extra MMA against a ones tile instead of
    // the bias warps (the variant the page's commented-out Sgemv suggests)
    const char* db = std::getenv("MMBWD_DBIAS");
    p.bias_mma = (dbias && db && std::strcmp(db, "ones") == 0) ? 1 : 0;
    return launch_common(plan, specs, p, sr ? 3 : 0, stream);
}

cudaError_t tc_launch_forward(const TcPlan& plan, void* out, const void* inp, const void* weight, const void* bias,
                              int64_t BT, int64_t C, int64_t OC, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const uint64_t bt = static_cast<uint64_t>(BT), c = static_cast<uint64_t>(C), oc = static_cast<uint64_t>(OC);
    const MapSpec specs[6] = {
        {inp, c, bt, TC_BK, TC_BM, CU_TENSOR_MAP_SWIZZLE_128B},      // inp, K-major A
        {weight, c, oc, TC_BK, 64, CU_TENSOR_MAP_SWIZZLE_128B},      // weight rows, K-major B (64 rows per box)
        {inp, c, bt, TC_BK, TC_BM, CU_TENSOR_MAP_SWIZZLE_128B},      // unused by forward items
        {weight, c, oc, TC_BK, 64, CU_TENSOR_MAP_SWIZZLE_128B},      // unused
        {out, oc, bt, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE},       // unused (nothing read back)
        {out, oc, bt, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE},       // unused
    };
    TcParams p{};
    p.BT = BT;
    p.C = C;
    p.OC = OC;
    p.n_dinp = OC;
    p.fwd_bias = static_cast<const __nv_bfloat16*>(bias);
    p.dinp = static_cast<__nv_bfloat16*>(out);
    return launch_common(plan, specs, p, 1, stream);
}

TcPlan tc_make_plan_x3_pair(int64_t BT, int64_t C, int64_t OC, int num_sms) {
    TcPlan best_pl{};
    // one correction setting for the launch: only where both reductions agree
    if ((OC > TC_X3_CORR_K) != (BT > TC_X3_CORR_K)) return best_pl;
    const int max_pairs = std::max(1, std::min(num_sms / 2, TC_MAX_PAIRS));
    const long force = env_long("MMBWD_TILE_N_X3", 0);
    double best = 1e300;
    for (int bn = 256; bn >= 128; bn -= 128) {
        if (force && bn != force) continue;
        TcPlan c{};
        c.x3 = 1;
        c.x3_corr = OC > TC_X3_CORR_K ? 1 : 0;
        c.dinp_kb = ceil_div_i(OC, TC_BK / 2);
        c.dw_kb = ceil_div_i(BT, TC_BK / 2);
        c.dinp_bn = c.dw_bn = bn;
        c.dinp_tiles_m = ceil_div_i(BT, TC_PAIR_BM);
        c.dw_tiles_m = ceil_div_i(OC, TC_PAIR_BM);
        c.dinp_tiles_n = c.dw_tiles_n = ceil_div_i(C, bn);
        c.n_dinp_items = c.dinp_tiles_m * c.dinp_tiles_n;
        c.n_dw_items = c.dw_tiles_m * c.dw_tiles_n;
        c.n_items = c.n_dinp_items + c.n_dw_items;
        c.splits = 1;
        c.kb_per_split = c.dw_kb;
        if (c.n_items > TC_MAX_SCHED_ITEMS) continue;
        const int pairs = std::max(1, std::min(c.n_items, max_pairs));
        c.grid = 2 * pairs;
        c.table = 1;
        c.est_us = assign_lpt(c, pairs);
        if (c.est_us < best - 1e-9) {
            best = c.est_us;
            best_pl = c;
        }
    }
    return best_pl;
}

namespace {
// Raw fp32 operand of an M x K (or N x K) product side: K-major, 32 K values
// by `rows` rows per box (128-byte swizzle, the high plane's layout), or
// MN-major, 64 M (N) values by 32 K rows per box (plain rows, split in the
// kernel). ld: elements between rows of the tensor.
MapSpec x3_operand(const float* t, bool mn, uint64_t mn_extent, uint64_t k_extent, int64_t ld, uint32_t rows) {
    const uint64_t pitch = static_cast<uint64_t>(ld) * 4;
    if (mn) return MapSpec{t, mn_extent, k_extent, 64, TC_BK / 2, CU_TENSOR_MAP_SWIZZLE_NONE, pitch};
    return MapSpec{t, k_extent, mn_extent, TC_BK / 2, rows, CU_TENSOR_MAP_SWIZZLE_128B, pitch};
}
}  // namespace

cudaError_t tc_launch_x3(const TcPlan& plan, float* D, const float* A, bool a_mn, int64_t lda, const float* B,
                         bool b_mn, int64_t ldb, int64_t M, int64_t N, int64_t K, float* dbias_or_null,
                         cudaStream_t stream) {
    const uint64_t m = static_cast<uint64_t>(M), n = static_cast<uint64_t>(N), k = static_cast<uint64_t>(K);
    const MapSpec a = x3_operand(A, a_mn, m, k, lda, TC_BM), b = x3_operand(B, b_mn, n, k, ldb, 64);
    const MapSpec specs[6] = {
        a, b, a, b,                                                      // (maps 2 and 3 unused)
        {D, n, m, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE, 0},            // D, L2 prefetch of old values
        {D, n, m, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE, 0},            // (dweight slot, unused)
    };
    TcParams p{};
    p.BT = M;
    p.C = K;
    p.OC = K;
    p.n_dinp = N;
    p.x3_corr = K > TC_X3_CORR_K ? 1 : 0;
    p.x3_mn = (a_mn ? 1 : 0) | (b_mn ? 2 : 0);
    p.x3_dbias = a_mn ? dbias_or_null : nullptr;
    p.dinp = reinterpret_cast<__nv_bfloat16*>(D);
    return launch_common(plan, specs, p, 2, stream);
}

cudaError_t tc_launch_x3_pair(const TcPlan& plan, float* dinp, float* dweight, float* dbias, const float* dout,
                              const float* inp, const float* weight, int64_t BT, int64_t C, int64_t OC,
                              cudaStream_t stream) {
    const uint64_t bt = static_cast<uint64_t>(BT), c = static_cast<uint64_t>(C), oc = static_cast<uint64_t>(OC);
    // dinp product (K = OC): A = dout K-major, B = weight MN-major (maps 0 and
    // 1); the outputs (L2 prefetch of old values): maps 4 and 5
    const MapSpec a1 = x3_operand(dout, false, bt, oc, OC, TC_BM), b1 = x3_operand(weight, true, c, oc, C, 64);
    const MapSpec specs[6] = {
        a1, b1, a1, b1,
        {dinp, c, bt, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE, 0},
        {dweight, c, oc, 128, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE, 0},
    };
    // dweight product (K = BT): A = dout^T and B = inp, both MN-major
    const MapSpec pair[2] = {x3_operand(dout, true, oc, bt, OC, TC_BM), x3_operand(inp, true, c, bt, C, 64)};
    TcParams p{};
    p.BT = BT;
    p.C = C;
    p.OC = OC;
    p.n_dinp = C;
    p.x3_corr = plan.x3_corr;
    p.x3_mn = 2 | 4 | 8;
    p.x3_dbias = dbias;
    p.dinp = reinterpret_cast<__nv_bfloat16*>(dinp);
    p.dweight = reinterpret_cast<__nv_bfloat16*>(dweight);
    return launch_common(plan, specs, p, 2, stream, pair);
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

// Internal declarations of the tensor-core kernel (tc_gemm.cu), shared with
// the C-ABI layer and the fp32 tensor-core path. The other kernels' internal
// declarations are in ops.h. Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mmbwd {

// ------------------------------------------------------------ bf16 tensor-core path
// Tile shape of the persistent tcgen05 kernel: a pair of CTAs (a cluster of 2
// on neighbouring SMs) computes a 256 x 256 tile with pair MMAs; each CTA holds
// 128 rows of the fp32 accumulator in its tensor memory and stages its 128
// rows of A and 128 columns of B, 64 elements of K per pipeline stage.
constexpr int TC_BM = 128;       // rows per CTA
constexpr int TC_PAIR_BM = 256;  // rows per CTA pair
constexpr int TC_BN = 256;       // widest tile (N of one MMA); each CTA stages half of the columns
constexpr int TC_BK = 64;
constexpr int TC_STAGES = 6;     // bf16 pipeline stages (32 KB each)
constexpr int TC_STAGES_X3 = 3;  // fp32 three-product stages (64 KB each)

// Wait sites reported in the device status word.
enum WaitSite : int {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_TMEM_EMPTY = 2,
    SITE_MMA_FULL = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_EPI_BIAS_FULL = 5,    // (retired: the bias warps store their sums themselves)
    SITE_BIAS_TMEM_EMPTY = 6,  // (retired)
    SITE_BIAS_FULL = 7,
    SITE_TEARDOWN = 8,
    SITE_SELFTEST = 9,
    SITE_FORWARD_FULL = 10,
    SITE_EPI_OLD = 11,
    SITE_CONV_RAW = 12,  // MODE 2: operand split warps waiting for a raw fp32 stage
    SITE_MMA_CONV = 13,  // MODE 2: MMA issuer waiting for both CTAs' split stages
};

// Schedule of a launch: which work items each CTA pair (a cluster of two CTAs)
// processes, in order (items of pair c: items[start[c] .. start[c+1])). It
// travels in the kernel parameters, so a launch needs no device memory for it.
constexpr int TC_MAX_PAIRS = 128;
constexpr int TC_MAX_SCHED_ITEMS = 3072;
struct TcSchedule {
    uint16_t start[TC_MAX_PAIRS + 1];
    uint16_t items[TC_MAX_SCHED_ITEMS];
};

// Work list of one call: the dweight (TN) items -- dweight tiles times the
// K splits -- and the dinp (NN) tiles, item w < n_dw_items being a dweight
// item. Items are assigned to CTA pairs longest first, each to the pair with
// the least work so far (`table` = 1); when a list is too long for the
// parameter table, pairs take items round-robin instead (`table` = 0).
struct TcPlan {
    int dinp_bn;       // tile width of the dinp product (128 or 256 columns of C)
    int dw_bn;         // tile width of the dweight product
    int dinp_tiles_n;  // ceil(C / dinp_bn)
    int dw_tiles_n;    // ceil(C / dw_bn)
    int dinp_tiles_m;  // ceil(BT / PAIR_BM): row tiles of dinp, one per CTA pair
    int dw_tiles_m;    // ceil(OC / PAIR_BM): row tiles of dweight, one per CTA pair
    int dinp_kb;       // ceil(OC / BK)
    int dw_kb;         // ceil(BT / BK)
    int splits;        // K splits of the dweight product
    int kb_per_split;  // k-blocks per split (the last may have fewer)
    int n_dw_items;    // dw_tiles_m * dw_tiles_n * splits
    int n_dinp_items;  // dinp_tiles_m * dinp_tiles_n
    int n_items;
    int table;         // 1: per-pair item lists in `sched`; 0: round-robin
    int x3;            // fp32 (three tf32 products, operands split in the kernel): tf32 item costs
    int x3_corr;       // fp32: the correction products in their own accumulator
    int grid;          // CTAs (twice the number of CTA pairs)
    double est_us;     // the planner's time estimate
    int fixup_grid;    // CTAs of the split-reduction pass (0 when splits == 1)
    size_t ws_partials_bytes;  // fp32 partial tiles (splits > 1 only)
    size_t ws_bias_bytes;      // fp32 partial bias sums (splits > 1 only)
    size_t ws_bytes() const { return ws_partials_bytes + ws_bias_bytes; }
    int launches() const { return splits > 1 ? 2 : 1; }
    TcSchedule sched;
};

struct TcParams {
    int64_t BT, C, OC;
    // Forward launches (the kernel's forward instantiation) run only "dinp-type"
    // items -- K-major A, rows over BT -- with a K-major B (weight rows) and an
    // overwrite epilogue: out = acc + bias. n_dinp is the N extent and row
    // stride of that product's output: C for the backward (dinp), OC for the
    // forward (out, passed in `dinp`).
    int64_t n_dinp;
    const __nv_bfloat16* fwd_bias;  // may be null
    __nv_bfloat16* dinp;
    __nv_bfloat16* dweight;
    __nv_bfloat16* dbias;  // may be null
    int dinp_bn, dw_bn, dinp_tiles_n, dw_tiles_n;
    int dinp_tiles_m, dw_tiles_m, dinp_kb, dw_kb, splits, kb_per_split;
    int n_dw_items, n_dinp_items, n_items, table;
    float* partials;       // [dw half tile][split][BM][dw_bn]; half tile = 128-row tile x column tile
    float* bias_partials;  // [dw 128-row tile][split][BM]
    unsigned long long timeout_ns;
    int sr;                         // stochastic rounding of the bf16 outputs (backward)
    unsigned long long sr_seed;
    int wide_maps;                  // TC_WIDE_* bits: operands that also have a two-box map
    int bias_mma;                   // dbias from an extra pair MMA against a ones tile (MMBWD_DBIAS=ones)
    int x3_corr;                    // MODE 2: hi.lo + lo.hi in their own accumulator (long K)
    // MODE 2: which raw fp32 operands arrive MN-major (and are transposed in
    // shared memory); the others arrive K-major. Bits: 1 A and 2 B of the
    // dinp-type items, 4 A and 8 B of the dweight items.
    int x3_mn;
    // MODE 2: fp32 dbias (overwritten) = the sums over K of A's rows, formed
    // on the items of column tile 0 whose A arrives MN-major; null: none
    float* x3_dbias;
};

// MODE 2 reductions longer than this keep the two correction products in an
// accumulator of their own (the tensor core rounds each accumulation toward
// zero; see the fp32 path's selection in the C-ABI layer).
constexpr int64_t TC_X3_CORR_K = 2048;

// Operands whose two 64-column halves can arrive in one TMA request.
constexpr int TC_WIDE_WEIGHT = 1;   // weight: B of dinp (backward), B of the forward
constexpr int TC_WIDE_DOUT_MN = 2;  // dout: A of dweight
constexpr int TC_WIDE_INP = 4;      // inp: B of dweight

// Plans (pure functions of the shape and the number of co-resident CTAs,
// twice the resident CTA pairs). Overrides for tuning and tests come from the
// environment: MMBWD_SPLITK (splits), MMBWD_GRID (CTAs, rounded to pairs),
// MMBWD_TILE_N ("dinp,dweight" tile widths); at launch, MMBWD_WIDE_MAPS=0
// loads every 64-column box with its own request.
TcPlan tc_make_plan(int64_t BT, int64_t C, int64_t OC, int num_sms);

// Plan of the forward out (BT x OC) = inp (BT x C) . weight^T (+ bias): only
// dinp-type items, K = C, N = OC.
TcPlan tc_make_plan_forward(int64_t BT, int64_t C, int64_t OC, int num_sms);

// One fp32 product D (M x N, row-major, leading dimension N) += A (M x K) .
// B (N x K)^T from the raw fp32 operands: the kernel splits every staged
// operand into its tf32 value (hi) and exact remainder (lo) in shared memory.
// An operand is K-major (row r of A, or of B, holds K contiguous values,
// leading dimension ld) or MN-major (row k holds the M, or N, contiguous
// values of K index k, leading dimension ld); leading dimensions in elements,
// multiples of 4. dbias_or_null: where A is MN-major, receives the sums of A's
// rows over K (overwritten).
TcPlan tc_make_plan_x3(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t tc_launch_x3(const TcPlan& plan, float* D, const float* A, bool a_mn, int64_t lda, const float* B,
                         bool b_mn, int64_t ldb, int64_t M, int64_t N, int64_t K, float* dbias_or_null,
                         cudaStream_t stream);
// Both fp32 products of the backward in one launch, their items (tiles of
// either product) assigned to CTA pairs longest first:
//   dinp (BT x C) += dout (BT x OC) . weight (OC x C)     A K-major, B MN-major
//   dweight (OC x C) += dout^T (OC x BT) . inp (BT x C)   A and B MN-major
// and dbias (fp32, overwritten, may be null) = the column sums of dout. The
// plan has n_items == 0 where one launch does not fit (then the products go
// to tc_launch_x3 one at a time).
TcPlan tc_make_plan_x3_pair(int64_t BT, int64_t C, int64_t OC, int num_sms);
cudaError_t tc_launch_x3_pair(const TcPlan& plan, float* dinp, float* dweight, float* dbias, const float* dout,
                              const float* inp, const float* weight, int64_t BT, int64_t C, int64_t OC,
                              cudaStream_t stream);
cudaError_t tc_launch_forward(const TcPlan& plan, void* out, const void* inp, const void* weight,
                              const void* bias, int64_t BT, int64_t C, int64_t OC, cudaStream_t stream);

// Launch the tensor-core kernel (and, with split dweight, the fixed-order
// split reduction after it on the same stream). `ws` must hold plan.ws_bytes()
// bytes. `sr`: stochastic rounding of the outputs with `sr_seed` (sr.cuh).
// Returns a cudaError_t.
cudaError_t tc_launch(const TcPlan& plan, void* dinp, void* dweight, void* dbias, const void* dout,
                      const void* inp, const void* weight, int64_t BT, int64_t C, int64_t OC,
                      void* ws, cudaStream_t stream, bool sr = false, uint64_t sr_seed = 0);

size_t tc_smem_bytes();

// How many clusters of `cluster_size` CTAs of the tensor-core kernel can be
// resident at once on the current device (0 if the query fails).
int tc_max_active_clusters(int cluster_size);

// Test hook of the launch functions (defined with the C ABI; see ops.h).
bool take_injected_launch_failure();

// Device status word of the tensor-core translation unit.
cudaError_t tc_read_status(int* code, int* info3, bool reset);
cudaError_t tc_selftest_wait(unsigned long long timeout_ns);

// Driver entry point for tensor-map encoding (resolved through the runtime).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

}  // namespace mmbwd

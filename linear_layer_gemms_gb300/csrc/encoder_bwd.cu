// GPT-2 encoder backward (llm.c llmc/encoder.cuh): dwte[inp[b,t]] += dout[b,t]
// and dwpe[t] += sum over b of dout[b,t], deterministic and without atomics on
// the data.
//
// The page buckets the positions of each token on the host every step (a hash
// map and a sort over host token ids, then two host-to-device copies). Here
// the bucketing stays on the device, in two launches:
//   1. enc_sort_wpe_kernel. A cluster of eight CTAs sorts the keys
//      (token << 15) | position stably by token in their shared memory (LSD
//      radix passes of 4 bits over the token bits, keys moved between the CTAs
//      through the cluster's shared memory), so each token's positions end
//      up contiguous and in increasing order, and writes the sorted keys and,
//      per window of 32 sorted slots, where the run of the window's first slot
//      begins and where the run of its last slot ends.
//      Token ids outside [0, V) are left out and reported in the status word.
//      The other blocks meanwhile form dwpe: one thread per (t, 16-byte
//      vector) sums dout over b in order, adds the old value, rounds once.
//   2. enc_window_kernel: one warp per (window of 32 sorted slots, group of
//      128 channels). The warp sums the window's dout rows in slot order, 16
//      in flight for bf16 and 8 for fp32, cutting at token changes. A token run that lies inside the
//      window is added to its old dwte row and rounded once. A run that
//      crosses a window edge belongs to a token spanning windows wa..wb: each
//      of those windows stores its fp32 partial and counts itself on the
//      token's counter (kept at window wa); the last to arrive adds the
//      partials in window order to the old row. Which warp is last varies,
//      the order of the sum does not, so repeated calls give identical bits.
// The second grid is sized from the upper bound B*T and its warps skip windows
// past the valid count the sort wrote, so the host never waits for the
// device. Both launch with programmatic stream serialization and wait for
// their predecessor before touching global memory.
#include <algorithm>
#include <climits>

#include "../../include/encoder_backward.h"
#include "../../include/mmbwd.h"
#include "ops.h"
#include "ptx.cuh"
#include "sr.cuh"

namespace mmbwd {

// Status word of the encoder kernels: [0] error code (positive), [1] first
// offending position, [2] its token id.
__device__ unsigned int g_enc_status[4];

namespace {

constexpr int ENC_SORT_THREADS = 1024;
// The sort of up to ENC_FAST_MAX positions: one cluster of ENC_CS_CTAS CTAs of
// ENC_CS_THREADS threads.
constexpr int ENC_CS_CTAS = 8;
constexpr int ENC_CS_THREADS = 256;
constexpr int ENC_WIN = 32;  // sorted slots per window (one per lane)
constexpr unsigned ENC_PAD = 0xFFFFFFFFu;
constexpr int ENC_DIGIT_BITS = 4;  // radix digit width per pass
constexpr int ENC_DIGITS = 1 << ENC_DIGIT_BITS;
// (digit, thread) counters, two digits (2k, 2k + 1) packed in the 16-bit halves
// of word k * 1024 + thread
constexpr int ENC_CNT = ENC_DIGITS / 2 * ENC_SORT_THREADS;
constexpr int ENC_CNT_WORDS = ENC_CNT + ENC_CNT / 32;  // with one pad word per 32
constexpr int ENC_CS_CNT = ENC_DIGITS / 2 * ENC_CS_THREADS;  // the same for one CTA of the sorting cluster
constexpr int ENC_CS_CNT_WORDS = ENC_CS_CNT + ENC_CS_CNT / 32;

// Word w, padded so that a warp's 32 threads (one word row each) and a
// thread's 8 consecutive words in the scan both fall in 32 distinct banks.
__device__ __forceinline__ int enc_cnt_at(int w) { return w + (w >> 5); }

__device__ __forceinline__ void enc_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream be scheduled now; it still waits (its
// own griddepcontrol.wait) for this grid to finish before reading anything.
__device__ __forceinline__ void enc_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T>
struct EncElem;
template <>
struct EncElem<float> {
    static constexpr int N = 4;
    __device__ static void add(const uint4& v, float (&a)[4]) {
        a[0] += __uint_as_float(v.x), a[1] += __uint_as_float(v.y);
        a[2] += __uint_as_float(v.z), a[3] += __uint_as_float(v.w);
    }
    __device__ static uint4 add_round(const uint4& old, const float (&s)[4]) {
        return make_uint4(__float_as_uint(__uint_as_float(old.x) + s[0]), __float_as_uint(__uint_as_float(old.y) + s[1]),
                          __float_as_uint(__uint_as_float(old.z) + s[2]), __float_as_uint(__uint_as_float(old.w) + s[3]));
    }
};
template <>
struct EncElem<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    __device__ static void add(const uint4& v, float (&a)[8]) {
        a[0] += lo(v.x), a[1] += hi(v.x), a[2] += lo(v.y), a[3] += hi(v.y);
        a[4] += lo(v.z), a[5] += hi(v.z), a[6] += lo(v.w), a[7] += hi(v.w);
    }
    __device__ static uint32_t rp(uint32_t old, float a, float b) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo(old) + a, hi(old) + b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static uint4 add_round(const uint4& old, const float (&s)[8]) {
        return make_uint4(rp(old.x, s[0], s[1]), rp(old.y, s[2], s[3]), rp(old.z, s[4], s[5]), rp(old.w, s[6], s[7]));
    }
};

// Four channels per lane (8 bytes of bf16 or 16 of fp32), for the window kernel.
template <typename T>
struct EncVec4;
template <>
struct EncVec4<float> {
    using V = uint4;
    __device__ static V zero() { return make_uint4(0u, 0u, 0u, 0u); }
    __device__ static V ld(const float* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ static V ld_plain(const float* p) { return *reinterpret_cast<const uint4*>(p); }
    __device__ static void st(float* p, V v) { *reinterpret_cast<uint4*>(p) = v; }
    __device__ static void add(const V& v, float (&a)[4]) { EncElem<float>::add(v, a); }
    __device__ static V add_round(const V& old, const float (&s)[4]) { return EncElem<float>::add_round(old, s); }
    __device__ static V add_sr(const V& old, const float (&s)[4], uint64_t) { return add_round(old, s); }  // fp32: exact
};
template <>
struct EncVec4<__nv_bfloat16> {
    using V = uint2;
    using E = EncElem<__nv_bfloat16>;
    __device__ static V zero() { return make_uint2(0u, 0u); }
    __device__ static V ld(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
    __device__ static V ld_plain(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
    __device__ static void st(__nv_bfloat16* p, V v) { *reinterpret_cast<uint2*>(p) = v; }
    __device__ static void add(const V& v, float (&a)[4]) {
        a[0] += E::lo(v.x), a[1] += E::hi(v.x), a[2] += E::lo(v.y), a[3] += E::hi(v.y);
    }
    __device__ static V add_round(const V& old, const float (&s)[4]) {
        return make_uint2(E::rp(old.x, s[0], s[1]), E::rp(old.y, s[2], s[3]));
    }
    // Stochastic rounding (sr.cuh): w is the generator word of these four
    // elements (their first index is a multiple of 4).
    __device__ static V add_sr(const V& old, const float (&s)[4], uint64_t w) {
        const float x[4] = {E::lo(old.x) + s[0], E::hi(old.x) + s[1], E::lo(old.y) + s[2], E::hi(old.y) + s[3]};
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = sr::round_bits(x[k], static_cast<uint32_t>(w >> (16 * k)) & 0xFFFFu);
        return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
};

struct EncTables {
    int* meta;           // [0] valid positions; [1..3] B*T, V, C of the problem
    unsigned long long* mb_alt;  // the multi-block sort's second key buffer (B*T > ENC_FAST_MAX)
    int* mb_hist;                // its per-(digit, tile) counts and offsets
    unsigned long long* skeys;  // [B*T] sorted keys (token << 32 | position); invalid slots all ones
    int* win_head;       // [windows] first slot of the run holding the window's first slot
    int* win_tail;       // [windows] last slot of the run holding the window's last slot
    unsigned* arrivals;  // [windows][G] windows done for the token whose run starts in the window
    float* partials;     // [windows][2][C] fp32 sums of a window's first / last run
    int sr;              // bf16 outputs rounded stochastically (sr.cuh) with `seed`
    unsigned long long seed;
};

// Exclusive scan of one value per thread over the block (up to 1024 threads,
// in thread order); returns the thread's prefix and writes the total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = static_cast<int>(threadIdx.x & 31), warp = static_cast<int>(threadIdx.x >> 5);
    const int nw = static_cast<int>(blockDim.x >> 5);
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    if (total) *total = warp_sums[31];
    __syncthreads();
    return before;
}

// dwpe rows, as the blocks after the first of the sort launch: thread v of
// `nthreads` takes vectors v, v + nthreads, ...; dout summed over b in order
// (four loads in flight), added to the old value, rounded once.
template <typename T>
__device__ void enc_wpe_part(T* __restrict__ dwpe, const T* __restrict__ dout, int B, int T_, int C, int64_t v0,
                             int64_t nthreads, int sr, uint64_t seed) {
    using E = EncElem<T>;
    constexpr int N = E::N;
    const int64_t nv = static_cast<int64_t>(T_) * C / N;
    const int64_t row = static_cast<int64_t>(T_) * C;
    for (int64_t v = v0; v < nv; v += nthreads) {
        const int64_t off = v * N;
        float acc[N];
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = 0.f;
        int b = 0;
        for (; b + 4 <= B; b += 4) {
            uint4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = __ldcs(reinterpret_cast<const uint4*>(dout + (b + u) * row + off));
#pragma unroll
            for (int u = 0; u < 4; ++u) E::add(x[u], acc);
        }
        for (; b < B; ++b) E::add(__ldcs(reinterpret_cast<const uint4*>(dout + b * row + off)), acc);
        uint4* dst = reinterpret_cast<uint4*>(dwpe + off);
        if constexpr (sizeof(T) == 2) {
            if (sr) {  // stochastic rounding (sr.cuh): two generator words per 8 elements
                const uint4 o = *dst;
                const uint64_t w0 = sr::word(seed, sr::DWPE, off), w1 = sr::word(seed, sr::DWPE, off + 4);
                const float lo4[4] = {acc[0], acc[1], acc[2], acc[3]}, hi4[4] = {acc[4], acc[5], acc[6], acc[7]};
                const uint2 a = EncVec4<T>::add_sr(make_uint2(o.x, o.y), lo4, w0);
                const uint2 b = EncVec4<T>::add_sr(make_uint2(o.z, o.w), hi4, w1);
                *dst = make_uint4(a.x, a.y, b.x, b.y);
                continue;
            }
        }
        *dst = E::add_round(*dst, acc);
    }
}

// Exclusive max-scan (over lower threads, -1 if none) and exclusive suffix
// min-scan (over higher threads, INT_MAX if none) of one value per thread.
__device__ void block_exclusive_max_and_suffix_min(int mx, int mn, int* warp_sums, int* warp_sums2, int* max_before,
                                                   int* min_after) {
    const int lane = static_cast<int>(threadIdx.x & 31), warp = static_cast<int>(threadIdx.x >> 5);
    const int nw = static_cast<int>(blockDim.x >> 5);
    int x = mx, y = mn;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, x, off);
        const int b = __shfl_down_sync(0xffffffffu, y, off);
        if (lane >= off) x = max(x, a);
        if (lane + off < 32) y = min(y, b);
    }
    if (lane == 31) warp_sums[warp] = x;
    if (lane == 0) warp_sums2[warp] = y;
    __syncthreads();
    if (warp == 0) {
        int a = lane < nw ? warp_sums[lane] : -1, b = lane < nw ? warp_sums2[lane] : INT_MAX;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, a, off);
            const int v = __shfl_down_sync(0xffffffffu, b, off);
            if (lane >= off) a = max(a, u);
            if (lane + off < 32) b = min(b, v);
        }
        warp_sums[lane] = a;   // max over warps 0..lane
        warp_sums2[lane] = b;  // min over warps lane..31
    }
    __syncthreads();
    const int xe = __shfl_up_sync(0xffffffffu, x, 1), ye = __shfl_down_sync(0xffffffffu, y, 1);
    int before = lane > 0 ? xe : -1, after = lane < 31 ? ye : INT_MAX;
    if (warp > 0) before = max(before, warp_sums[warp - 1]);
    if (warp + 1 < nw) after = min(after, warp_sums2[warp + 1]);
    __syncthreads();
    *max_before = before;
    *min_after = after;
}

// The sort, by one cluster of ENC_CS_CTAS CTAs (blocks 0 .. ENC_CS_CTAS - 1 of
// the launch), for NPC = KPL * ENC_CS_THREADS key slots per CTA (the cluster's
// ENC_CS_CTAS * NPC >= B*T). CTA c holds slots c NPC .. c NPC + NPC - 1 in its
// shared memory, thread t the KPL consecutive ones from c NPC + t KPL. The keys
// start in position order (padding, all ones, after the last position), so a
// stable sort by token leaves each token's positions in increasing order and
// the padding last. A pass over a 4-bit digit:
//   - each CTA ranks its keys among its own keys of equal digit: each thread
//     counts its keys per digit in registers (its keys' ranks among its own
//     keys of equal digit come with it) and stores the counts, two digits per
//     word, at word (digit / 2, thread); one block scan over the words (whose
//     16-bit halves add independently) gives each thread its first slot per
//     digit in the CTA's (digit, thread) order, and the CTA's count per digit;
//   - behind a cluster barrier every CTA reads the eight CTAs' counts (shared
//     memory across the cluster) and finds where its keys of each digit start
//     in the whole sorted order: after every key of a lower digit, and after
//     the keys of the same digit held by lower CTAs;
//   - each key is stored straight into the other buffer of the CTA that holds
//     its new slot, and a second cluster barrier makes the stores visible.
// Slot order is (CTA, thread, key) order throughout, so the pass is stable.
// The window tables follow, their cross-CTA parts (the slot before a CTA's
// first, the valid count, the run starts before and after a CTA) read
// through the cluster's shared memory.
// Blocks ENC_CS_CTAS.. form dwpe (enc_wpe_part).
template <typename T, int KPL>
__global__ void __cluster_dims__(ENC_CS_CTAS, 1, 1) __launch_bounds__(ENC_CS_THREADS, 1)
    enc_sort_wpe_kernel(const int32_t* __restrict__ inp, int BT, int V, int passes, int G, EncTables tb,
                        T* __restrict__ dwpe, const T* __restrict__ dout, int B, int T_, int C) {
    enc_grid_wait();
    enc_launch_dependents();
    const int tid = static_cast<int>(threadIdx.x);
    if (blockIdx.x >= ENC_CS_CTAS) {
        enc_wpe_part<T>(dwpe, dout, B, T_, C, static_cast<int64_t>(blockIdx.x - ENC_CS_CTAS) * ENC_CS_THREADS + tid,
                        static_cast<int64_t>(gridDim.x - ENC_CS_CTAS) * ENC_CS_THREADS, tb.sr, tb.seed);
        return;
    }
    constexpr int NPC = KPL * ENC_CS_THREADS;
    constexpr unsigned PADT = ENC_PAD >> 15;  // the padding's token field
    const int c = static_cast<int>(ptx::cluster_ctarank());
    // two key buffers of NPC (the passes alternate), then the packed counters
    extern __shared__ __align__(16) unsigned enc_smem[];
    auto kbuf = [&](int b) { return enc_smem + (b ? NPC : 0); };
    int* cnt = reinterpret_cast<int*>(enc_smem + 2 * NPC);
    __shared__ int warp_sums[32], warp_sums2[32];
    __shared__ int row_start[ENC_DIGITS / 2 + 1];
    __shared__ int dstart[ENC_DIGITS + 1];                // this CTA's first slot of each digit (its own order)
    __shared__ int hist[ENC_DIGITS];                      // this CTA's keys of each digit (read by the cluster)
    __shared__ int allh[ENC_CS_CTAS][ENC_DIGITS];
    __shared__ int gbase[ENC_DIGITS];                     // where this CTA's keys of each digit start
    __shared__ int xinfo[3];  // valid slots of this CTA, its last run start, its first run start (read by the cluster)
    const int i0l = tid * KPL, g0 = c * NPC + i0l;  // this thread's first slot: local, global
    unsigned k[KPL];
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
        const int i = g0 + r;
        unsigned key = ENC_PAD;
        if (i < BT) {
            const int tok = inp[i];
            if (tok >= 0 && tok < V) {
                key = (static_cast<unsigned>(tok) << 15) | static_cast<unsigned>(i);
            } else if (atomicCAS(&g_enc_status[0], 0u, static_cast<unsigned>(-MMBWD_ERR_SHAPE)) == 0u) {
                g_enc_status[1] = static_cast<unsigned>(i);
                g_enc_status[2] = static_cast<unsigned>(tok);
            }
        }
        k[r] = key;
    }
    int cur = 0;
    for (int pass = 0; pass < passes; ++pass) {
        const int sh = 15 + pass * ENC_DIGIT_BITS;
        if (pass > 0) {
#pragma unroll
            for (int r = 0; r < KPL; ++r) k[r] = kbuf(cur)[i0l + r];
        }
        // per-thread digit counts in 8-bit fields (digits 0-7 in c0, 8-15 in
        // c1); a key's rank is its digit's count before it
        uint64_t c0 = 0, c1 = 0;
        int rank[KPL];
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
            const unsigned d = (k[r] >> sh) & (ENC_DIGITS - 1);
            const int f = 8 * static_cast<int>(d & 7u);
            rank[r] = static_cast<int>((((d & 8u) ? c1 : c0) >> f) & 0xFFu);
            if (d & 8u) c1 += uint64_t(1) << f;
            else c0 += uint64_t(1) << f;
        }
#pragma unroll
        for (int kk = 0; kk < ENC_DIGITS / 2; ++kk) {
            const uint64_t cw = kk < 4 ? c0 : c1;
            const int f = 16 * (kk & 3);
            cnt[enc_cnt_at(kk * ENC_CS_THREADS + tid)] =
                static_cast<int>(((cw >> f) & 0xFFu) | (((cw >> (f + 8)) & 0xFFu) << 16));
        }
        __syncthreads();
        {
            int loc[ENC_DIGITS / 2];
            int sum = 0;
#pragma unroll
            for (int q = 0; q < ENC_DIGITS / 2; ++q) {
                loc[q] = cnt[enc_cnt_at(tid * (ENC_DIGITS / 2) + q)];
                sum += loc[q];
            }
            int total = 0;
            int before = block_exclusive_scan(sum, warp_sums, &total);
            if ((tid & (ENC_CS_THREADS / (ENC_DIGITS / 2) - 1)) == 0)
                row_start[tid / (ENC_CS_THREADS / (ENC_DIGITS / 2))] = before;
            if (tid == 0) row_start[ENC_DIGITS / 2] = total;
#pragma unroll
            for (int q = 0; q < ENC_DIGITS / 2; ++q) {
                cnt[enc_cnt_at(tid * (ENC_DIGITS / 2) + q)] = before;
                before += loc[q];
            }
        }
        __syncthreads();
        // this CTA's first slot of digit d: every key of a lower digit (the two
        // halves of the word-row prefixes hold the even and the odd digits)
        if (tid <= ENC_DIGITS) {
            const int d = tid;
            int st = NPC;
            if (d < ENC_DIGITS) {
                const unsigned rs = static_cast<unsigned>(row_start[d >> 1]), rs1 = static_cast<unsigned>(row_start[(d >> 1) + 1]);
                st = static_cast<int>((d & 1) ? (rs >> 16) + (rs1 & 0xFFFFu) : (rs & 0xFFFFu) + (rs >> 16));
            }
            dstart[d] = st;
        }
        __syncthreads();
        if (tid < ENC_DIGITS) hist[tid] = dstart[tid + 1] - dstart[tid];
        ptx::cluster_sync();  // every CTA's counts are visible
        if (tid < ENC_CS_CTAS * ENC_DIGITS) {
            const int cc = tid / ENC_DIGITS, d = tid % ENC_DIGITS;
            allh[cc][d] = static_cast<int>(ptx::ld_dsmem_u32(ptx::mapa(ptx::smem_u32(&hist[d]), static_cast<uint32_t>(cc))));
        }
        __syncthreads();
        if (tid < ENC_DIGITS) {
            const int d = tid;
            int b = 0;
            for (int dd = 0; dd < d; ++dd)
                for (int cc = 0; cc < ENC_CS_CTAS; ++cc) b += allh[cc][dd];
            for (int cc = 0; cc < c; ++cc) b += allh[cc][d];
            gbase[d] = b;
        }
        __syncthreads();
        const uint32_t nb = ptx::smem_u32(kbuf(cur ^ 1));
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
            const unsigned d = (k[r] >> sh) & (ENC_DIGITS - 1);
            const int kk = static_cast<int>(d >> 1);
            const unsigned pw = static_cast<unsigned>(cnt[enc_cnt_at(kk * ENC_CS_THREADS + tid)]);
            const unsigned rs = static_cast<unsigned>(row_start[kk]), rs1 = static_cast<unsigned>(row_start[kk + 1]);
            const unsigned first = (d & 1u) ? (pw >> 16) + (rs1 & 0xFFFFu) : (pw & 0xFFFFu) + (rs >> 16);
            const int g = gbase[d] + static_cast<int>(first) + rank[r] - dstart[d];  // the key's new slot
            ptx::st_dsmem_u32(ptx::mapa(nb + 4u * static_cast<uint32_t>(g % NPC), static_cast<uint32_t>(g / NPC)), k[r]);
        }
        ptx::cluster_sync();  // the stored keys are visible; this CTA's buffers are free again
        cur ^= 1;
    }
    unsigned* keys = kbuf(cur);
    if (passes == 0) {  // V == 0: every key is padding and stays where it is
#pragma unroll
        for (int r = 0; r < KPL; ++r) keys[i0l + r] = k[r];
        ptx::cluster_sync();  // (the CTA after reads this CTA's last slot)
    }

    // Each thread takes its KPL consecutive sorted slots with the token of the
    // slot before (in the CTA before for a CTA's first slot).
    unsigned tk[KPL];
#pragma unroll
    for (int r = 0; r < KPL; ++r) tk[r] = keys[i0l + r] >> 15;
    unsigned tk_prev = PADT;
    if (tid > 0)
        tk_prev = keys[i0l - 1] >> 15;
    else if (c > 0)
        tk_prev = ptx::ld_dsmem_u32(ptx::mapa(ptx::smem_u32(&keys[NPC - 1]), static_cast<uint32_t>(c - 1))) >> 15;
    int nvalid_local = 0;
#pragma unroll
    for (int r = 0; r < KPL; ++r) nvalid_local += tk[r] != PADT;
    // run starts (a valid slot whose token differs from the slot before's)
    int first_start = INT_MAX, last_start = -1;
    bool start0 = false;
#pragma unroll
    for (int r = KPL - 1; r >= 0; --r) {
        const int i = g0 + r;
        const bool st = tk[r] != PADT && (i == 0 || tk[r] != (r > 0 ? tk[r - 1] : tk_prev));
        if (st) {
            first_start = i;
            if (last_start < 0) last_start = i;
        }
        if (r == 0) start0 = st;
    }
    if (tid == 0) {
        xinfo[1] = -1;
        xinfo[2] = INT_MAX;
    }
    int cta_valid = 0;
    block_exclusive_scan(nvalid_local, warp_sums, &cta_valid);  // (its barriers order the stores above)
    if (last_start >= 0) atomicMax(&xinfo[1], last_start);
    if (first_start < INT_MAX) atomicMin(&xinfo[2], first_start);
    if (tid == 0) xinfo[0] = cta_valid;
    int open_start = -1, next_start = INT_MAX;
    block_exclusive_max_and_suffix_min(last_start, first_start, warp_sums, warp_sums2, &open_start, &next_start);
    ptx::cluster_sync();  // every CTA's valid count and run starts are visible
    int nvalid = 0;
    for (int cc = 0; cc < ENC_CS_CTAS; ++cc) {
        const uint32_t a = ptx::smem_u32(xinfo);
        nvalid += static_cast<int>(ptx::ld_dsmem_u32(ptx::mapa(a, static_cast<uint32_t>(cc))));
        if (cc < c)
            open_start = max(open_start, static_cast<int>(ptx::ld_dsmem_u32(ptx::mapa(a + 4u, static_cast<uint32_t>(cc)))));
        if (cc > c)
            next_start = min(next_start, static_cast<int>(ptx::ld_dsmem_u32(ptx::mapa(a + 8u, static_cast<uint32_t>(cc)))));
    }
    for (int i = tid; i < NPC; i += ENC_CS_THREADS) {  // coalesced; (token, position) widened to 32 + 32 bits
        const int gi = c * NPC + i;
        if (gi < nvalid) tb.skeys[gi] = (static_cast<unsigned long long>(keys[i] >> 15) << 32) | (keys[i] & 0x7FFFu);
    }
    // the run holding a window's first slot starts at the largest start at or
    // before it, the run holding its last slot ends before the smallest start
    // after it
    if ((g0 & (ENC_WIN - 1)) == 0 && g0 < nvalid) tb.win_head[g0 / ENC_WIN] = start0 ? g0 : open_start;
    const int ilast = g0 + KPL - 1;
    if (((ilast + 1) & (ENC_WIN - 1)) == 0 && ilast < nvalid) tb.win_tail[ilast / ENC_WIN] = min(next_start, nvalid) - 1;
    const int nwin_g = (nvalid + ENC_WIN - 1) / ENC_WIN * G;
    for (int e = c * ENC_CS_THREADS + tid; e < nwin_g; e += ENC_CS_CTAS * ENC_CS_THREADS) tb.arrivals[e] = 0u;
    if (c == 0 && tid == 0) {
        tb.meta[0] = nvalid;
        tb.meta[1] = BT;  // the problem these tables describe
        tb.meta[2] = V;
        tb.meta[3] = C;
    }
    ptx::cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// Finishes one run that crosses a window edge (see the file comment), the
// token's windows being span.x..span.y: stores this window's partial (slot q:
// 0 for the run entering at the window's first slot, 1 for the run leaving at
// its last), counts the window on the token's counter, and if it is the last
// of windows wa..wb clears the counter and adds their partials in window order
// (window wa's slot 1, then slot 0 of the others) to the old dwte row.
// Warp-uniform.
template <typename T>
__device__ void enc_cross_run(T* __restrict__ dwte, const EncTables& tb, int C, int c, bool active, int lane, int w,
                              int g, int G, int q, int2 span, unsigned tok, const float (&acc)[4],
                              typename EncVec4<T>::V old) {
    using EV = EncVec4<T>;
    constexpr int PB = 16;  // partials in flight
    const int wa = span.x, wb = span.y, nw = wb - wa + 1;
    if (active)
        __stcg(reinterpret_cast<float4*>(tb.partials + (static_cast<int64_t>(w) * 2 + q) * C + c),
               make_float4(acc[0], acc[1], acc[2], acc[3]));
    __threadfence();
    __syncwarp();
    unsigned done = 0;
    const int64_t ci = static_cast<int64_t>(wa) * G + g;
    if (lane == 0) done = atomicAdd(&tb.arrivals[ci], 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != static_cast<unsigned>(nw - 1)) return;  // not the last window of the token
    if (lane == 0) tb.arrivals[ci] = 0u;  // every window has counted: cleared for the next call with this plan
    if (!active) return;
    __threadfence();
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < nw; k += PB) {
        float4 pv[PB];
#pragma unroll
        for (int u = 0; u < PB; ++u) {
            const int64_t idx = (static_cast<int64_t>(wa + k + u) * 2 + (k + u == 0 ? 1 : 0)) * C + c;
            pv[u] = k + u < nw ? __ldcg(reinterpret_cast<const float4*>(tb.partials + idx))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < PB; ++u)
            if (k + u < nw) sum[0] += pv[u].x, sum[1] += pv[u].y, sum[2] += pv[u].z, sum[3] += pv[u].w;
    }
    const int64_t e = static_cast<int64_t>(tok) * C + c;
    EV::st(dwte + e, tb.sr ? EV::add_sr(old, sum, sr::word(tb.seed, sr::DWTE, e)) : EV::add_round(old, sum));
}

// One warp per (window of 32 sorted slots, group of 128 channels); lane l
// holds slot 32 w + l and channels 4 l..4 l + 3 of the group. Runs of equal
// tokens are cut with one ballot. The rows are summed in slot order, RB at a
// time (16 for bf16, 8 for fp32: 4 KB per warp in flight, with every warp of
// the grid resident at once), with the old dwte row of every run that ends in
// the batch loaded alongside.
// Loads that do not depend on each other are issued together (the keys are
// read before the valid count is known, at indexes clamped to the table).
// Lanes past C take part in the shuffles only.
// One-dimensional grid of blocks of GPB = blockDim / 32 warps: blocks
// [0, nwin ngb) are window blocks, ngb = ceil(G / GPB) per window, block b
// serving window b / ngb with warp k taking channel group (b mod ngb) GPB + k,
// so that the warps reading the slices of the same dout and dwte rows run side
// by side; `wpe_blocks` more blocks form dwpe (a planned run, whose sort launch
// had none). The tables must describe this problem (the sort records B*T, V
// and C beside them); otherwise the status word reports it and nothing is
// written.
template <typename T>
__global__ void __launch_bounds__(256, 2) enc_window_kernel(T* __restrict__ dwte, T* __restrict__ dwpe,
                                                           const T* __restrict__ dout, int C, int BT, int B, int T_,
                                                           int V, int nwin, int G, int wpe_blocks, EncTables tb) {
    using EV = EncVec4<T>;
    using V4 = typename EV::V;
    constexpr int RB = sizeof(T) == 2 ? 16 : 8;  // rows in flight
    constexpr unsigned NONE = 0xFFFFFFFFu;
    constexpr unsigned long long NONE64 = ~0ull;
    enc_grid_wait();
    enc_launch_dependents();
    const int bid = static_cast<int>(blockIdx.x);
    if (tb.meta[1] != BT || tb.meta[2] != V || tb.meta[3] != C) {  // tables of another problem
        if (threadIdx.x == 0 && atomicCAS(&g_enc_status[0], 0u, static_cast<unsigned>(-MMBWD_ERR_SHAPE)) == 0u) {
            g_enc_status[1] = 0xFFFFFFFFu;
            g_enc_status[2] = static_cast<unsigned>(tb.meta[1]);
        }
        return;
    }
    const int gpb = static_cast<int>(blockDim.x >> 5), ngb = (G + gpb - 1) / gpb;
    if (bid >= nwin * ngb) {
        enc_wpe_part<T>(dwpe, dout, B, T_, C, static_cast<int64_t>(bid - nwin * ngb) * blockDim.x + threadIdx.x,
                        static_cast<int64_t>(wpe_blocks) * blockDim.x, tb.sr, tb.seed);
        return;
    }
    const int nvalid = tb.meta[0];
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int w = bid / ngb;
    const int g = (bid - w * ngb) * gpb + warp;
    if (g >= G) return;  // the last group block of a window may be partly empty
    const int base = w * ENC_WIN;
    if (base >= BT) return;
    const int c = (g * 32 + lane) * 4;
    const bool active = c < C;
    const unsigned long long key = tb.skeys[min(base + lane, BT - 1)];
    const unsigned long long pkey = base > 0 ? tb.skeys[base - 1] : NONE64;
    const unsigned long long nkey = base + ENC_WIN < BT ? tb.skeys[base + ENC_WIN] : NONE64;
    const int hstart = tb.win_head[w], tend = tb.win_tail[w];  // read only where defined (below)
    if (base >= nvalid) return;
    const int nv = min(ENC_WIN, nvalid - base);
    const bool valid = lane < nv;
    const unsigned tok = static_cast<unsigned>(key >> 32);
    unsigned ptok = __shfl_up_sync(0xffffffffu, tok, 1);
    if (lane == 0) ptok = base > 0 ? static_cast<unsigned>(pkey >> 32) : NONE;
    const unsigned smask = __ballot_sync(0xffffffffu, valid && tok != ptok);  // run starts
    const unsigned tok0 = __shfl_sync(0xffffffffu, tok, 0), tokl = __shfl_sync(0xffffffffu, tok, nv - 1);
    const bool head_cross = (smask & 1u) == 0;  // the first run began in an earlier window
    const bool tail_cross = nv == ENC_WIN && base + ENC_WIN < nvalid && static_cast<unsigned>(nkey >> 32) == tokl;
    // windows wa..wb of the crossing runs: the head run's began at win_head; it
    // ends here unless it fills the window and crosses the tail too, where its
    // end and the tail run's end are win_tail
    const int whead = head_cross ? hstart / ENC_WIN : w;
    const int wtail = tail_cross ? tend / ENC_WIN : w;
    const int2 hspan = make_int2(whead, (smask == 0u && tail_cross) ? wtail : w);
    const int2 tspan = make_int2(w, wtail);
    // run ends: slot j ends a run where slot j + 1 starts one or j is the last
    const unsigned vmask = nv == ENC_WIN ? 0xffffffffu : (1u << nv) - 1u;
    const unsigned emask = ((smask >> 1) | (1u << (nv - 1))) & vmask;

    float acc[4] = {0.f, 0.f, 0.f, 0.f}, hacc[4] = {0.f, 0.f, 0.f, 0.f}, tacc[4] = {0.f, 0.f, 0.f, 0.f};
    V4 hold = EV::zero(), told = EV::zero();
#pragma unroll 1
    for (int j0 = 0; j0 < ENC_WIN; j0 += RB) {
        if (j0 < nv) {  // warp-uniform
            V4 v[RB], o[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                constexpr unsigned one = 1u;
                const int j = j0 + u;  // compile-time slot
                const unsigned long long kj = __shfl_sync(0xffffffffu, key, j);
                const int64_t r = static_cast<int64_t>(kj & 0xFFFFFFFFull), t = static_cast<int64_t>(kj >> 32);
                v[u] = (active && ((vmask >> j) & one)) ? EV::ld(dout + r * C + c) : EV::zero();
                o[u] = (active && ((emask >> j) & one)) ? EV::ld_plain(dwte + t * C + c) : EV::zero();
            }
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int j = j0 + u;
                if ((vmask >> j) & 1u) {  // warp-uniform
                    EV::add(v[u], acc);
                    if ((emask >> j) & 1u) {  // run ends at slot j (warp-uniform)
                        const int64_t t = static_cast<int64_t>(__shfl_sync(0xffffffffu, key, j) >> 32);
                        const unsigned below = j == 31 ? 0xffffffffu : (2u << j) - 1u;
                        const bool is_head = head_cross && (smask & below) == 0;
                        const bool is_tail = tail_cross && j == nv - 1;
                        if (is_head) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) hacc[e] = acc[e];
                            hold = o[u];
                        } else if (is_tail) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) tacc[e] = acc[e];
                            told = o[u];
                        } else if (active) {
                            EV::st(dwte + t * C + c, tb.sr ? EV::add_sr(o[u], acc, sr::word(tb.seed, sr::DWTE, t * C + c))
                                                           : EV::add_round(o[u], acc));
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[e] = 0.f;
                    }
                }
            }
        }
    }
    // A run that fills the window and crosses both edges is the head run.
    if (head_cross) enc_cross_run<T>(dwte, tb, C, c, active, lane, w, g, G, 0, hspan, tok0, hacc, hold);
    if (tail_cross && smask != 0u)
        enc_cross_run<T>(dwte, tb, C, c, active, lane, w, g, G, 1, tspan, tokl, tacc, told);
}

// ---------------------------------------------------------------------------
// The sort for more than ENC_FAST_MAX positions: a stable LSD radix sort of the
// 64-bit keys (token << 32 | position) on 4-bit digits of the token, spread
// over tiles of MB_TILE keys, three launches a pass and no wait between blocks:
//   hist     every tile counts its keys per digit (H[digit][tile]);
//   scan     one block turns H into exclusive prefixes in (digit, tile) order:
//            where each tile's keys of each digit start in the output;
//   scatter  every tile ranks its keys stably by digit (the packed per-thread
//            counters of the cluster sort) and writes them there.
// The initial keys are in position order, so the positions of a token end up
// in increasing order. A last launch derives the window tables from the
// sorted keys by binary search (a run is the range of one token).
constexpr int ENC_FAST_MAX = 16384;  // positions the cluster sort takes
constexpr int MB_KPT = 8;            // keys per thread of a tile
constexpr int MB_TILE = MB_KPT * ENC_SORT_THREADS;

__device__ __forceinline__ unsigned mb_digit(unsigned long long k, int sh) {
    return static_cast<unsigned>(k >> (32 + sh)) & (ENC_DIGITS - 1);
}

// Keys in position order; ids outside [0, V) become padding (all ones, sorted
// last) and are reported in the status word.
__global__ void __launch_bounds__(256) enc_mb_keys_kernel(const int32_t* __restrict__ inp, int BT, int V,
                                                          unsigned long long* __restrict__ dst) {
    enc_grid_wait();
    enc_launch_dependents();
    for (int i = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); i < BT;
         i += static_cast<int>(gridDim.x * blockDim.x)) {
        const int tok = inp[i];
        unsigned long long key = ~0ull;
        if (tok >= 0 && tok < V) {
            key = (static_cast<unsigned long long>(tok) << 32) | static_cast<unsigned>(i);
        } else if (atomicCAS(&g_enc_status[0], 0u, static_cast<unsigned>(-MMBWD_ERR_SHAPE)) == 0u) {
            g_enc_status[1] = static_cast<unsigned>(i);
            g_enc_status[2] = static_cast<unsigned>(tok);
        }
        dst[i] = key;
    }
}

// H[d * ntiles + tile] = keys of the tile with digit d (integer counts).
__global__ void __launch_bounds__(ENC_SORT_THREADS) enc_mb_hist_kernel(const unsigned long long* __restrict__ src,
                                                                      int BT, int sh, int ntiles, int* __restrict__ H) {
    enc_grid_wait();
    enc_launch_dependents();
    __shared__ int cnt[ENC_DIGITS];
    const int tid = static_cast<int>(threadIdx.x), lane = tid & 31;
    if (tid < ENC_DIGITS) cnt[tid] = 0;
    __syncthreads();
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * MB_TILE;
    int mine[ENC_DIGITS];
#pragma unroll
    for (int d = 0; d < ENC_DIGITS; ++d) mine[d] = 0;
#pragma unroll
    for (int r = 0; r < MB_KPT; ++r) {
        const int64_t i = i0 + static_cast<int64_t>(r) * ENC_SORT_THREADS + tid;  // coalesced
        const bool in = i < BT;
        const unsigned d = in ? mb_digit(src[i], sh) : 0u;
#pragma unroll
        for (int dd = 0; dd < ENC_DIGITS; ++dd) mine[dd] += __popc(__ballot_sync(0xffffffffu, in && d == dd));
    }
    if (lane < ENC_DIGITS) {
        int v = 0;
#pragma unroll
        for (int dd = 0; dd < ENC_DIGITS; ++dd) v = dd == lane ? mine[dd] : v;
        atomicAdd(&cnt[lane], v);
    }
    __syncthreads();
    if (tid < ENC_DIGITS) H[tid * ntiles + blockIdx.x] = cnt[tid];
}

// In place: H becomes its exclusive prefix sums (one block, in index order).
__global__ void __launch_bounds__(ENC_SORT_THREADS) enc_mb_scan_kernel(int* __restrict__ H, int n) {
    enc_grid_wait();
    enc_launch_dependents();
    __shared__ int warp_sums[32];
    int carry = 0;
    for (int b0 = 0; b0 < n; b0 += ENC_SORT_THREADS) {
        const int i = b0 + static_cast<int>(threadIdx.x);
        const int v = i < n ? H[i] : 0;
        int total = 0;
        const int before = block_exclusive_scan(v, warp_sums, &total);
        if (i < n) H[i] = carry + before;
        carry += total;
    }
}

// Stable scatter of one tile by the digit at `sh`: thread t owns keys
// i0 + t*MB_KPT .. +MB_KPT-1 (keys past BT take no part); their slots in the
// tile sorted by digit come from the packed counters as in the cluster
// sort, and O (the scanned H) gives where the tile's keys of each digit go.
__global__ void __launch_bounds__(ENC_SORT_THREADS, 1)
    enc_mb_scatter_kernel(const unsigned long long* __restrict__ src, unsigned long long* __restrict__ dst, int BT,
                          int sh, int ntiles, const int* __restrict__ O) {
    enc_grid_wait();
    enc_launch_dependents();
    __shared__ int cnt[ENC_CNT_WORDS];
    __shared__ int warp_sums[32];
    __shared__ int row_start[ENC_DIGITS / 2 + 1];
    __shared__ int gofs[ENC_DIGITS];
    const int tid = static_cast<int>(threadIdx.x);
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * MB_TILE + static_cast<int64_t>(tid) * MB_KPT;
    if (tid < ENC_DIGITS) gofs[tid] = O[tid * ntiles + blockIdx.x];
    unsigned long long k[MB_KPT];
    unsigned dg[MB_KPT];
    int rank[MB_KPT];
    uint64_t c0 = 0, c1 = 0;
#pragma unroll
    for (int r = 0; r < MB_KPT; ++r) {
        const bool in = i0 + r < BT;
        k[r] = in ? src[i0 + r] : ~0ull;
        dg[r] = mb_digit(k[r], sh);
        const int f = 8 * static_cast<int>(dg[r] & 7u);
        rank[r] = static_cast<int>((((dg[r] & 8u) ? c1 : c0) >> f) & 0xFFu);
        if (in) {
            if (dg[r] & 8u) c1 += uint64_t(1) << f;
            else c0 += uint64_t(1) << f;
        }
    }
#pragma unroll
    for (int kk = 0; kk < ENC_DIGITS / 2; ++kk) {
        const uint64_t c = kk < 4 ? c0 : c1;
        const int f = 16 * (kk & 3);
        cnt[enc_cnt_at(kk * ENC_SORT_THREADS + tid)] = static_cast<int>(((c >> f) & 0xFFu) | (((c >> (f + 8)) & 0xFFu) << 16));
    }
    __syncthreads();
    {
        int loc[ENC_DIGITS / 2];
        int sum = 0;
#pragma unroll
        for (int q = 0; q < ENC_DIGITS / 2; ++q) {
            loc[q] = cnt[enc_cnt_at(tid * (ENC_DIGITS / 2) + q)];
            sum += loc[q];
        }
        int total = 0;
        int before = block_exclusive_scan(sum, warp_sums, &total);
        if ((tid & (ENC_SORT_THREADS / (ENC_DIGITS / 2) - 1)) == 0)
            row_start[tid / (ENC_SORT_THREADS / (ENC_DIGITS / 2))] = before;
        if (tid == 0) row_start[ENC_DIGITS / 2] = total;
#pragma unroll
        for (int q = 0; q < ENC_DIGITS / 2; ++q) {
            cnt[enc_cnt_at(tid * (ENC_DIGITS / 2) + q)] = before;
            before += loc[q];
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < MB_KPT; ++r) {
        if (i0 + r >= BT) continue;
        const unsigned d = dg[r];
        const int kk = static_cast<int>(d >> 1);
        const unsigned pw = static_cast<unsigned>(cnt[enc_cnt_at(kk * ENC_SORT_THREADS + tid)]);
        const unsigned rs = static_cast<unsigned>(row_start[kk]), rs1 = static_cast<unsigned>(row_start[kk + 1]);
        // the tile's first slot of digit d and this key's slot in the sorted tile
        const unsigned dstart = (d & 1u) ? (rs >> 16) + (rs1 & 0xFFFFu) : (rs & 0xFFFFu) + (rs >> 16);
        const unsigned first = (d & 1u) ? (pw >> 16) + (rs1 & 0xFFFFu) : (pw & 0xFFFFu) + (rs >> 16);
        dst[gofs[d] + static_cast<int64_t>(first + rank[r] - dstart)] = k[r];
    }
}

__device__ __forceinline__ int mb_lower_bound(const unsigned long long* keys, int n, unsigned tok) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<unsigned>(keys[mid] >> 32) < tok) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Window tables from the sorted keys: valid count (the first padding key),
// per window of 32 slots where the run (token) of its first slot begins and
// where the run of its last slot ends, the problem's sizes, cleared counters.
__global__ void __launch_bounds__(256) enc_mb_tables_kernel(int BT, int V, int C, int G, EncTables tb) {
    enc_grid_wait();
    enc_launch_dependents();
    const int nvalid = mb_lower_bound(tb.skeys, BT, 0xFFFFFFFFu);
    const int nwin = (nvalid + ENC_WIN - 1) / ENC_WIN;
    const int stride = static_cast<int>(gridDim.x * blockDim.x);
    const int g0 = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    for (int w = g0; w < nwin; w += stride) {
        const int base = w * ENC_WIN, last = min(base + ENC_WIN, nvalid) - 1;
        tb.win_head[w] = mb_lower_bound(tb.skeys, nvalid, static_cast<unsigned>(tb.skeys[base] >> 32));
        const unsigned tl = static_cast<unsigned>(tb.skeys[last] >> 32);
        tb.win_tail[w] = (tl == 0xFFFFFFFEu ? nvalid : mb_lower_bound(tb.skeys, nvalid, tl + 1u)) - 1;
    }
    for (int e = g0; e < nwin * G; e += stride) tb.arrivals[e] = 0u;
    if (g0 == 0) {
        tb.meta[0] = nvalid;
        tb.meta[1] = BT;
        tb.meta[2] = V;
        tb.meta[3] = C;
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

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace {

int enc_groups(int64_t C, int N) { return static_cast<int>((C / N + 31) / 32); }

template <typename T>
const void* enc_sort_fn(int kpl) {
    switch (kpl) {
        case 1: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 1>);
        case 2: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 2>);
        case 4: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 4>);
        default: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 8>);
    }
}

}  // namespace

namespace {

// The tables of one problem, laid out from `base`: meta, sorted keys, the two
// per-window tables, the per-(window, channel group) counters. Returns the
// bytes they take.
size_t enc_tables_layout(uint8_t* base, int64_t BT, int64_t C, EncTables* tb) {
    const size_t n = static_cast<size_t>(BT), nwin = (n + ENC_WIN - 1) / ENC_WIN;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + off : nullptr;
        off += a256(bytes);
        return p;
    };
    uint8_t* meta = take(4 * 4);
    uint8_t* skeys = take(n * 8);
    uint8_t* whead = take(nwin * 4);
    uint8_t* wtail = take(nwin * 4);
    uint8_t* arr = take(nwin * static_cast<size_t>(enc_groups(C, 4)) * 4);
    const bool mb = BT > ENC_FAST_MAX;
    uint8_t* alt = mb ? take(n * 8) : nullptr;
    uint8_t* hist = mb ? take(static_cast<size_t>(ENC_DIGITS) * ((n + MB_TILE - 1) / MB_TILE) * 4) : nullptr;
    if (tb) {
        tb->mb_alt = reinterpret_cast<unsigned long long*>(alt);
        tb->mb_hist = reinterpret_cast<int*>(hist);
        tb->meta = reinterpret_cast<int*>(meta);
        tb->skeys = reinterpret_cast<unsigned long long*>(skeys);
        tb->win_head = reinterpret_cast<int*>(whead);
        tb->win_tail = reinterpret_cast<int*>(wtail);
        tb->arrivals = reinterpret_cast<unsigned*>(arr);
    }
    return off;
}

size_t enc_partials_bytes(int64_t BT, int64_t C) {
    const size_t nwin = (static_cast<size_t>(BT) + ENC_WIN - 1) / ENC_WIN;
    return a256(nwin * 2 * static_cast<size_t>(C) * 4);
}

// The multi-block sort (B*T > ENC_FAST_MAX) and the window tables: keys,
// then per pass hist, scan and scatter (the buffers alternate so that the last
// pass writes tb.skeys), then the tables.
cudaError_t enc_mb_sort_launch(const int32_t* inp, int BT, int64_t V, int64_t C, const EncTables& tb,
                               cudaStream_t stream) {
    int token_bits = 0;
    while ((int64_t(1) << token_bits) <= V) ++token_bits;
    const int passes = (token_bits + ENC_DIGIT_BITS - 1) / ENC_DIGIT_BITS;
    int ntiles = (BT + MB_TILE - 1) / MB_TILE, BTi = BT, Vi = static_cast<int>(V), Ci = static_cast<int>(C);
    int G = enc_groups(C, 4);
    unsigned long long* src = (passes % 2 == 0) ? tb.skeys : tb.mb_alt;
    const int kblocks = std::max(1, std::min((BT + 255) / 256, 4096));
    {
        void* args[] = {const_cast<int32_t**>(&inp), &BTi, &Vi, &src};
        cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&enc_mb_keys_kernel), dim3(kblocks), dim3(256), 0,
                                   stream, args);
        if (e != cudaSuccess) return e;
    }
    int* H = tb.mb_hist;
    int nh = ENC_DIGITS * ntiles;
    for (int pass = 0; pass < passes; ++pass) {
        int sh = pass * ENC_DIGIT_BITS;
        unsigned long long* dst = src == tb.skeys ? tb.mb_alt : tb.skeys;
        void* hargs[] = {&src, &BTi, &sh, &ntiles, &H};
        cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&enc_mb_hist_kernel), dim3(ntiles),
                                   dim3(ENC_SORT_THREADS), 0, stream, hargs);
        if (e != cudaSuccess) return e;
        void* sargs[] = {&H, &nh};
        e = launch_pdl(reinterpret_cast<const void*>(&enc_mb_scan_kernel), dim3(1), dim3(ENC_SORT_THREADS), 0, stream,
                       sargs);
        if (e != cudaSuccess) return e;
        void* xargs[] = {&src, &dst, &BTi, &sh, &ntiles, &H};
        e = launch_pdl(reinterpret_cast<const void*>(&enc_mb_scatter_kernel), dim3(ntiles), dim3(ENC_SORT_THREADS), 0,
                       stream, xargs);
        if (e != cudaSuccess) return e;
        src = dst;
    }
    EncTables t = tb;
    void* targs[] = {&BTi, &Vi, &Ci, &G, &t};
    const int nwin = (BT + ENC_WIN - 1) / ENC_WIN;
    return launch_pdl(reinterpret_cast<const void*>(&enc_mb_tables_kernel),
                      dim3(static_cast<unsigned>(std::max(1, std::min((nwin * G + 255) / 256, 4096)))), dim3(256), 0,
                      stream, targs);
}

// The sort: block 0 builds the tables; `wpe_blocks` more blocks form dwpe.
// Above ENC_FAST_MAX positions the multi-block sort runs instead and forms no
// dwpe (the caller adds dwpe blocks to the window launch).
cudaError_t enc_sort_launch(const int32_t* inp, int BT, int64_t V, int64_t C, int64_t B, int64_t T, int dtype,
                            const EncTables& tb, void* dwpe, const void* dout, int wpe_blocks, cudaStream_t stream) {
    if (BT > ENC_FAST_MAX) return enc_mb_sort_launch(inp, BT, V, C, tb, stream);
    int kpl = 1;  // keys per thread of the sorting cluster (at most 8: ENC_FAST_MAX positions)
    while (kpl * ENC_CS_THREADS * ENC_CS_CTAS < BT) kpl <<= 1;
    // sort on the smallest b with 2^b > V: the padding's digits (all ones) then
    // exceed those of every valid token, so the padding sorts last even where
    // invalid ids sit between valid ones
    int token_bits = 0;
    while ((int64_t(1) << token_bits) <= V) ++token_bits;
    int passes = (token_bits + ENC_DIGIT_BITS - 1) / ENC_DIGIT_BITS;
    const size_t sort_smem = (2 * static_cast<size_t>(kpl) * ENC_CS_THREADS + ENC_CS_CNT_WORDS) * 4;
    const void* ks = dtype == MMBWD_F32 ? enc_sort_fn<float>(kpl) : enc_sort_fn<__nv_bfloat16>(kpl);
    cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sort_smem));
    if (e != cudaSuccess) return e;
    int BTi = BT, Vi = static_cast<int>(V), Ci = static_cast<int>(C), Bi = static_cast<int>(B), Ti = static_cast<int>(T);
    int G = enc_groups(C, 4);
    EncTables t = tb;
    void* args[] = {const_cast<int32_t**>(&inp), &BTi, &Vi, &passes, &G, &t,
                    &dwpe, const_cast<void**>(&dout), &Bi, &Ti, &Ci};
    // the sorting cluster, then whole clusters of dwpe blocks
    const int grid = ENC_CS_CTAS + (wpe_blocks + ENC_CS_CTAS - 1) / ENC_CS_CTAS * ENC_CS_CTAS;
    return launch_pdl(ks, dim3(static_cast<unsigned>(grid)), dim3(ENC_CS_THREADS), sort_smem, stream, args);
}

// The window sums (and, with wpe_blocks > 0, dwpe) over tables `tb`.
cudaError_t enc_window_launch(void* dwte, void* dwpe, const void* dout, int64_t B, int64_t T, int64_t C, int64_t V,
                              int dtype, const EncTables& tb, int wpe_blocks, cudaStream_t stream) {
    int BTi = static_cast<int>(B * T), Ci = static_cast<int>(C), Bi = static_cast<int>(B), Ti = static_cast<int>(T),
        Vi = static_cast<int>(V);
    const int nwin = (BTi + ENC_WIN - 1) / ENC_WIN;
    int nw = nwin, G = enc_groups(C, 4), wb = wpe_blocks;
    const int gpb = std::min(G, 8), ngb = (G + gpb - 1) / gpb;  // warps (channel groups) per block
    EncTables t = tb;
    void* args[] = {&dwte, &dwpe, const_cast<void**>(&dout), &Ci, &BTi, &Bi, &Ti, &Vi, &nw, &G, &wb, &t};
    const void* k = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&enc_window_kernel<float>)
                                       : reinterpret_cast<const void*>(&enc_window_kernel<__nv_bfloat16>);
    return launch_pdl(k, dim3(static_cast<unsigned>(nwin * ngb + wpe_blocks)), dim3(32 * gpb), 0, stream, args);
}

}  // namespace

// Workspace of the one-call form: the tables, then the partials.
size_t enc_workspace_bytes(int64_t BT, int64_t C) {
    return enc_tables_layout(nullptr, BT, C, nullptr) + enc_partials_bytes(BT, C);
}

size_t enc_plan_bytes(int64_t BT, int64_t C) { return enc_tables_layout(nullptr, BT, C, nullptr); }
size_t enc_run_workspace_bytes(int64_t BT, int64_t C) { return enc_partials_bytes(BT, C); }

cudaError_t enc_launch(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                       int64_t V, int dtype, void* ws, int num_sms, cudaStream_t stream, bool sr, uint64_t seed) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const int BT = static_cast<int>(B * T);
    const int N = dtype == MMBWD_F32 ? 4 : 8;  // elements per 16-byte vector (dwpe)
    EncTables tb{};
    uint8_t* w = static_cast<uint8_t*>(ws);
    const size_t tbytes = enc_tables_layout(w, BT, C, &tb);
    tb.partials = reinterpret_cast<float*>(w + tbytes);
    tb.sr = sr ? 1 : 0;
    tb.seed = seed;
    if (BT > ENC_FAST_MAX) {  // multi-block sort; dwpe beside the window sums, as in a planned run
        cudaError_t e = enc_sort_launch(inp, BT, V, C, B, T, dtype, tb, nullptr, nullptr, 0, stream);
        if (e != cudaSuccess) return e;
        const int64_t width = 32 * std::min(enc_groups(C, 4), 8);
        const int wb = static_cast<int>(std::min<int64_t>((T * C / N + width - 1) / width, 2 * std::max(num_sms, 1)));
        return enc_window_launch(dwte, dwpe, dout, B, T, C, V, dtype, tb, wb, stream);
    }
    // the sorting cluster, and blocks of one 16-byte dwpe vector per thread
    const int64_t wpe_threads = (T * C / N + ENC_CS_THREADS - 1) / ENC_CS_THREADS;
    const int wpe_blocks = static_cast<int>(std::min<int64_t>(wpe_threads, 4 * std::max(num_sms, 1)));
    cudaError_t e = enc_sort_launch(inp, BT, V, C, B, T, dtype, tb, dwpe, dout, wpe_blocks, stream);
    if (e != cudaSuccess) return e;
    return enc_window_launch(dwte, dwpe, dout, B, T, C, V, dtype, tb, 0, stream);
}

cudaError_t enc_prepare_launch(void* plan, const int32_t* inp, int64_t B, int64_t T, int64_t C, int64_t V,
                               cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    EncTables tb{};
    enc_tables_layout(static_cast<uint8_t*>(plan), B * T, C, &tb);
    return enc_sort_launch(inp, static_cast<int>(B * T), V, C, B, T, MMBWD_BF16, tb, nullptr, nullptr, 0, stream);
}

cudaError_t enc_run_planned_launch(void* dwte, void* dwpe, const void* dout, void* plan, int64_t B, int64_t T,
                                   int64_t C, int64_t V, int dtype, void* ws, int num_sms, cudaStream_t stream, bool sr,
                                   uint64_t seed) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    const int N = dtype == MMBWD_F32 ? 4 : 8;
    EncTables tb{};
    enc_tables_layout(static_cast<uint8_t*>(plan), B * T, C, &tb);
    tb.partials = static_cast<float*>(ws);
    tb.sr = sr ? 1 : 0;
    tb.seed = seed;
    // dwpe blocks of the window blocks' width (one 16-byte vector per thread), at most two per SM
    const int64_t vecs = T * C / N;
    const int64_t width = 32 * std::min(enc_groups(C, 4), 8);
    const int wpe_blocks = static_cast<int>(std::min<int64_t>((vecs + width - 1) / width, 2 * std::max(num_sms, 1)));
    return enc_window_launch(dwte, dwpe, dout, B, T, C, V, dtype, tb, wpe_blocks, stream);
}

cudaError_t enc_read_status(int* code, int* info3, bool reset) {
    unsigned int h[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(h, g_enc_status, sizeof(h));
    if (e != cudaSuccess) return e;
    *code = h[0] ? -static_cast<int>(h[0]) : MMBWD_OK;
    if (info3) {
        info3[0] = static_cast<int>(h[1]);
        info3[1] = static_cast<int>(h[2]);
        info3[2] = 0;
    }
    if (reset) {
        const unsigned int z[4] = {0, 0, 0, 0};
        e = cudaMemcpyToSymbol(g_enc_status, z, sizeof(z));
    }
    return e;
}

}  // namespace mmbwd

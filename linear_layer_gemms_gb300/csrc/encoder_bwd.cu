// GPT-2 encoder backward (llm.c llmc/encoder.cuh): dwte[inp[b,t]] += dout[b,t]
// and dwpe[t] += sum over b of dout[b,t], deterministic and without atomics on
// the data.
//
// The page buckets the positions of each token on the host every step (a hash
// map and a sort over host token ids, then two host-to-device copies). Here
// the bucketing stays on the device, in two launches:
//   1. enc_sort_wpe_kernel. Block 0 (1024 threads) sorts the keys
//      (token << 15) | position stably by token in shared memory (LSD radix
//      passes of 4 bits over the token bits), so each token's positions end
//      up contiguous and in increasing order; block scans then cut the sorted
//      list into segments (one per token present) and chunks of at most 32
//      positions (a long segment is several chunks), and write the tables.
//      Token ids outside [0, V) are left out and reported in the status word.
//      The other blocks meanwhile form dwpe: one thread per (t, 16-byte
//      vector) sums dout over b in order, adds the old value, rounds once.
//   2. enc_chunk_kernel: one warp per (chunk, group of channels) sums its
//      positions' dout rows in order. A segment of one chunk is finished at
//      once (added to the old dwte row, rounded once). A longer segment's
//      chunks write fp32 partials and count themselves on a per-(segment,
//      channel group) counter; the last to arrive adds the partials in chunk
//      order to the old row. Which warp is last varies, the order of the sum
//      does not, so repeated calls give identical bits.
// The second grid is sized from the upper bound B*T and loops over the chunk
// count the sort wrote, so the host never waits for the device. Both launch
// with programmatic stream serialization and wait for their predecessor
// before touching global memory.
#include <algorithm>

#include "../../include/encoder_backward.h"
#include "../../include/mmbwd.h"
#include "internal.h"

namespace mmbwd {

// Status word of the encoder kernels: [0] error code (positive), [1] first
// offending position, [2] its token id.
__device__ unsigned int g_enc_status[4];

namespace {

constexpr int ENC_SORT_THREADS = 1024;
constexpr int ENC_CHUNK = 32;  // positions per chunk
constexpr unsigned ENC_PAD = 0xFFFFFFFFu;
constexpr int ENC_DIGIT_BITS = 4;  // radix digit width per pass
constexpr int ENC_DIGITS = 1 << ENC_DIGIT_BITS;
constexpr int ENC_CNT = ENC_DIGITS * ENC_SORT_THREADS;  // (digit, thread) counters
constexpr int ENC_CNT_WORDS = ENC_CNT + ENC_CNT / 32;   // with one pad word per 32

// Counter e = digit * 1024 + thread, padded so that a warp's 32 threads (one
// digit each) and a thread's 16 consecutive counters in the scan both fall in
// 32 distinct banks.
__device__ __forceinline__ int enc_cnt_at(int e) { return e + (e >> 5); }

__device__ __forceinline__ void enc_grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

struct EncTables {
    int* meta;          // [0] valid positions, [1] chunks, [2] segments
    int* rows;          // [B*T] positions in sorted order
    int2* chunk;        // [B*T + 1] per chunk: first sorted index, segment (sentinel: valid positions, segments)
    int2* seg;          // [B*T + 1] per segment: token id, first chunk (sentinel: 0, chunks)
    unsigned* arrivals; // [B*T][G] chunks of a segment done, per channel group
    float* partials;    // [B*T][C] fp32 chunk sums (segments of several chunks)
};

// Exclusive scan of one value per thread over the block (1024 threads, in
// thread order); returns the thread's prefix and writes the total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = static_cast<int>(threadIdx.x & 31), warp = static_cast<int>(threadIdx.x >> 5);
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
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
                             int64_t nthreads) {
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
        *dst = E::add_round(*dst, acc);
    }
}

// Block 0: sort, segments, chunks, for NP = KPL * 1024 >= B*T key slots.
// Thread t owns the KPL consecutive slots from t KPL. The keys start in
// position order (padding, all ones, after the last position), so a stable
// sort by token leaves each token's positions in increasing order and the
// padding last. A pass over a 4-bit digit (no warp votes):
//   - each thread ranks its keys among its own keys of equal digit
//     (compares in registers) and stores its count per digit at counter
//     (digit, thread);
//   - one block scan over the counters in (digit, thread) order turns them into
//     each thread's first slot per digit;
//   - each key goes to first slot + rank, back into the same shared buffer.
// Thread order is slot order, so the pass is stable.
// Blocks 1.. form dwpe (enc_wpe_part).
template <typename T, int KPL>
__global__ void __launch_bounds__(ENC_SORT_THREADS, 1)
    enc_sort_wpe_kernel(const int32_t* __restrict__ inp, int BT, int V, int passes, int G, EncTables tb,
                        T* __restrict__ dwpe, const T* __restrict__ dout, int B, int T_, int C) {
    enc_grid_wait();
    const int tid = static_cast<int>(threadIdx.x);
    if (blockIdx.x > 0) {
        enc_wpe_part<T>(dwpe, dout, B, T_, C, static_cast<int64_t>(blockIdx.x - 1) * ENC_SORT_THREADS + tid,
                        static_cast<int64_t>(gridDim.x - 1) * ENC_SORT_THREADS);
        return;
    }
    constexpr int NP = KPL * ENC_SORT_THREADS;
    extern __shared__ __align__(16) unsigned enc_smem[];  // keys[NP], then counters[ENC_CNT_WORDS]
    unsigned* keys = enc_smem;
    int* cnt = reinterpret_cast<int*>(enc_smem + NP);
    __shared__ int warp_sums[32];
    const int lane = tid & 31, warp = tid >> 5;
    const int i0 = tid * KPL;
    unsigned k[KPL];
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
        const int i = i0 + r;
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
    for (int pass = 0; pass < passes; ++pass) {
        const int sh = 15 + pass * ENC_DIGIT_BITS;
        if (pass > 0) {
            if constexpr (KPL >= 4) {
#pragma unroll
                for (int q = 0; q < KPL / 4; ++q) {
                    const uint4 v = reinterpret_cast<const uint4*>(keys + i0)[q];
                    k[4 * q] = v.x, k[4 * q + 1] = v.y, k[4 * q + 2] = v.z, k[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int r = 0; r < KPL; ++r) k[r] = keys[i0 + r];
            }
        }
#pragma unroll
        for (int q = 0; q < ENC_DIGITS; ++q) cnt[enc_cnt_at(tid * ENC_DIGITS + q)] = 0;
        int rank[KPL];  // earlier keys of this thread with the same digit
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
            const unsigned d = (k[r] >> sh) & (ENC_DIGITS - 1);
            int n = 0;
#pragma unroll
            for (int q = 0; q < r; ++q) n += ((k[q] >> sh) & (ENC_DIGITS - 1)) == d;
            rank[r] = n;
        }
        __syncthreads();  // counters zeroed; every thread has read its keys
#pragma unroll
        for (int r = 0; r < KPL; ++r)  // in order: the last store per digit is the count
            cnt[enc_cnt_at(static_cast<int>((k[r] >> sh) & (ENC_DIGITS - 1)) * ENC_SORT_THREADS + tid)] = rank[r] + 1;
        __syncthreads();
        {
            int loc[ENC_DIGITS];
            int sum = 0;
#pragma unroll
            for (int q = 0; q < ENC_DIGITS; ++q) {
                loc[q] = cnt[enc_cnt_at(tid * ENC_DIGITS + q)];
                sum += loc[q];
            }
            int before = block_exclusive_scan(sum, warp_sums, nullptr);
#pragma unroll
            for (int q = 0; q < ENC_DIGITS; ++q) {
                cnt[enc_cnt_at(tid * ENC_DIGITS + q)] = before;
                before += loc[q];
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < KPL; ++r)
            keys[cnt[enc_cnt_at(static_cast<int>((k[r] >> sh) & (ENC_DIGITS - 1)) * ENC_SORT_THREADS + tid)] + rank[r]] =
                k[r];
        __syncthreads();
    }
    if (passes == 0) {  // V == 0: every key is padding
#pragma unroll
        for (int r = 0; r < KPL; ++r) keys[i0 + r] = k[r];
        __syncthreads();
    }

    // Each thread takes its KPL consecutive sorted slots, read once into
    // registers with the token of the slot before; the scans below combine
    // the threads' runs in thread order.
    unsigned tk[KPL];  // token of each slot (the padding reads as all ones)
#pragma unroll
    for (int r = 0; r < KPL; ++r) tk[r] = keys[i0 + r] >> 15;
    const unsigned tk_prev = i0 > 0 ? keys[i0 - 1] >> 15 : ENC_PAD;
    int nvalid_local = 0;
#pragma unroll
    for (int r = 0; r < KPL; ++r) nvalid_local += tk[r] != (ENC_PAD >> 15);
    int nvalid = 0;
    block_exclusive_scan(nvalid_local, warp_sums, &nvalid);
    // sorted positions, coalesced
    for (int i = tid; i < nvalid; i += ENC_SORT_THREADS) tb.rows[i] = static_cast<int>(keys[i] & 0x7FFFu);
    // segment starts (token changes)
    bool starts[KPL];
    int seg_local = 0;
    int last_start_local = -1;  // last segment start inside this thread's slots
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
        const int i = i0 + r;
        starts[r] = i < nvalid && (i == 0 || tk[r] != (r > 0 ? tk[r - 1] : tk_prev));
        if (starts[r]) {
            ++seg_local;
            last_start_local = i;
        }
    }
    int nseg = 0;
    const int seg_before = block_exclusive_scan(seg_local, warp_sums, &nseg);
    // the start of the segment open at this thread's first slot: the largest
    // segment start to the left (an exclusive max-scan over the threads)
    int open_start = -1;
    {
        int x = last_start_local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x = max(x, y);
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w = max(w, y);
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int excl_in_warp = __shfl_up_sync(0xffffffffu, x, 1);
        open_start = lane > 0 ? excl_in_warp : -1;
        if (warp > 0) open_start = max(open_start, warp_sums[warp - 1]);
        __syncthreads();
    }
    // chunk starts: a segment start, or every ENC_CHUNK positions into a segment
    bool cstarts[KPL];
    int chunk_local = 0;
    {
        int os = open_start;
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
            const int i = i0 + r;
            if (starts[r]) os = i;
            cstarts[r] = i < nvalid && (starts[r] || (i - os) % ENC_CHUNK == 0);
            chunk_local += cstarts[r];
        }
    }
    int nchunk = 0;
    const int chunk_before = block_exclusive_scan(chunk_local, warp_sums, &nchunk);
    // tables; a segment's arrival counters are cleared when its second chunk starts
    int sid = seg_before - 1, cid = chunk_before - 1;
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
        const int i = i0 + r;
        if (cstarts[r]) {
            ++cid;
            if (starts[r]) {
                open_start = i;
                ++sid;
                tb.seg[sid] = make_int2(static_cast<int>(tk[r]), cid);
            }
            tb.chunk[cid] = make_int2(i, sid);
            if (i - open_start == ENC_CHUNK)
                for (int g = 0; g < G; ++g) tb.arrivals[static_cast<int64_t>(sid) * G + g] = 0u;
        }
    }
    if (tid == 0) {
        tb.chunk[nchunk] = make_int2(nvalid, nseg);
        tb.seg[nseg] = make_int2(0, nchunk);
        tb.meta[0] = nvalid;
        tb.meta[1] = nchunk;
        tb.meta[2] = nseg;
    }
}

// One warp per (chunk, channel group of 32 vectors), looping over the chunks:
// the chunk's dout rows in sorted (position) order, sixteen loads in flight,
// into an fp32 sum. A one-chunk segment goes straight to its dwte row;
// otherwise the partial is stored and the last of the segment's chunks to
// arrive adds all partials in chunk order (eight at a time in flight) to the
// row. The table reads that do not depend on each other are issued together.
// Lanes past C take part in the shuffles only.
template <typename T>
__global__ void __launch_bounds__(256) enc_chunk_kernel(T* __restrict__ dwte, const T* __restrict__ dout, int C,
                                                       EncTables tb) {
    using E = EncElem<T>;
    constexpr int N = E::N;
    constexpr int RB = 16;  // rows in flight
    constexpr int PB = 8;   // partials in flight
    enc_grid_wait();
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int c = (static_cast<int>(blockIdx.y) * 32 + lane) * N;
    const bool active = c < C;
    const int nchunk = tb.meta[1];
    for (int cid = static_cast<int>(blockIdx.x) * 8 + warp; cid < nchunk; cid += static_cast<int>(gridDim.x) * 8) {
        const int2 ch = tb.chunk[cid], ch1 = tb.chunk[cid + 1];
        const int s0 = ch.x, sid = ch.y;
        const int n = ch1.x - s0;  // 1..ENC_CHUNK
        const int my_row = lane < n ? tb.rows[s0 + lane] : 0;
        const int2 sg = tb.seg[sid], sg1 = tb.seg[sid + 1];
        const int k0 = sg.y, nk = sg1.y - k0;
        const int64_t tok = sg.x;
        float acc[N];
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = 0.f;
        for (int j0 = 0; j0 < n; j0 += RB) {
            uint4 v[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int64_t r = __shfl_sync(0xffffffffu, my_row, (j0 + u) & 31);
                v[u] = (active && j0 + u < n) ? __ldg(reinterpret_cast<const uint4*>(dout + r * C + c))
                                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < RB; ++u)
                if (j0 + u < n) E::add(v[u], acc);
        }
        if (nk > 1) {
            float* part = tb.partials + static_cast<int64_t>(cid) * C + c;
            if (active) {
#pragma unroll
                for (int e = 0; e < N; e += 4)
                    __stcg(reinterpret_cast<float4*>(part + e), make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]));
            }
            __threadfence();
            __syncwarp();
            unsigned done = 0;
            if (lane == 0) done = atomicAdd(&tb.arrivals[static_cast<int64_t>(sid) * gridDim.y + blockIdx.y], 1u);
            done = __shfl_sync(0xffffffffu, done, 0);
            if (done != static_cast<unsigned>(nk - 1)) continue;  // not the last chunk of the segment
            __threadfence();
#pragma unroll
            for (int e = 0; e < N; ++e) acc[e] = 0.f;
            if (active) {
                const float* src = tb.partials + static_cast<int64_t>(k0) * C + c;
                for (int k = 0; k < nk; k += PB) {
                    float4 pv[PB][N / 4];
#pragma unroll
                    for (int u = 0; u < PB; ++u)
#pragma unroll
                        for (int e = 0; e < N / 4; ++e)
                            pv[u][e] = k + u < nk ? __ldcg(reinterpret_cast<const float4*>(src + static_cast<int64_t>(k + u) * C) + e)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < PB; ++u)
                        if (k + u < nk) {
#pragma unroll
                            for (int e = 0; e < N / 4; ++e) {
                                acc[4 * e] += pv[u][e].x, acc[4 * e + 1] += pv[u][e].y;
                                acc[4 * e + 2] += pv[u][e].z, acc[4 * e + 3] += pv[u][e].w;
                            }
                        }
                }
            }
        }
        if (active) {
            uint4* dst = reinterpret_cast<uint4*>(dwte + tok * C + c);
            *dst = E::add_round(*dst, acc);
        }
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
        case 8: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 8>);
        default: return reinterpret_cast<const void*>(&enc_sort_wpe_kernel<T, 16>);
    }
}

}  // namespace

// Sized for fp32 (4 elements per vector, the most channel groups).
size_t enc_workspace_bytes(int64_t BT, int64_t C) {
    const size_t n = static_cast<size_t>(BT);
    return a256(4 * 4) + a256(n * 4) + a256((n + 1) * 8) + a256((n + 1) * 8) +
           a256(n * static_cast<size_t>(enc_groups(C, 4)) * 4) + a256(n * static_cast<size_t>(C) * 4);
}

cudaError_t enc_launch(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                       int64_t V, int dtype, void* ws, int num_sms, cudaStream_t stream) {
    const int BT = static_cast<int>(B * T);
    const int N = dtype == MMBWD_F32 ? 4 : 8;
    int G = enc_groups(C, N);
    uint8_t* w = static_cast<uint8_t*>(ws);
    EncTables tb{};
    auto take = [&](size_t bytes) {
        uint8_t* p = w;
        w += a256(bytes);
        return p;
    };
    tb.meta = reinterpret_cast<int*>(take(4 * 4));
    tb.rows = reinterpret_cast<int*>(take(static_cast<size_t>(BT) * 4));
    tb.chunk = reinterpret_cast<int2*>(take((static_cast<size_t>(BT) + 1) * 8));
    tb.seg = reinterpret_cast<int2*>(take((static_cast<size_t>(BT) + 1) * 8));
    tb.arrivals = reinterpret_cast<unsigned*>(take(static_cast<size_t>(BT) * enc_groups(C, 4) * 4));
    tb.partials = reinterpret_cast<float*>(take(static_cast<size_t>(BT) * C * 4));
    int kpl = 1;
    while (kpl * ENC_SORT_THREADS < BT) kpl <<= 1;
    // sort on the smallest b with 2^b > V: the padding's digits (all ones) then
    // exceed those of every valid token, so the padding sorts last even where
    // invalid ids sit between valid ones
    int token_bits = 0;
    while ((int64_t(1) << token_bits) <= V) ++token_bits;
    int passes = (token_bits + ENC_DIGIT_BITS - 1) / ENC_DIGIT_BITS;
    const size_t sort_smem = (static_cast<size_t>(kpl) * ENC_SORT_THREADS + ENC_CNT_WORDS) * 4;
    const void* ks = dtype == MMBWD_F32 ? enc_sort_fn<float>(kpl) : enc_sort_fn<__nv_bfloat16>(kpl);
    cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sort_smem));
    if (e != cudaSuccess) return e;
    int Vi = static_cast<int>(V), Ci = static_cast<int>(C), Bi = static_cast<int>(B), Ti = static_cast<int>(T);
    {
        // block 0 sorts; one wave of blocks (at most one per SM besides it) forms dwpe
        const int64_t wpe_threads = (T * C / N + ENC_SORT_THREADS - 1) / ENC_SORT_THREADS;
        const int wpe_blocks = static_cast<int>(std::min<int64_t>(wpe_threads, std::max(num_sms - 1, 1)));
        void* args[] = {const_cast<int32_t**>(&inp), const_cast<int*>(&BT), &Vi, &passes, &G, &tb,
                        &dwpe, const_cast<void**>(&dout), &Bi, &Ti, &Ci};
        e = launch_pdl(ks, dim3(static_cast<unsigned>(1 + wpe_blocks)), dim3(ENC_SORT_THREADS), sort_smem, stream,
                       args);
        if (e != cudaSuccess) return e;
    }
    {
        // about four blocks of eight warps per SM in all (two waves at two
        // resident blocks per SM); each warp loops over chunks
        const int per_group = std::max(1, 4 * num_sms / G);
        const int gx = std::min((BT + 7) / 8, per_group);
        void* args[] = {&dwte, const_cast<void**>(&dout), &Ci, &tb};
        const void* k = dtype == MMBWD_F32 ? reinterpret_cast<const void*>(&enc_chunk_kernel<float>)
                                           : reinterpret_cast<const void*>(&enc_chunk_kernel<__nv_bfloat16>);
        e = launch_pdl(k, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(G)), dim3(256), 0, stream, args);
    }
    return e;
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

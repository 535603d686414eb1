// C ABI of the matmul_backward library: argument checks, the shape-only plan,
// the per-device workspace and the launches. See include/mmbwd.h for the
// contract of every entry point.
#include "../../include/mmbwd.h"
#include "../../include/layernorm_backward.h"
#include "../../include/encoder_backward.h"
#include "internal.h"
#include "ops.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace mmbwd {

EncodeTiledFn get_encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    int arch_checked = 0;  // 0 unknown, 1 ok, -1 not sm_103
    int num_sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::atomic<int> g_fail_allocs{0};
std::atomic<int> g_fail_launches{0};

// One NVTX range per entry point call (named after the entry point), so a
// timeline tool shows where each call's host work and launches happen.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Plans depend only on (BT, C, OC, SM count) and the tuning overrides; the
// schedule search is cached so that a call costs a table lookup.
struct PlanKey {
    int64_t BT, C, OC;
    int sms, fwd;
    long splitk, grid, tile_n;
    bool operator==(const PlanKey& o) const {
        return BT == o.BT && C == o.C && OC == o.OC && sms == o.sms && fwd == o.fwd && splitk == o.splitk &&
               grid == o.grid && tile_n == o.tile_n;
    }
};
constexpr int kPlanCache = 32;
PlanKey g_plan_keys[kPlanCache];
TcPlan g_plans[kPlanCache];
int g_plan_count = 0, g_plan_next = 0;

long env_long(const char* name) {
    const char* s = std::getenv(name);
    return (s && *s) ? std::strtol(s, nullptr, 10) : 0;
}

// "<dinp>,<dweight>" tile-width override as one number for the cache key.
long env_tile_n() {
    const char* s = std::getenv("MMBWD_TILE_N");
    int a = 0, b = 0;
    return (s && std::sscanf(s, "%d,%d", &a, &b) == 2) ? 1000L * a + b : 0;
}

// Caller holds g_mutex.
const TcPlan& cached_plan(int64_t BT, int64_t C, int64_t OC, int sms, int fwd = 0) {
    const PlanKey k{BT, C, OC, sms, fwd, env_long("MMBWD_SPLITK"), env_long("MMBWD_GRID"), env_tile_n()};
    for (int i = 0; i < g_plan_count; ++i)
        if (g_plan_keys[i] == k) return g_plans[i];
    const int slot = g_plan_next;
    g_plan_next = (g_plan_next + 1) % kPlanCache;
    if (g_plan_count < kPlanCache) ++g_plan_count;
    g_plan_keys[slot] = k;
    g_plans[slot] = fwd ? tc_make_plan_forward(BT, C, OC, sms) : tc_make_plan(BT, C, OC, sms);
    return g_plans[slot];
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A tensor argument: its first byte and its size in bytes.
struct Span {
    const void* p;
    size_t n;
};

// Every non-empty tensor must lie in device memory of the current device
// `dev` (its first and its last byte): the kernels and their tensor maps
// address it directly, and no call is meant to reach host memory or another
// GPU's memory through a mapping. Checked before anything is enqueued.
int check_local(const Span* t, int n, int dev) {
    for (int i = 0; i < n; ++i) {
        if (!t[i].p || t[i].n == 0) continue;
        const void* ends[2] = {t[i].p, static_cast<const uint8_t*>(t[i].p) + (t[i].n - 1)};
        for (const void* q : ends) {
            cudaPointerAttributes a{};
            if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
                cudaGetLastError();
                return MMBWD_ERR_MEMORY;
            }
            if (a.type != cudaMemoryTypeDevice || a.device != dev) return MMBWD_ERR_MEMORY;
        }
    }
    return MMBWD_OK;
}

// a * b without overflow beyond 2^62; returns false on overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > (int64_t(1) << 62) / a) return false;
    *out = a * b;
    return true;
}

struct Shape {
    int64_t BT = 0, n_dinp = 0, n_dw = 0, n_dout = 0;
    size_t es = 0;
};

int check_shape(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, Shape* s) {
    if (dtype != MMBWD_F32 && dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    if (B < 0 || T < 0 || C < 0 || OC < 0) return MMBWD_ERR_SHAPE;
    if (!mul_ok(B, T, &s->BT) || !mul_ok(s->BT, C, &s->n_dinp) || !mul_ok(OC, C, &s->n_dw) ||
        !mul_ok(s->BT, OC, &s->n_dout))
        return MMBWD_ERR_SHAPE;
    s->es = dtype == MMBWD_F32 ? 4 : 2;
    // Limits of the launch geometry and the tensor maps (dims < 2^31, tile counts in int).
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (s->BT > lim || C > lim || OC > lim) return MMBWD_ERR_SHAPE;
    if ((s->BT + 127) / 128 * ((C + 255) / 256) > lim / 32) return MMBWD_ERR_SHAPE;
    if ((OC + 127) / 128 * ((C + 255) / 256) > lim / 32) return MMBWD_ERR_SHAPE;
    if ((C + 127) / 128 > 65535) return MMBWD_ERR_SHAPE;  // fp32 path grid.y
    int64_t bytes = 0;
    if (!mul_ok(s->n_dout, static_cast<int64_t>(s->es), &bytes) ||
        !mul_ok(s->n_dinp, static_cast<int64_t>(s->es), &bytes) ||
        !mul_ok(s->n_dw, static_cast<int64_t>(s->es), &bytes))
        return MMBWD_ERR_SHAPE;
    return MMBWD_OK;
}

int device_state(DeviceState** out, int* dev_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MMBWD_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    if (d.arch_checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MMBWD_ERR_CUDA;
        d.arch_checked = (major == 10 && minor == 3) ? 1 : -1;
        d.num_sms = sms;
        if (d.arch_checked == 1) {
            // CTAs the persistent kernel can keep resident: whole pairs only.
            const int pairs = tc_max_active_clusters(2);
            if (pairs > 0 && 2 * pairs < sms) d.num_sms = 2 * pairs;
        }
    }
    if (d.arch_checked != 1) return MMBWD_ERR_ARCH;
    *out = &d;
    *dev_out = dev;
    return MMBWD_OK;
}

// fp32 path: three tf32 products on the tensor cores for every shape they take
// (faster than the fp32 FMA kernel at every size measured, from 8 x 8 x 8 at
// 7.7 against 11.4 us to the GPT-2 XL layers at 658 against 4291 us), fp32
// FMAs for the rest. MMBWD_F32_PATH = "ffma" or "x3" forces one (the latter
// where the shape allows it).
// The tensor core rounds every accumulation toward zero, so the tensor-core
// path's error grows with the reduction length: measured at GPT-2 XL sizes,
// 4e-5 of the 1e-4 bound at K = 6400, 8e-5 at K = 16384, 1.9e-4 at K = 32768
// (scaled error |gpu - ref| / (|ref| + rms(ref))). Both products' reduction
// lengths (OC for dinp, B*T for dweight; C for the forward) stay within
// X3_MAX_K, even when the path is forced.
constexpr int64_t X3_MAX_K = 8192;

bool use_x3(int64_t BT, int64_t C, int64_t OC) {
    if (!x3_shape_ok(BT, C, OC) || OC > X3_MAX_K || BT > X3_MAX_K) return false;
    if (const char* f = std::getenv("MMBWD_F32_PATH")) {
        if (std::strcmp(f, "ffma") == 0) return false;
        if (std::strcmp(f, "x3") == 0) return true;
    }
    return true;
}

bool use_x3_forward(int64_t BT, int64_t C, int64_t OC) {
    if (!x3_forward_shape_ok(BT, C, OC) || C > X3_MAX_K) return false;
    if (const char* f = std::getenv("MMBWD_F32_PATH")) {
        if (std::strcmp(f, "ffma") == 0) return false;
        if (std::strcmp(f, "x3") == 0) return true;
    }
    return true;
}

// Grow the device's workspace to `need` bytes (its contents need no initial value).
int ensure_workspace(DeviceState& d, size_t need, cudaStream_t stream) {
    if (need <= d.ws_bytes) return MMBWD_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MMBWD_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return MMBWD_ERR_CAPTURE;
    if (g_fail_allocs.load() > 0) {
        g_fail_allocs.fetch_sub(1);
        return MMBWD_ERR_ALLOC;
    }
    if (d.ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return MMBWD_ERR_CUDA;
        cudaFree(d.ws);
        d.ws = nullptr;
        d.ws_bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
        cudaGetLastError();
        return MMBWD_ERR_ALLOC;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p);
        return MMBWD_ERR_CUDA;
    }
    d.ws = p;
    d.ws_bytes = need;
    return MMBWD_OK;
}

}  // namespace

bool take_injected_launch_failure() {
    int n = g_fail_launches.load();
    while (n > 0)
        if (g_fail_launches.compare_exchange_weak(n, n - 1)) return true;
    return false;
}

}  // namespace mmbwd

using namespace mmbwd;

extern "C" {

int mmbwd_version(void) { return 10000; }

const char* mmbwd_strerror(int code) {
    switch (code) {
        case MMBWD_OK: return "ok";
        case MMBWD_ERR_NULL: return "a required pointer is NULL";
        case MMBWD_ERR_DTYPE: return "dtype must be MMBWD_F32 or MMBWD_BF16";
        case MMBWD_ERR_SHAPE: return "a size is negative, too large, or a product overflows";
        case MMBWD_ERR_ALIGN: return "pointers must be 16-byte aligned and C, OC times the element size multiples of 16 bytes";
        case MMBWD_ERR_ALIAS: return "an output overlaps an input or another output";
        case MMBWD_ERR_ALLOC: return "workspace allocation failed";
        case MMBWD_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case MMBWD_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
        case MMBWD_ERR_ARCH: return "the current device is not sm_103 (GB300)";
        case MMBWD_ERR_CAPTURE: return "the workspace must grow but the stream is being captured";
        case MMBWD_ERR_SCRATCH: return "the problem needs more scratch than the library's fixed buffer holds";
        case MMBWD_ERR_MEMORY: return "a tensor is not in device memory of the current device";
        default: return "unknown status code";
    }
}

size_t mmbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype) {
    Shape s;
    if (check_shape(B, T, C, OC, dtype, &s) != MMBWD_OK) return 0;
    if (s.BT == 0 || C == 0 || OC == 0) return 0;
    if (dtype == MMBWD_F32) return 0;  // both fp32 paths work in place
    int sms = 0;
    {
        std::lock_guard<std::mutex> g(g_mutex);
        DeviceState* d = nullptr;
        int dev = 0;
        if (device_state(&d, &dev) == MMBWD_OK) sms = d->num_sms;
    }
    if (sms <= 0) sms = 152;  // no usable device: size for a full GB300
    return tc_make_plan(s.BT, C, OC, sms).ws_bytes();
}

int mmbwd_plan_info(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, int num_sms, int* out, int n) {
    Shape s;
    const int rc = check_shape(B, T, C, OC, dtype, &s);
    if (rc != MMBWD_OK) return rc;
    if (!out || n < 0) return MMBWD_ERR_NULL;
    int v[15] = {0};
    if (num_sms <= 0) {  // the current device's resident CTAs (a full GB300 without a device)
        std::lock_guard<std::mutex> g(g_mutex);
        DeviceState* d = nullptr;
        int dev = 0;
        num_sms = device_state(&d, &dev) == MMBWD_OK ? d->num_sms : 152;
    }
    if (dtype == MMBWD_BF16) {
        const TcPlan pl = tc_make_plan(s.BT, C, OC, num_sms);
        const int vals[15] = {1, pl.grid, pl.n_items, pl.splits, pl.kb_per_split, pl.n_dinp_items,
                              pl.n_dw_items / (pl.splits > 0 ? pl.splits : 1), pl.table,
                              TC_PAIR_BM, pl.dinp_bn, pl.dw_bn, TC_BK, TC_STAGES, pl.launches(), 1};
        for (int i = 0; i < 15; ++i) v[i] = vals[i];
    } else if (use_x3(s.BT, C, OC)) {
        // both products (and dbias) in one launch, or one launch each where
        // they cannot share one
        static thread_local TcPlan pp;
        pp = tc_make_plan_x3_pair(s.BT, C, OC, num_sms);
        if (pp.n_items > 0) {
            const int vals[15] = {2, pp.grid, pp.n_items, 1, 0, pp.n_dinp_items, pp.n_dw_items, pp.table,
                                  TC_PAIR_BM, pp.dinp_bn, pp.dw_bn, TC_BK / 2, TC_STAGES_X3, 1, 1};
            for (int i = 0; i < 15; ++i) v[i] = vals[i];
        } else {
            const TcPlan p1 = tc_make_plan_x3(s.BT, C, OC, num_sms), p2 = tc_make_plan_x3(OC, C, s.BT, num_sms);
            const int vals[15] = {2, std::max(p1.grid, p2.grid), p1.n_items + p2.n_items, 1, 0, p1.n_items,
                                  p2.n_items, 0, TC_PAIR_BM, p1.dinp_bn, p2.dinp_bn, TC_BK / 2, TC_STAGES_X3, 2, 1};
            for (int i = 0; i < 15; ++i) v[i] = vals[i];
        }
    } else {
        const int gm = static_cast<int>((s.BT + SIMT_BM - 1) / SIMT_BM), gn = static_cast<int>((C + SIMT_BN - 1) / SIMT_BN);
        const int go = static_cast<int>((OC + SIMT_BM - 1) / SIMT_BM);
        const int vals[15] = {0, gm * gn + go * gn, gm * gn + go * gn, 1, 0, gm * gn, go * gn, 0, SIMT_BM, SIMT_BN, SIMT_BN, SIMT_BK, 2, 2, 0};
        for (int i = 0; i < 15; ++i) v[i] = vals[i];
    }
    const int m = n < 15 ? n : 15;
    for (int i = 0; i < m; ++i) out[i] = v[i];
    return m;
}

namespace {

// mmbwd_run and mmbwd_run_sr: `sr` selects stochastic rounding of the bf16
// outputs with `seed` (sr.cuh).
int run_backward(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
                 int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, bool sr, uint64_t seed,
                 cudaStream_t stream) {
    Shape s;
    int rc = check_shape(B, T, C, OC, dtype, &s);
    if (rc != MMBWD_OK) return rc;
    const size_t es = s.es;
    const size_t b_dinp = static_cast<size_t>(s.n_dinp) * es, b_dw = static_cast<size_t>(s.n_dw) * es,
                 b_db = static_cast<size_t>(OC) * es, b_dout = static_cast<size_t>(s.n_dout) * es,
                 b_inp = static_cast<size_t>(s.n_dinp) * es, b_w = static_cast<size_t>(s.n_dw) * es;

    // NULL only where the tensor is empty (dbias NULL means "skip the bias").
    if ((b_dinp && !dinp) || (b_dw && !dweight) || (b_dout && !dout) || (b_inp && !inp) || (b_w && !weight))
        return MMBWD_ERR_NULL;
    const void* ptrs[6] = {dinp, dweight, dbias, dout, inp, weight};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0 || (static_cast<size_t>(OC) * es) % 16 != 0) return MMBWD_ERR_ALIGN;

    // Outputs overlap neither inputs nor each other.
    const void* outs[3] = {dinp, dweight, dbias};
    const size_t nouts[3] = {b_dinp, b_dw, b_db};
    const void* ins[3] = {dout, inp, weight};
    const size_t nins[3] = {b_dout, b_inp, b_w};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j)
            if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return MMBWD_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return MMBWD_ERR_ALIAS;
    }

    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[6] = {{dinp, b_dinp}, {dweight, b_dw}, {dbias, b_db}, {dout, b_dout}, {inp, b_inp}, {weight, b_w}};
    rc = check_local(spans, 6, dev);
    if (rc != MMBWD_OK) return rc;

    cudaError_t e = cudaSuccess;
    if (OC == 0) return MMBWD_OK;  // empty sums everywhere; dbias has no elements
    if (s.BT == 0) {
        if (dbias) e = cudaMemsetAsync(dbias, 0, b_db, stream);  // the empty sum
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    if (C == 0) {
        if (dbias) e = colsum_launch(dbias, dout, s.BT, OC, dtype, sr, seed, stream);
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }

    if (dtype == MMBWD_F32) {
        if (use_x3(s.BT, C, OC)) {
            e = x3_launch(static_cast<float*>(dinp), static_cast<float*>(dweight), static_cast<float*>(dbias),
                          static_cast<const float*>(dout), static_cast<const float*>(inp),
                          static_cast<const float*>(weight), s.BT, C, OC, d->num_sms, stream);
        } else {
            e = simt_launch(static_cast<float*>(dinp), static_cast<float*>(dweight), static_cast<float*>(dbias),
                            static_cast<const float*>(dout), static_cast<const float*>(inp),
                            static_cast<const float*>(weight), s.BT, C, OC, stream);
        }
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }

    const TcPlan plan = cached_plan(s.BT, C, OC, d->num_sms);
    rc = ensure_workspace(*d, plan.ws_bytes(), stream);
    if (rc != MMBWD_OK) return rc;
    e = tc_launch(plan, dinp, dweight, dbias, dout, inp, weight, s.BT, C, OC, d->ws, stream, sr, seed);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

}  // namespace

int mmbwd_run(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
              int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, cudaStream_t stream) {
    NvtxRange nvtx("mmbwd_run");
    return run_backward(dinp, dweight, dbias, dout, inp, weight, B, T, C, OC, dtype, false, 0, stream);
}

int mmbwd_run_sr(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
                 int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, uint64_t seed, cudaStream_t stream) {
    NvtxRange nvtx("mmbwd_run_sr");
    if (dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    return run_backward(dinp, dweight, dbias, dout, inp, weight, B, T, C, OC, dtype, true, seed, stream);
}

int mmbwd_release(void) {
    std::lock_guard<std::mutex> g(g_mutex);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MMBWD_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    if (d.ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return MMBWD_ERR_CUDA;
        if (cudaFree(d.ws) != cudaSuccess) return MMBWD_ERR_CUDA;
        d.ws = nullptr;
        d.ws_bytes = 0;
    }
    return MMBWD_OK;
}

int mmbwd_device_status(int reset, int* info) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MMBWD_ERR_CUDA;
    int code = MMBWD_OK, ln_code = MMBWD_OK, ln_info[3] = {0, 0, 0};
    if (tc_read_status(&code, info, reset != 0) != cudaSuccess) return MMBWD_ERR_CUDA;
    if (ln_read_status(&ln_code, ln_info, reset != 0) != cudaSuccess) return MMBWD_ERR_CUDA;
    if (code == MMBWD_OK && ln_code != MMBWD_OK) {
        code = ln_code;
        if (info)
            for (int i = 0; i < 3; ++i) info[i] = ln_info[i];
    }
    int enc_code = MMBWD_OK, enc_info[3] = {0, 0, 0};
    if (enc_read_status(&enc_code, enc_info, reset != 0) != cudaSuccess) return MMBWD_ERR_CUDA;
    if (code == MMBWD_OK && enc_code != MMBWD_OK) {
        code = enc_code;
        if (info)
            for (int i = 0; i < 3; ++i) info[i] = enc_info[i];
    }
    return code;
}

int mmbwd_selftest_wait_timeout(uint64_t timeout_ns) {
    {
        std::lock_guard<std::mutex> g(g_mutex);
        DeviceState* d = nullptr;
        int dev = 0;
        const int rc = device_state(&d, &dev);
        if (rc != MMBWD_OK) return rc;
    }
    if (tc_selftest_wait(timeout_ns) != cudaSuccess) return MMBWD_ERR_CUDA;
    int code = MMBWD_OK;
    if (tc_read_status(&code, nullptr, true) != cudaSuccess) return MMBWD_ERR_CUDA;
    return code;
}

void mmbwd_debug_fail_next_alloc(int n) { g_fail_allocs.store(n < 0 ? 0 : n); }

void mmbwd_debug_fail_next_launch(int n) { g_fail_launches.store(n < 0 ? 0 : n); }

int mmbwd_forward(void* out, const void* inp, const void* weight, const void* bias, int64_t B, int64_t T,
                  int64_t C, int64_t OC, int dtype, cudaStream_t stream) {
    NvtxRange nvtx("mmbwd_forward");
    Shape s;
    int rc = check_shape(B, T, C, OC, dtype, &s);
    if (rc != MMBWD_OK) return rc;
    const size_t es = s.es;
    const size_t b_out = static_cast<size_t>(s.n_dout) * es, b_inp = static_cast<size_t>(s.n_dinp) * es,
                 b_w = static_cast<size_t>(s.n_dw) * es, b_b = static_cast<size_t>(OC) * es;
    if ((b_out && !out) || (b_inp && !inp) || (b_w && !weight)) return MMBWD_ERR_NULL;
    const void* ptrs[4] = {out, inp, weight, bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0 || (static_cast<size_t>(OC) * es) % 16 != 0) return MMBWD_ERR_ALIGN;
    if (overlaps(out, b_out, inp, b_inp) || overlaps(out, b_out, weight, b_w) || overlaps(out, b_out, bias, b_b))
        return MMBWD_ERR_ALIAS;

    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[4] = {{out, b_out}, {inp, b_inp}, {weight, b_w}, {bias, b_b}};
    rc = check_local(spans, 4, dev);
    if (rc != MMBWD_OK) return rc;
    cudaError_t e = cudaSuccess;
    if (s.BT == 0 || OC == 0) return MMBWD_OK;  // no output element
    if (C == 0) {                                // the empty product: out = bias (or 0)
        e = fill_rows_launch(out, bias, s.BT, OC, dtype, stream);
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    if (dtype == MMBWD_F32) {
        if (use_x3_forward(s.BT, C, OC)) {
            e = x3_forward_launch(static_cast<float*>(out), static_cast<const float*>(inp),
                                  static_cast<const float*>(weight), static_cast<const float*>(bias), s.BT, C, OC,
                                  d->num_sms, stream);
        } else {
            e = simt_forward_launch(static_cast<float*>(out), static_cast<const float*>(inp),
                                    static_cast<const float*>(weight), static_cast<const float*>(bias), s.BT, C, OC,
                                    stream);
        }
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    const TcPlan& plan = cached_plan(s.BT, C, OC, d->num_sms, 1);
    e = tc_launch_forward(plan, out, inp, weight, bias, s.BT, C, OC, stream);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

int mmbwd_forward_path(int64_t B, int64_t T, int64_t C, int64_t OC, int dtype) {
    Shape s;
    const int rc = check_shape(B, T, C, OC, dtype, &s);
    if (rc != MMBWD_OK) return rc;
    if (dtype == MMBWD_BF16) return 1;
    return use_x3_forward(s.BT, C, OC) ? 2 : 0;
}

// ---------------------------------------------------------------------------
// Encoder backward (encoder_backward.h)

namespace {

int enc_check(int64_t B, int64_t T, int64_t C, int64_t V, int dtype, int64_t* BT) {
    if (dtype != MMBWD_F32 && dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    if (B < 0 || T < 0 || C < 0 || V < 0) return MMBWD_ERR_SHAPE;
    if (!mul_ok(B, T, BT) || *BT > ENCBWD_MAX_POSITIONS || V > ENCBWD_MAX_VOCAB) return MMBWD_ERR_SHAPE;
    int64_t x = 0;
    if (!mul_ok(*BT, C, &x) || !mul_ok(V, C, &x) || C > ENCBWD_MAX_CHANNELS) return MMBWD_ERR_SHAPE;
    return MMBWD_OK;
}

}  // namespace

size_t encbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int64_t V, int dtype) {
    int64_t BT = 0;
    if (enc_check(B, T, C, V, dtype, &BT) != MMBWD_OK || BT == 0 || C == 0) return 0;
    return enc_workspace_bytes(BT, C);
}

namespace {

int run_encoder(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                int64_t V, int dtype, bool sr, uint64_t seed, cudaStream_t stream) {
    int64_t BT = 0;
    int rc = enc_check(B, T, C, V, dtype, &BT);
    if (rc != MMBWD_OK) return rc;
    const size_t es = dtype == MMBWD_F32 ? 4 : 2;
    const size_t b_out = static_cast<size_t>(BT) * C * es, b_wte = static_cast<size_t>(V) * C * es,
                 b_wpe = static_cast<size_t>(T) * C * es, b_inp = static_cast<size_t>(BT) * 4;
    if ((b_out && (!dout || !dwpe)) || (b_inp && !inp) || (b_wte && !dwte)) return MMBWD_ERR_NULL;
    const void* vecs[3] = {dwte, dwpe, dout};
    for (const void* p : vecs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(inp) & 3u) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0) return MMBWD_ERR_ALIGN;
    if (overlaps(dwte, b_wte, dwpe, b_wpe) || overlaps(dwte, b_wte, dout, b_out) || overlaps(dwte, b_wte, inp, b_inp) ||
        overlaps(dwpe, b_wpe, dout, b_out) || overlaps(dwpe, b_wpe, inp, b_inp))
        return MMBWD_ERR_ALIAS;

    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[4] = {{dwte, b_wte}, {dwpe, b_wpe}, {dout, b_out}, {inp, b_inp}};
    rc = check_local(spans, 4, dev);
    if (rc != MMBWD_OK) return rc;
    if (BT == 0 || C == 0) return MMBWD_OK;  // empty sums: nothing changes
    rc = ensure_workspace(*d, enc_workspace_bytes(BT, C), stream);
    if (rc != MMBWD_OK) return rc;
    const cudaError_t e = enc_launch(dwte, dwpe, dout, inp, B, T, C, V, dtype, d->ws, d->num_sms, stream, sr, seed);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

}  // namespace

int encbwd_run(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
               int64_t V, int dtype, cudaStream_t stream) {
    NvtxRange nvtx("encbwd_run");
    return run_encoder(dwte, dwpe, dout, inp, B, T, C, V, dtype, false, 0, stream);
}

int encbwd_run_sr(void* dwte, void* dwpe, const void* dout, const int32_t* inp, int64_t B, int64_t T, int64_t C,
                  int64_t V, int dtype, uint64_t seed, cudaStream_t stream) {
    NvtxRange nvtx("encbwd_run_sr");
    if (dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    return run_encoder(dwte, dwpe, dout, inp, B, T, C, V, dtype, true, seed, stream);
}

size_t encbwd_plan_bytes(int64_t B, int64_t T, int64_t C, int64_t V, int dtype) {
    int64_t BT = 0;
    if (enc_check(B, T, C, V, dtype, &BT) != MMBWD_OK || BT == 0 || C == 0) return 0;
    return enc_plan_bytes(BT, C);
}

int encbwd_prepare(void* plan, size_t plan_bytes, const int32_t* inp, int64_t B, int64_t T, int64_t C, int64_t V,
                   int dtype, cudaStream_t stream) {
    NvtxRange nvtx("encbwd_prepare");
    int64_t BT = 0;
    int rc = enc_check(B, T, C, V, dtype, &BT);
    if (rc != MMBWD_OK) return rc;
    const size_t es = dtype == MMBWD_F32 ? 4 : 2;
    if ((static_cast<size_t>(C) * es) % 16 != 0) return MMBWD_ERR_ALIGN;
    if (BT == 0 || C == 0) return MMBWD_OK;  // nothing to bucket; a planned run of this size does nothing
    if (!plan || !inp) return MMBWD_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(plan) & 255u) || (reinterpret_cast<uintptr_t>(inp) & 3u)) return MMBWD_ERR_ALIGN;
    const size_t need = enc_plan_bytes(BT, C);
    if (plan_bytes < need) return MMBWD_ERR_SHAPE;
    if (overlaps(plan, need, inp, static_cast<size_t>(BT) * 4)) return MMBWD_ERR_ALIAS;
    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[2] = {{plan, need}, {inp, static_cast<size_t>(BT) * 4}};
    rc = check_local(spans, 2, dev);
    if (rc != MMBWD_OK) return rc;
    const cudaError_t e = enc_prepare_launch(plan, inp, B, T, C, V, stream);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

int encbwd_run_planned(void* dwte, void* dwpe, const void* dout, void* plan, int64_t B, int64_t T, int64_t C,
                       int64_t V, int dtype, const uint64_t* sr_seed, cudaStream_t stream) {
    NvtxRange nvtx("encbwd_run_planned");
    int64_t BT = 0;
    int rc = enc_check(B, T, C, V, dtype, &BT);
    if (rc != MMBWD_OK) return rc;
    if (sr_seed && dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    const size_t es = dtype == MMBWD_F32 ? 4 : 2;
    const size_t b_out = static_cast<size_t>(BT) * C * es, b_wte = static_cast<size_t>(V) * C * es,
                 b_wpe = static_cast<size_t>(T) * C * es;
    if ((b_out && (!dout || !dwpe || !plan)) || (b_wte && !dwte)) return MMBWD_ERR_NULL;
    const void* vecs[3] = {dwte, dwpe, dout};
    for (const void* p : vecs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(plan) & 255u) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0) return MMBWD_ERR_ALIGN;
    const size_t b_plan = (BT && C) ? enc_plan_bytes(BT, C) : 0;
    if (overlaps(dwte, b_wte, dwpe, b_wpe) || overlaps(dwte, b_wte, dout, b_out) || overlaps(dwpe, b_wpe, dout, b_out) ||
        overlaps(plan, b_plan, dwte, b_wte) || overlaps(plan, b_plan, dwpe, b_wpe) || overlaps(plan, b_plan, dout, b_out))
        return MMBWD_ERR_ALIAS;
    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[4] = {{dwte, b_wte}, {dwpe, b_wpe}, {dout, b_out}, {plan, b_plan}};
    rc = check_local(spans, 4, dev);
    if (rc != MMBWD_OK) return rc;
    if (BT == 0 || C == 0) return MMBWD_OK;
    rc = ensure_workspace(*d, enc_run_workspace_bytes(BT, C), stream);
    if (rc != MMBWD_OK) return rc;
    const cudaError_t e = enc_run_planned_launch(dwte, dwpe, dout, plan, B, T, C, V, dtype, d->ws, d->num_sms, stream,
                                                 sr_seed != nullptr, sr_seed ? *sr_seed : 0);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// LayerNorm backward (layernorm_backward.h)

namespace {

struct LnShape {
    int64_t BT = 0, n = 0;
    size_t es = 0;
};

int ln_check_shape(int64_t B, int64_t T, int64_t C, int dtype, LnShape* s) {
    if (dtype != MMBWD_F32 && dtype != MMBWD_BF16) return MMBWD_ERR_DTYPE;
    if (B < 0 || T < 0 || C < 0) return MMBWD_ERR_SHAPE;
    if (!mul_ok(B, T, &s->BT) || !mul_ok(s->BT, C, &s->n)) return MMBWD_ERR_SHAPE;
    if (C > (dtype == MMBWD_F32 ? LNBWD_MAX_C_F32 : LNBWD_MAX_C_BF16)) return MMBWD_ERR_SHAPE;
    s->es = dtype == MMBWD_F32 ? 4 : 2;
    int64_t bytes = 0;
    if (!mul_ok(s->n, static_cast<int64_t>(s->es), &bytes)) return MMBWD_ERR_SHAPE;
    return MMBWD_OK;
}

int ln_num_sms(int* sms) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MMBWD_ERR_CUDA;
    return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? MMBWD_OK
                                                                                          : MMBWD_ERR_CUDA;
}

}  // namespace

size_t lnbwd_workspace_bytes(int64_t B, int64_t T, int64_t C, int dtype) {
    LnShape s;
    if (ln_check_shape(B, T, C, dtype, &s) != MMBWD_OK || s.BT == 0 || C == 0) return 0;
    if (C % ln_vec_elems(dtype) != 0) return 0;
    int sms = 0;
    if (ln_num_sms(&sms) != MMBWD_OK) return 0;
    LnPlan plan;
    if (ln_make_plan(s.BT, static_cast<int>(C), dtype, sms, &plan) != cudaSuccess) return 0;
    return plan.ws_bytes;
}

int lnbwd_run(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
              const float* mean, const float* rstd, int64_t B, int64_t T, int64_t C, int dtype,
              cudaStream_t stream) {
    NvtxRange nvtx("lnbwd_run");
    LnShape s;
    int rc = ln_check_shape(B, T, C, dtype, &s);
    if (rc != MMBWD_OK) return rc;
    const size_t es = s.es;
    const size_t b_rows = static_cast<size_t>(s.n) * es, b_col = static_cast<size_t>(C) * es,
                 b_stat = static_cast<size_t>(s.BT) * 4;
    // NULL only where the tensor is empty.
    if ((b_rows && (!dinp || !dout || !inp)) || (b_col && (!dweight || !dbias || !weight)) ||
        (b_stat && (!mean || !rstd)))
        return MMBWD_ERR_NULL;
    const void* vec_ptrs[6] = {dinp, dweight, dbias, dout, inp, weight};
    for (const void* p : vec_ptrs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(mean) | reinterpret_cast<uintptr_t>(rstd)) & 3u) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0) return MMBWD_ERR_ALIGN;

    const void* outs[3] = {dinp, dweight, dbias};
    const size_t nouts[3] = {b_rows, b_col, b_col};
    const void* ins[5] = {dout, inp, weight, mean, rstd};
    const size_t nins[5] = {b_rows, b_rows, b_col, b_stat, b_stat};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return MMBWD_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return MMBWD_ERR_ALIAS;
    }

    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    const Span spans[8] = {{dinp, b_rows}, {dweight, b_col}, {dbias, b_col},  {dout, b_rows},
                           {inp, b_rows},  {weight, b_col},  {mean, b_stat}, {rstd, b_stat}};
    rc = check_local(spans, 8, dev);
    if (rc != MMBWD_OK) return rc;
    if (s.BT == 0 || C == 0) return MMBWD_OK;  // empty sums: nothing changes
    int sms = 0;
    rc = ln_num_sms(&sms);
    if (rc != MMBWD_OK) return rc;
    LnPlan plan;
    if (ln_make_plan(s.BT, static_cast<int>(C), dtype, sms, &plan) != cudaSuccess) return MMBWD_ERR_CUDA;
    rc = ensure_workspace(*d, plan.ws_bytes, stream);
    if (rc != MMBWD_OK) return rc;
    const cudaError_t e = ln_launch(plan, dinp, dweight, dbias, dout, inp, weight, mean, rstd, s.BT,
                                    static_cast<int>(C), dtype, d->ws, stream);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// mmbwd_run_static_scratch: the backward pass without any device allocation.
// The split partials of the bf16 path live in a fixed file-scope device array
// instead of the grown workspace. In host code `g_static_scratch` only names
// a host-side stand-in, so its device address is looked up once per device
// with cudaGetSymbolAddress and that address is what the kernels receive.
namespace mmbwd {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MMBWD_STATIC_SCRATCH_BYTES];
void* g_static_scratch_addr[kMaxDevices];  // device address per device, set on first use

// The argument checks of mmbwd_run, for this entry point.
int check_run_args(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp, const void* weight,
                   int64_t B, int64_t T, int64_t C, int64_t OC, int dtype, Shape* s) {
    const int rc = check_shape(B, T, C, OC, dtype, s);
    if (rc != MMBWD_OK) return rc;
    const size_t es = s->es;
    const size_t b_dinp = static_cast<size_t>(s->n_dinp) * es, b_dw = static_cast<size_t>(s->n_dw) * es,
                 b_db = static_cast<size_t>(OC) * es, b_dout = static_cast<size_t>(s->n_dout) * es;
    if ((b_dinp && !dinp) || (b_dw && !dweight) || (b_dout && !dout) || (b_dinp && !inp) || (b_dw && !weight))
        return MMBWD_ERR_NULL;
    const void* ptrs[6] = {dinp, dweight, dbias, dout, inp, weight};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MMBWD_ERR_ALIGN;
    if ((static_cast<size_t>(C) * es) % 16 != 0 || (static_cast<size_t>(OC) * es) % 16 != 0) return MMBWD_ERR_ALIGN;
    const void* outs[3] = {dinp, dweight, dbias};
    const size_t nouts[3] = {b_dinp, b_dw, b_db};
    const void* ins[3] = {dout, inp, weight};
    const size_t nins[3] = {b_dout, b_dinp, b_dw};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j)
            if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return MMBWD_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return MMBWD_ERR_ALIAS;
    }
    return MMBWD_OK;
}

}  // namespace
}  // namespace mmbwd

extern "C" int mmbwd_run_static_scratch(void* dinp, void* dweight, void* dbias, const void* dout, const void* inp,
                                        const void* weight, int64_t B, int64_t T, int64_t C, int64_t OC, int dtype,
                                        cudaStream_t stream) {
    NvtxRange nvtx("mmbwd_run_static_scratch");
    Shape s;
    int rc = check_run_args(dinp, dweight, dbias, dout, inp, weight, B, T, C, OC, dtype, &s);
    if (rc != MMBWD_OK) return rc;

    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* d = nullptr;
    int dev = 0;
    rc = device_state(&d, &dev);
    if (rc != MMBWD_OK) return rc;
    {
        const size_t es = s.es, b_x = static_cast<size_t>(s.n_dinp) * es, b_w = static_cast<size_t>(s.n_dw) * es;
        const Span spans[6] = {{dinp, b_x},
                               {dweight, b_w},
                               {dbias, static_cast<size_t>(OC) * es},
                               {dout, static_cast<size_t>(s.n_dout) * es},
                               {inp, b_x},
                               {weight, b_w}};
        rc = check_local(spans, 6, dev);
        if (rc != MMBWD_OK) return rc;
    }
    if (!g_static_scratch_addr[dev]) {  // first call on this device: it is the current device
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr) {
            cudaGetLastError();
            return MMBWD_ERR_CUDA;
        }
        g_static_scratch_addr[dev] = addr;
    }

    cudaError_t e = cudaSuccess;
    if (OC == 0) return MMBWD_OK;
    if (s.BT == 0) {
        if (dbias) e = cudaMemsetAsync(dbias, 0, static_cast<size_t>(OC) * s.es, stream);
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    if (C == 0) {
        if (dbias) e = colsum_launch(dbias, dout, s.BT, OC, dtype, false, 0, stream);
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    if (dtype == MMBWD_F32) {  // neither fp32 path uses scratch: mmbwd_run's choice
        if (use_x3(s.BT, C, OC))
            e = x3_launch(static_cast<float*>(dinp), static_cast<float*>(dweight), static_cast<float*>(dbias),
                          static_cast<const float*>(dout), static_cast<const float*>(inp),
                          static_cast<const float*>(weight), s.BT, C, OC, d->num_sms, stream);
        else
            e = simt_launch(static_cast<float*>(dinp), static_cast<float*>(dweight), static_cast<float*>(dbias),
                            static_cast<const float*>(dout), static_cast<const float*>(inp),
                            static_cast<const float*>(weight), s.BT, C, OC, stream);
        return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
    }
    const TcPlan& plan = cached_plan(s.BT, C, OC, d->num_sms);
    if (plan.ws_bytes() > MMBWD_STATIC_SCRATCH_BYTES) return MMBWD_ERR_SCRATCH;
    e = tc_launch(plan, dinp, dweight, dbias, dout, inp, weight, s.BT, C, OC, g_static_scratch_addr[dev], stream);
    return e == cudaSuccess ? MMBWD_OK : MMBWD_ERR_CUDA;
}

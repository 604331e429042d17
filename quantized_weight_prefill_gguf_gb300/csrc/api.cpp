// api.cpp -- the C ABI declared in include/mq.h: argument validation,
// handles, the f16 cache, the split-K workspace, the device status word,
// tensor-map encoding, the M gate and dispatch to the kernels.
//
// Nothing here computes on the host: every step of the GEMM and of the
// decode runs in the library's CUDA kernels.  There is no CPU fallback; a
// missing device or kernel image is an error.
#include "mq.h"

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "mq_internal.h"

struct mq_weight {
    int type;
    int64_t N, K, ldk;
    int64_t nblocks;
    int qk, bb;
    const uint8_t *qdata;
    __half *cache;       // null when registered with MQ_REG_NO_CACHE
    bool cache_owned;    // false: cache is the caller's F16 weight itself
    int device;
    CUtensorMap tm_cache;
    int raw_g;           // > 0: the fused path reads raw blocks through raw_maps
    mq::RawMaps raw_maps;
    uint8_t *w8;         // MQ_REG_E4M3: e4m3 codes [N, ldk8], else null
    float *w8_scale;     // MQ_REG_E4M3: one scale per row [N]
    int64_t ldk8;
    CUtensorMap tm_w8;
};

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
std::unordered_set<mq_weight *> g_live;
thread_local std::string t_detail;
std::atomic<int64_t> g_launches{0};
std::atomic<int64_t> g_gate{-1};

struct DevState {
    bool init = false;
    int sms = 0;
    unsigned *status = nullptr;
    float *ws = nullptr;
    int64_t ws_bytes = 0;
};
DevState g_dev[kMaxDevices];

// ---------------------------------------------------------------- tracing
constexpr int64_t kTraceCap = 1 << 16;

struct TraceRec {
    mq_trace_record r;
    cudaEvent_t ev[3];
    bool aux;
};

std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;   // grows; events are reused across enables
int64_t g_trace_n = 0;

// Start a record for a call on stream s; returns its index or -1.
int64_t trace_begin(cudaStream_t s, int kind, int type, int64_t M, int64_t N, int64_t K)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace_on || g_trace_n >= kTraceCap)
        return -1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
        return -1;
    if (static_cast<int64_t>(g_trace.size()) <= g_trace_n) {
        TraceRec t{};
        for (auto &e : t.ev)
            if (cudaEventCreate(&e) != cudaSuccess)
                return -1;
        g_trace.push_back(t);
    }
    TraceRec &t = g_trace[g_trace_n];
    t.r = mq_trace_record{kind, type, M, N, K, 0.f, 0.f};
    t.aux = false;
    cudaEventRecord(t.ev[0], s);
    return g_trace_n++;
}

void trace_mark(int64_t idx, int which, cudaStream_t s, bool aux = false)
{
    if (idx < 0)
        return;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    cudaEventRecord(g_trace[idx].ev[which], s);
    if (which == 2)
        g_trace[idx].aux = aux;
}

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_detail = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(MQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool log_on()
{
    static int on = -1;
    if (on < 0) {
        const char *v = getenv("MQ_LOG");
        on = (v && *v && *v != '0') ? 1 : 0;
    }
    return on == 1;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// F32 / F16 / BF16: the weight is already a matrix of floats; its f16 form
// is the GEMM operand directly, so it has no fused path of its own.
bool is_float_type(int type) { return type == MQ_TYPE_F32 || type == MQ_TYPE_F16 || type == MQ_TYPE_BF16; }

const char *kTypeList = "F32=0, F16=1, Q4_0=2, Q5_0=6, Q5_1=7, Q8_0=8, Q4_K=12, Q5_K=13, Q6_K=14, BF16=30";

bool block_format(int type, int &qk, int &bb)
{
    switch (type) {
    case MQ_TYPE_F32: qk = 1; bb = 4; return true;
    case MQ_TYPE_F16: qk = 1; bb = 2; return true;
    case MQ_TYPE_BF16: qk = 1; bb = 2; return true;
    case MQ_TYPE_Q4_0: qk = 32; bb = 18; return true;
    case MQ_TYPE_Q5_0: qk = 32; bb = 22; return true;
    case MQ_TYPE_Q5_1: qk = 32; bb = 24; return true;
    case MQ_TYPE_Q8_0: qk = 32; bb = 34; return true;
    case MQ_TYPE_Q4_K: qk = 256; bb = 144; return true;
    case MQ_TYPE_Q5_K: qk = 256; bb = 176; return true;
    case MQ_TYPE_Q6_K: qk = 256; bb = 210; return true;
    default: return false;
    }
}

// Current device's state, created on first use: SM count, status word.
int device_state(DevState **out, int *dev_out = nullptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(MQ_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MQ_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevState &d = g_dev[dev];
    if (!d.init) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3)
            return fail(MQ_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                        prop.major, prop.minor);
        e = cudaMalloc(&d.status, sizeof(unsigned));
        if (e != cudaSuccess)
            return fail(MQ_ERR_OOM, "status word: %s", cudaGetErrorString(e));
        e = cudaMemset(d.status, 0, sizeof(unsigned));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(status)");
        d.sms = prop.multiProcessorCount;
        d.init = true;
    }
    *out = &d;
    if (dev_out)
        *dev_out = dev;
    return MQ_OK;
}

// Grow the workspace of `d` to `bytes` (synchronizes the device before
// freeing the old buffer, so no enqueued kernel still uses it).
int grow_workspace(DevState &d, int64_t bytes)
{
    if (bytes <= d.ws_bytes)
        return MQ_OK;
    if (d.ws) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize before workspace growth");
        cudaFree(d.ws);
        d.ws = nullptr;
        d.ws_bytes = 0;
    }
    void *p = nullptr;
    cudaError_t e = cudaMalloc(&p, static_cast<size_t>(bytes));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MQ_ERR_OOM, "split-K workspace of %lld bytes: %s", (long long)bytes, cudaGetErrorString(e));
    }
    d.ws = static_cast<float *>(p);
    d.ws_bytes = bytes;
    return MQ_OK;
}

int check_handle(mq_handle w)
{
    if (!w)
        return fail(MQ_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live.count(w))
        return fail(MQ_ERR_INVALID, "handle %p is not a live registered weight (released or never registered)",
                    (void *)w);
    return MQ_OK;
}

int64_t env_int(const char *name, int64_t dflt)
{
    const char *v = getenv(name);
    if (!v || !*v)
        return dflt;
    char *end = nullptr;
    long long x = strtoll(v, &end, 10);
    return (end && *end == '\0') ? x : dflt;
}

// Token count at and above which mq_gemm_auto takes the cached path: the
// measured fused/cached crossover on GB300.  The fused path's token tiles
// stop at 128, so from M = 129 on it decodes every weight tile once per
// token tile; back to back, the fused path is faster up to M = 128 and the
// cached path from M = 129 on every shape measured (7B gate, down and o, the
// Q8_0 pair, the Llama-3.1-8B gate; e.g. 7B down at M = 160: 37.0 us cached
// against 54.7 us fused).
int64_t current_gate()
{
    int64_t g = g_gate.load();
    if (g > 0)
        return g;
    return env_int("MQ_M_GATE", 129);
}

// Whether 256-token tiles run as 2-SM MMAs (tcgen05.mma.cta_group::2,
// the default; MQ_2SM=0 keeps multicast CTA pairs).
bool two_sm_wanted() { return env_int("MQ_2SM", 1) != 0; }

// Clusters of two to plan the cached or e4m3 GEMM with (0: single CTAs).
// CTA pairs (on unless MQ_PAIR=0, for tiles at least 64 tokens wide, when
// the device can hold clusters of two of the kernel) take adjacent weight-row
// tiles of one token tile: at 256 tokens as one 2-SM MMA tile, narrower as
// two CTAs sharing the token tile by multicast.
int pair_clusters(int64_t M, int64_t N, int64_t K, int sms, int bn_override, int kstep, bool e4m3)
{
    if (env_int("MQ_PAIR", 1) == 0)
        return 0;
    const mq::GemmPlan p0 = mq::plan_gemm(M, N, K, sms, false, 0, bn_override, kstep);
    return p0.bn >= 64 ? mq::pair_clusters_for(p0.bn, e4m3, p0.bn == 256 && two_sm_wanted()) : 0;
}

// 2-SM MMAs for a CTA-pair plan with 256-token tiles.
int two_sm_on(const mq::GemmPlan &p)
{
    return (p.pair && p.bn == 256 && two_sm_wanted()) ? 1 : 0;
}

// Plan, workspace and launch of one GEMM: one weight (cached or fused), or a
// group of weights that share K and X (cached; every member's N a multiple
// of 128), run as one weight stacked along N.
int run_gemm_group(const void *x, const mq_handle *ws, float *const *ys, int count, int64_t M, cudaStream_t s,
                   bool fused)
{
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    const mq_handle w = ws[0];
    int64_t n_total = 0;
    for (int g = 0; g < count; ++g)
        n_total += ws[g]->N;

    const bool splitk_on = env_int("MQ_SPLITK", 1) != 0;
    // Tuning override of the cached path's tile width (tokens per tile).
    int bn_override = static_cast<int>(env_int("MQ_BN", 0));
    if (bn_override != 32 && bn_override != 64 && bn_override != 128 && bn_override != 256)
        bn_override = 0;
    const int pc = fused ? 0 : pair_clusters(M, n_total, w->K, d->sms, bn_override, mq::kKStepF16, false);
    const int64_t want =
        splitk_on ? mq::plan_ws_bytes_wanted(M, n_total, w->K, d->sms, fused, bn_override, mq::kKStepF16, pc) : 0;
    if (want > d->ws_bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(s, &cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaStreamIsCapturing");
        if (cs == cudaStreamCaptureStatusNone) {
            std::lock_guard<std::mutex> lk(g_mu);
            rc = grow_workspace(*d, want);
            if (rc)
                return rc;
        }
    }
    mq::GemmPlan plan =
        mq::plan_gemm(M, n_total, w->K, d->sms, fused, splitk_on ? d->ws_bytes : 0, bn_override, mq::kKStepF16, pc);
    plan.two_sm = two_sm_on(plan);

    CUtensorMap tm_x;
    CUresult cr = mq::encode_f16_2d(&tm_x, x, M, w->K, w->K, 64, plan.pair ? plan.bn / 2 : plan.bn);
    if (cr != CUDA_SUCCESS)
        return fail(MQ_ERR_CUDA, "tensor map for x (M=%lld, K=%lld, box 64x%d): CUresult %d", (long long)M,
                    (long long)w->K, plan.bn, (int)cr);

    mq::GemmArgs a{};
    a.y = ys[0];
    a.ws = d->ws;
    a.status = d->status;
    a.wq = w->qdata;
    a.M = M;
    a.N = n_total;
    a.K = w->K;
    a.m_tiles = static_cast<int>((M + plan.bn - 1) / plan.bn);
    a.kblocks = static_cast<int>((w->K + 63) / 64);
    a.full_tiles = plan.full_tiles;
    a.split = plan.split;
    a.units = plan.units;
    a.kb_align = plan.kb_align;
    a.qtype = w->type;
    a.pair = plan.pair;
    a.groups = count;
    mq::WMaps maps{};
    mq::RawMapsG raw{};
    int nt = 0;
    for (int g = 0; g < count; ++g) {
        a.g_tile0[g] = nt;
        a.g_y[g] = ys[g];
        a.g_N[g] = ws[g]->N;
        a.g_wq[g] = ws[g]->qdata;
        nt += static_cast<int>((ws[g]->N + 127) / 128);
        if (fused)
            raw.w[g] = ws[g]->raw_maps;
        else
            maps.m[g] = ws[g]->tm_cache;
    }
    a.g_tile0[count] = nt;
    a.n_tiles = nt;

    if (log_on())
        fprintf(stderr, "[mq] %s M=%lld N=%lld K=%lld groups=%d bn=%d tiles=%d split=%d full=%d units=%d grid=%d\n",
                fused ? "fused" : "cached", (long long)M, (long long)n_total, (long long)w->K, count, plan.bn,
                plan.tiles, plan.split, plan.full_tiles, plan.units, plan.grid);

    const int64_t tr = trace_begin(s, fused ? MQ_TRACE_GEMM_FUSED : MQ_TRACE_GEMM_CACHED, w->type, M, n_total, w->K);
    a.raw_g = w->raw_g;
    a.raw_rb = w->K / w->qk * w->bb;
    // Failure injection for tests: the weight producer issues nothing, the
    // kernel's bounded waits run out (about 1 s), it exits cleanly and
    // mq_stream_status() reports MQ_ERR_DEVICE.
    a.stall_producer = env_int("MQ_INJECT_PRODUCER_STALL", 0) != 0 ? 1 : 0;
    if (!fused)
        mq::set_output_maps(maps, a);
    cudaError_t e = fused ? mq::launch_gemm_fused(tm_x, raw, a, plan, s)
                          : mq::launch_gemm_cached(maps, tm_x, a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fused ? "fused GEMM launch" : "cached GEMM launch");
    trace_mark(tr, 1, s);
    e = mq::launch_splitk_reduce(a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "split-K reduce launch");
    trace_mark(tr, 2, s, plan.split > 1 && plan.tiles > plan.full_tiles);
    return MQ_OK;
}

int run_gemm(const void *x, mq_handle w, float *y, int64_t M, cudaStream_t s, bool fused)
{
    return run_gemm_group(x, &w, &y, 1, M, s, fused);
}

int check_gemm_args(const void *x, mq_handle w, float *y, int64_t M)
{
    int rc = check_handle(w);
    if (rc)
        return rc;
    if (!x)
        return fail(MQ_ERR_INVALID, "x is NULL");
    if (!y)
        return fail(MQ_ERR_INVALID, "y is NULL");
    if (M < 1)
        return fail(MQ_ERR_SHAPE, "M=%lld: need M >= 1", (long long)M);
    if (M > 0x7FFFFFFFLL)
        return fail(MQ_ERR_SHAPE, "M=%lld exceeds 2^31-1", (long long)M);
    if (!aligned16(x))
        return fail(MQ_ERR_ALIGN, "x=%p is not 16-byte aligned", x);
    if (!aligned16(y))
        return fail(MQ_ERR_ALIGN, "y=%p is not 16-byte aligned", (void *)y);
    return MQ_OK;
}

}  // namespace

namespace mq {

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool pdl_enabled()
{
    static const bool on = env_int("MQ_PDL", 1) != 0;
    return on;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {

CUresult encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, int esize, const void *base, int64_t rows,
                   int64_t cols, int64_t ld, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                   CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
{
    static PFN_encodeTiled fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return CUDA_ERROR_NOT_FOUND;
        fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

CUresult encode_f32_out_2d(CUtensorMap *map, void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows)
{
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, ld, 128, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

void set_output_maps(WMaps &maps, GemmArgs &a)
{
    a.y_tma = 0;
    if (env_int("MQ_TMA_Y", 1) == 0)
        return;
    for (int g = 0; g < a.groups; ++g) {
        const uintptr_t b = reinterpret_cast<uintptr_t>(a.g_y[g]);
        if ((b & 15u) != 0 || (a.g_N[g] & 3) != 0)
            return;
        if (encode_f32_out_2d(&maps.y[g], a.g_y[g], a.M, a.g_N[g], a.g_N[g], kYBoxRows) != CUDA_SUCCESS)
            return;
    }
    a.y_tma = 1;
}

CUresult encode_f16_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                       int box_rows)
{
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, rows, cols, ld, box_cols, box_rows);
}

CUresult encode_u8_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                      int box_rows)
{
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, ld, box_cols, box_rows);
}

int set_error(int code, const char *what, cudaError_t e)
{
    if (e != cudaSuccess)
        return fail(code, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return fail(code, "%s", what);
}

// The cached GEMM with caller-provided split-K scratch and status word; it
// allocates nothing (no device_state(), no workspace growth).  Rejects a
// problem whose split-K plan needs more than scratch_bytes.
int gemm_cached_into_scratch(const void *x, mq_handle w, float *y, int64_t M, cudaStream_t s, float *scratch,
                             int64_t scratch_bytes, unsigned *status)
{
    int rc = check_gemm_args(x, w, y, M);
    if (rc)
        return rc;
    if (!w->cache)
        return fail(MQ_ERR_NO_CACHE, "weight was registered with MQ_REG_NO_CACHE; this entry point reads the f16 cache");
    int dev = 0, sms = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    if (major != 10 || minor != 3)
        return fail(MQ_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    if (dev != w->device)
        return fail(MQ_ERR_INVALID, "weight was registered on device %d, current device is %d", w->device, dev);
    // One plan, made as if scratch were unlimited, is both checked against
    // the scratch size and launched, so the check cannot drift from what the
    // kernels write.  Single CTAs only (no pair clusters, no 2-SM MMAs).
    const GemmPlan plan = plan_gemm(M, w->N, w->K, sms, false, INT64_MAX);
    if (plan.pair != 0 || plan.two_sm != 0)
        return fail(MQ_ERR_INVALID, "internal: the scratch plan must use single CTAs");
    if (plan.ws_bytes > scratch_bytes)
        return fail(MQ_ERR_SHAPE,
                    "M=%lld N=%lld K=%lld needs %lld bytes of split-K scratch; the static scratch holds %lld bytes",
                    (long long)M, (long long)w->N, (long long)w->K, (long long)plan.ws_bytes,
                    (long long)scratch_bytes);

    CUtensorMap tm_x;
    CUresult cr = encode_f16_2d(&tm_x, x, M, w->K, w->K, 64, plan.bn);
    if (cr != CUDA_SUCCESS)
        return fail(MQ_ERR_CUDA, "tensor map for x (M=%lld, K=%lld, box 64x%d): CUresult %d", (long long)M,
                    (long long)w->K, plan.bn, (int)cr);
    GemmArgs a{};
    a.y = y;
    a.ws = scratch;
    a.status = status;
    a.wq = w->qdata;
    a.M = M;
    a.N = w->N;
    a.K = w->K;
    a.m_tiles = static_cast<int>((M + plan.bn - 1) / plan.bn);
    a.n_tiles = static_cast<int>((w->N + 127) / 128);
    a.kblocks = static_cast<int>((w->K + 63) / 64);
    a.full_tiles = plan.full_tiles;
    a.split = plan.split;
    a.units = plan.units;
    a.kb_align = plan.kb_align;
    a.qtype = w->type;
    a.groups = 1;
    a.g_tile0[0] = 0;
    a.g_tile0[1] = a.n_tiles;
    a.g_y[0] = y;
    a.g_N[0] = w->N;
    WMaps maps{};
    maps.m[0] = w->tm_cache;
    set_output_maps(maps, a);
    e = launch_gemm_cached(maps, tm_x, a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cached GEMM launch");
    e = launch_splitk_reduce(a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "split-K reduce launch");
    return MQ_OK;
}

}  // namespace mq

extern "C" {

int mq_version(void) { return 100; }

int64_t mq_launch_count(void) { return g_launches.load(); }

const char *mq_last_error_detail(void) { return t_detail.c_str(); }

const char *mq_error_string(int status)
{
    switch (status) {
    case MQ_OK: return "ok";
    case MQ_ERR_INVALID: return "invalid argument or handle";
    case MQ_ERR_UNSUPPORTED_TYPE: return "unsupported block type";
    case MQ_ERR_SHAPE: return "shape precondition violated";
    case MQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MQ_ERR_NO_CACHE: return "weight has no f16 cache";
    case MQ_ERR_OOM: return "device allocation failed";
    case MQ_ERR_CUDA: return "CUDA error";
    case MQ_ERR_DEVICE: return "device-side error flagged by a kernel";
    case MQ_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
    }
}

int mq_register_weight(mq_type type, const void *qdata, int64_t N, int64_t K, uint32_t flags, void *stream,
                       mq_handle *out)
{
    if (!out)
        return fail(MQ_ERR_INVALID, "out is NULL");
    *out = nullptr;
    int qk = 0, bb = 0;
    if (!block_format(type, qk, bb))
        return fail(MQ_ERR_UNSUPPORTED_TYPE, "type id %d is not supported (supported: %s); the weight has no kernel",
                    (int)type, kTypeList);
    if (flags & ~(MQ_REG_NO_CACHE | MQ_REG_NO_KPAD | MQ_REG_KPAD | MQ_REG_E4M3))
        return fail(MQ_ERR_INVALID, "unknown flag bits 0x%x", flags);
    if ((flags & MQ_REG_NO_KPAD) && (flags & MQ_REG_KPAD))
        return fail(MQ_ERR_INVALID, "MQ_REG_NO_KPAD and MQ_REG_KPAD are exclusive");
    if (!qdata)
        return fail(MQ_ERR_INVALID, "qdata is NULL");
    if (N < 1 || K < 8 || (K % 8) != 0)
        return fail(MQ_ERR_SHAPE, "N=%lld K=%lld: need N >= 1, K >= 8, K %% 8 == 0", (long long)N, (long long)K);
    if (N > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL)
        return fail(MQ_ERR_SHAPE, "N=%lld K=%lld: each must be below 2^31", (long long)N, (long long)K);
    if ((N * K) % qk != 0)
        return fail(MQ_ERR_SHAPE, "N*K=%lld is not a whole number of %d-element blocks", (long long)(N * K), qk);
    if (!aligned16(qdata))
        return fail(MQ_ERR_ALIGN, "qdata=%p is not 16-byte aligned", qdata);
    if ((flags & MQ_REG_E4M3) && ((flags & MQ_REG_NO_CACHE) || K % 16 != 0))
        return fail(MQ_ERR_INVALID, "MQ_REG_E4M3 quantizes the f16 cache: it needs the cache (no MQ_REG_NO_CACHE) "
                                    "and K %% 16 == 0 (K=%lld)", (long long)K);
    if ((flags & MQ_REG_NO_CACHE) && (type == MQ_TYPE_F32 || type == MQ_TYPE_BF16))
        return fail(MQ_ERR_INVALID, "type %d: an F32 or BF16 weight is read through its f16 copy; MQ_REG_NO_CACHE "
                                    "applies to block formats and F16", (int)type);

    DevState *d = nullptr;
    int dev = 0;
    int rc = device_state(&d, &dev);
    if (rc)
        return rc;

    int64_t ldk = K;
    const int64_t kpad_env = env_int("MQ_KPAD", -1);   // 0: never, 1: always, else by rule
    if (flags & MQ_REG_KPAD)
        ldk = K + 64;
    else if (flags & MQ_REG_NO_KPAD)
        ldk = K;
    else if (kpad_env == 0)
        ldk = K;
    else if (kpad_env == 1)
        ldk = K + 64;
    else
        ldk = ((2 * K) % 2048 == 0) ? K + 64 : K;

    mq_weight *w = new mq_weight();
    w->type = type;
    w->N = N;
    w->K = K;
    w->ldk = ldk;
    w->qk = qk;
    w->bb = bb;
    w->nblocks = N * K / qk;
    w->qdata = static_cast<const uint8_t *>(qdata);
    w->cache = nullptr;
    w->cache_owned = false;
    w->w8 = nullptr;
    w->w8_scale = nullptr;
    w->ldk8 = 0;
    w->device = dev;
    w->raw_g = env_int("MQ_RAW_TMA", 1) ? mq::encode_raw_maps(&w->raw_maps, qdata, type, N, K) : 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (type == MQ_TYPE_F16 && (ldk == K || (flags & MQ_REG_NO_CACHE))) {
        // An F16 weight whose rows need no padding is the GEMM operand as it
        // stands: read it in place (no copy, nothing allocated).
        w->ldk = K;
        w->cache = static_cast<__half *>(const_cast<void *>(qdata));
        CUresult cr = mq::encode_f16_2d(&w->tm_cache, w->cache, N, K, K, 64, 128);
        if (cr != CUDA_SUCCESS) {
            delete w;
            return fail(MQ_ERR_CUDA, "tensor map for the F16 weight: CUresult %d", (int)cr);
        }
    } else if (!(flags & MQ_REG_NO_CACHE)) {
        const size_t bytes = static_cast<size_t>(N) * static_cast<size_t>(ldk) * 2;
        void *p = nullptr;
        cudaError_t e = env_int("MQ_FAULT_ALLOC", 0) ? cudaErrorMemoryAllocation : cudaMalloc(&p, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            delete w;
            return fail(MQ_ERR_OOM, "f16 cache of %zu bytes (N=%lld, ldk=%lld): %s", bytes, (long long)N,
                        (long long)ldk, cudaGetErrorString(e));
        }
        w->cache = static_cast<__half *>(p);
        w->cache_owned = true;
        const int64_t tr = trace_begin(s, MQ_TRACE_DECODE, type, 0, N, K);
        e = mq::launch_dequant(type, qdata, w->nblocks, w->cache, K, ldk, s);
        trace_mark(tr, 1, s);
        trace_mark(tr, 2, s);
        if (e == cudaSuccess && ldk > K)
            e = cudaMemset2DAsync(w->cache + K, static_cast<size_t>(ldk) * 2, 0, static_cast<size_t>(ldk - K) * 2,
                                  static_cast<size_t>(N), s);
        if (e != cudaSuccess) {
            cudaFree(w->cache);
            delete w;
            return cuda_fail(e, "decode into the f16 cache");
        }
        CUresult cr = mq::encode_f16_2d(&w->tm_cache, w->cache, N, K, ldk, 64, 128);
        if (cr != CUDA_SUCCESS) {
            cudaStreamSynchronize(s);
            cudaFree(w->cache);
            delete w;
            return fail(MQ_ERR_CUDA, "tensor map for the f16 cache: CUresult %d", (int)cr);
        }
    }
    if (flags & MQ_REG_E4M3) {
        // The 8-bit copy: each cache row quantized to e4m3 with its own
        // scale; rows padded by one 128-byte line when they are a multiple
        // of 2048 bytes (the cache's rule, in bytes).
        int64_t ldk8 = (K % 2048 == 0) ? K + 128 : K;
        if (flags & MQ_REG_KPAD)
            ldk8 = K + 128;
        else if (flags & MQ_REG_NO_KPAD)
            ldk8 = K;
        void *p8 = nullptr, *ps = nullptr;
        cudaError_t e = cudaMalloc(&p8, static_cast<size_t>(N) * static_cast<size_t>(ldk8));
        if (e == cudaSuccess)
            e = cudaMalloc(&ps, static_cast<size_t>(N) * sizeof(float));
        if (e != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p8);
            if (w->cache_owned) {
                cudaStreamSynchronize(s);
                cudaFree(w->cache);
            }
            delete w;
            return fail(MQ_ERR_OOM, "e4m3 copy of %lld x %lld bytes: %s", (long long)N, (long long)ldk8,
                        cudaGetErrorString(e));
        }
        w->w8 = static_cast<uint8_t *>(p8);
        w->w8_scale = static_cast<float *>(ps);
        w->ldk8 = ldk8;
        const int64_t tr = trace_begin(s, MQ_TRACE_DECODE, type, 0, N, K);
        e = mq::launch_quant_e4m3(w->cache, N, K, w->ldk, w->w8, ldk8, w->w8_scale, s);
        trace_mark(tr, 1, s);
        trace_mark(tr, 2, s);
        if (e == cudaSuccess && ldk8 > K)
            e = cudaMemset2DAsync(w->w8 + K, static_cast<size_t>(ldk8), 0, static_cast<size_t>(ldk8 - K),
                                  static_cast<size_t>(N), s);
        CUresult cr = CUDA_SUCCESS;
        if (e == cudaSuccess)
            cr = mq::encode_u8_2d(&w->tm_w8, w->w8, N, K, ldk8, 128, 128);
        if (e != cudaSuccess || cr != CUDA_SUCCESS) {
            cudaStreamSynchronize(s);
            cudaFree(w->w8);
            cudaFree(w->w8_scale);
            if (w->cache_owned)
                cudaFree(w->cache);
            delete w;
            return e != cudaSuccess ? cuda_fail(e, "e4m3 quantization of the cache")
                                    : fail(MQ_ERR_CUDA, "tensor map for the e4m3 copy: CUresult %d", (int)cr);
        }
    }
    if (log_on())
        fprintf(stderr, "[mq] register type=%d N=%lld K=%lld ldk=%lld cache=%s e4m3=%s\n", (int)type, (long long)N,
                (long long)K, (long long)ldk, w->cache ? "yes" : "no", w->w8 ? "yes" : "no");
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_live.insert(w);
    }
    *out = w;
    return MQ_OK;
}

int mq_release_weight(mq_handle w)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!w || !g_live.count(w))
            return fail(MQ_ERR_INVALID, "handle %p is not a live registered weight", (void *)w);
        g_live.erase(w);
    }
    if ((w->cache && w->cache_owned) || w->w8) {
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(w->device);
        cudaDeviceSynchronize();
        if (w->cache_owned)
            cudaFree(w->cache);
        cudaFree(w->w8);
        cudaFree(w->w8_scale);
        cudaSetDevice(cur);
    }
    delete w;
    return MQ_OK;
}

int mq_weight_info(mq_handle w, int64_t *N, int64_t *K, int64_t *ldk, const void **f16_cache)
{
    int rc = check_handle(w);
    if (rc)
        return rc;
    if (N) *N = w->N;
    if (K) *K = w->K;
    if (ldk) *ldk = w->ldk;
    if (f16_cache) *f16_cache = w->cache;
    return MQ_OK;
}

int mq_dequantize(mq_type type, const void *qdata, int64_t N, int64_t K, void *out_f16, int64_t ldo, void *stream)
{
    int qk = 0, bb = 0;
    if (!block_format(type, qk, bb))
        return fail(MQ_ERR_UNSUPPORTED_TYPE, "type id %d is not supported (%s)", (int)type, kTypeList);
    if (!qdata || !out_f16)
        return fail(MQ_ERR_INVALID, "%s is NULL", qdata ? "out_f16" : "qdata");
    if (N < 1 || K < 8 || (K % 8) != 0 || ldo < K || (ldo % 8) != 0)
        return fail(MQ_ERR_SHAPE, "N=%lld K=%lld ldo=%lld: need N >= 1, K >= 8, K %% 8 == 0, ldo >= K, ldo %% 8 == 0",
                    (long long)N, (long long)K, (long long)ldo);
    if ((N * K) % qk != 0)
        return fail(MQ_ERR_SHAPE, "N*K=%lld is not a whole number of %d-element blocks", (long long)(N * K), qk);
    if (!aligned16(qdata) || !aligned16(out_f16))
        return fail(MQ_ERR_ALIGN, "%s is not 16-byte aligned", aligned16(qdata) ? "out_f16" : "qdata");
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t tr = trace_begin(s, MQ_TRACE_DECODE, type, 0, N, K);
    cudaError_t e = mq::launch_dequant(type, qdata, N * K / qk, static_cast<__half *>(out_f16), K, ldo, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "dequantize launch");
    trace_mark(tr, 1, s);
    trace_mark(tr, 2, s);
    return MQ_OK;
}

int mq_gemm(const void *x, mq_handle w, float *y, int64_t M, void *stream)
{
    int rc = check_gemm_args(x, w, y, M);
    if (rc)
        return rc;
    if (!w->cache)
        return fail(MQ_ERR_NO_CACHE, "weight was registered with MQ_REG_NO_CACHE; use mq_gemm_fused");
    return run_gemm(x, w, y, M, static_cast<cudaStream_t>(stream), false);
}

int mq_gemm_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream)
{
    if (!w || !y)
        return fail(MQ_ERR_INVALID, "%s is NULL", w ? "y" : "w");
    if (count < 1 || count > mq::kMaxGroup)
        return fail(MQ_ERR_INVALID, "count=%d: need 1 <= count <= %d", count, mq::kMaxGroup);
    bool one_launch = true;
    for (int g = 0; g < count; ++g) {
        int rc = check_gemm_args(x, w[g], y[g], M);
        if (rc)
            return rc;
        if (!w[g]->cache)
            return fail(MQ_ERR_NO_CACHE, "member %d was registered with MQ_REG_NO_CACHE; grouped calls read the f16 cache", g);
        if (w[g]->K != w[0]->K)
            return fail(MQ_ERR_SHAPE, "member %d has K=%lld, member 0 has K=%lld: a group shares X", g,
                        (long long)w[g]->K, (long long)w[0]->K);
        if (w[g]->device != w[0]->device)
            return fail(MQ_ERR_INVALID, "member %d is registered on device %d, member 0 on %d", g, w[g]->device,
                        w[0]->device);
        if (w[g]->N % 128 != 0)
            one_launch = false;
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (one_launch || count == 1)
        return run_gemm_group(x, w, y, count, M, s, false);
    // A member whose N is not a multiple of the 128-row tile would share a
    // tile with the next member: run the members one after another instead.
    for (int g = 0; g < count; ++g) {
        int rc = run_gemm(x, w[g], y[g], M, s, false);
        if (rc)
            return rc;
    }
    return MQ_OK;
}

int mq_gemm_fused(const void *x, mq_handle w, float *y, int64_t M, void *stream)
{
    int rc = check_gemm_args(x, w, y, M);
    if (rc)
        return rc;
    if (is_float_type(w->type))   // nothing to decode on chip: the f16 operand exists
        return run_gemm(x, w, y, M, static_cast<cudaStream_t>(stream), false);
    if (w->K % 64 != 0)
        return fail(MQ_ERR_SHAPE, "fused path needs K %% 64 == 0 (K=%lld)", (long long)w->K);
    if (w->raw_g == 0 && (w->nblocks * w->bb) % 16 != 0)
        return fail(MQ_ERR_SHAPE, "fused path needs the block stream length (%lld bytes) to be a multiple of 16",
                    (long long)(w->nblocks * w->bb));
    return run_gemm(x, w, y, M, static_cast<cudaStream_t>(stream), true);
}

int mq_gemm_fused_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream)
{
    if (!w || !y)
        return fail(MQ_ERR_INVALID, "%s is NULL", w ? "y" : "w");
    if (count < 1 || count > mq::kMaxGroup)
        return fail(MQ_ERR_INVALID, "count=%d: need 1 <= count <= %d", count, mq::kMaxGroup);
    bool one_launch = true;
    for (int g = 0; g < count; ++g) {
        int rc = check_gemm_args(x, w[g], y[g], M);
        if (rc)
            return rc;
        if (w[g]->K != w[0]->K)
            return fail(MQ_ERR_SHAPE, "member %d has K=%lld, member 0 has K=%lld: a group shares X", g,
                        (long long)w[g]->K, (long long)w[0]->K);
        if (w[g]->type != w[0]->type)
            return fail(MQ_ERR_INVALID, "member %d has type %d, member 0 has type %d: a fused group decodes one format",
                        g, w[g]->type, w[0]->type);
        if (w[g]->device != w[0]->device)
            return fail(MQ_ERR_INVALID, "member %d is registered on device %d, member 0 on %d", g, w[g]->device,
                        w[0]->device);
        if (w[g]->raw_g != w[0]->raw_g)
            one_launch = false;
        if (w[g]->N % 128 != 0)
            one_launch = false;
    }
    if (is_float_type(w[0]->type))   // nothing to decode on chip: the f16 operands exist
        return mq_gemm_grouped(x, w, count, y, M, stream);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!one_launch || count == 1) {
        // A member whose N is not a multiple of the 128-row tile would share a
        // tile with the next one: run the members one after another instead.
        for (int g = 0; g < count; ++g) {
            int rc = mq_gemm_fused(x, w[g], y[g], M, stream);
            if (rc)
                return rc;
        }
        return MQ_OK;
    }
    if (w[0]->K % 64 != 0)
        return fail(MQ_ERR_SHAPE, "fused path needs K %% 64 == 0 (K=%lld)", (long long)w[0]->K);
    for (int g = 0; g < count; ++g)
        if (w[g]->raw_g == 0 && (w[g]->nblocks * w[g]->bb) % 16 != 0)
            return fail(MQ_ERR_SHAPE,
                        "fused path needs member %d's block stream length (%lld bytes) to be a multiple of 16", g,
                        (long long)(w[g]->nblocks * w[g]->bb));
    return run_gemm_group(x, w, y, count, M, s, true);
}

int mq_gemm_auto_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream)
{
    if (!w || !y)
        return fail(MQ_ERR_INVALID, "%s is NULL", w ? "y" : "w");
    if (count < 1 || count > mq::kMaxGroup)
        return fail(MQ_ERR_INVALID, "count=%d: need 1 <= count <= %d", count, mq::kMaxGroup);
    bool all_cached = true, fused_ok = true;
    for (int g = 0; g < count; ++g) {
        int rc = check_handle(w[g]);
        if (rc)
            return rc;
        all_cached = all_cached && w[g]->cache != nullptr;
        fused_ok = fused_ok && !is_float_type(w[g]->type) && w[g]->type == w[0]->type && w[g]->K % 64 == 0 &&
                   (w[g]->raw_g > 0 || (w[g]->nblocks * w[g]->bb) % 16 == 0);
    }
    if (!all_cached || (M < current_gate() && fused_ok))
        return mq_gemm_fused_grouped(x, w, count, y, M, stream);
    return mq_gemm_grouped(x, w, count, y, M, stream);
}

int mq_gemm_auto(const void *x, mq_handle w, float *y, int64_t M, void *stream)
{
    int rc = check_gemm_args(x, w, y, M);
    if (rc)
        return rc;
    const bool fused_ok = (w->K % 64 == 0) && (w->raw_g > 0 || (w->nblocks * w->bb) % 16 == 0);
    if (!w->cache || (M < current_gate() && fused_ok))
        return mq_gemm_fused(x, w, y, M, stream);
    return mq_gemm(x, w, y, M, stream);
}

int mq_gemm_scratch(const void *x, mq_handle w, float *y, int64_t M, void *scratch, int64_t scratch_bytes,
                    void *stream)
{
    int rc = check_gemm_args(x, w, y, M);
    if (rc)
        return rc;
    if (!scratch)
        return fail(MQ_ERR_INVALID, "scratch is NULL");
    if (!aligned16(scratch))
        return fail(MQ_ERR_ALIGN, "scratch=%p is not 16-byte aligned", scratch);
    const int64_t need = 2 * w->N * w->ldk;
    if (scratch_bytes < need)
        return fail(MQ_ERR_SHAPE, "scratch of %lld bytes; the f16 [N=%lld, ldk=%lld] weight needs %lld",
                    (long long)scratch_bytes, (long long)w->N, (long long)w->ldk, (long long)need);
    DevState *d = nullptr;
    rc = device_state(&d);
    if (rc)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    mq_weight tmp = *w;
    tmp.cache = static_cast<__half *>(scratch);
    tmp.cache_owned = false;
    CUresult cr = mq::encode_f16_2d(&tmp.tm_cache, tmp.cache, w->N, w->K, w->ldk, 64, 128);
    if (cr != CUDA_SUCCESS)
        return fail(MQ_ERR_CUDA, "tensor map for the scratch: CUresult %d", (int)cr);
    const int64_t tr = trace_begin(s, MQ_TRACE_DECODE, w->type, M, w->N, w->K);
    cudaError_t e = mq::launch_dequant(w->type, w->qdata, w->nblocks, tmp.cache, w->K, w->ldk, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode into the scratch");
    trace_mark(tr, 1, s);
    trace_mark(tr, 2, s);
    return run_gemm(x, &tmp, y, M, s, false);
}

int mq_debug_schedule(int64_t M, int64_t N, int64_t K, int sms, int path, int pair_clusters, int64_t *plan_out,
                      int32_t *units, int64_t cap, int64_t *count)
{
    if (M < 1 || N < 1 || K < 1 || sms < 1 || path < 0 || path > 2 || pair_clusters < 0 || !plan_out || !count ||
        (cap > 0 && !units))
        return fail(MQ_ERR_INVALID, "mq_debug_schedule: bad argument");
    const bool fused = path == 1;
    const int kstep = path == 2 ? mq::kKStepE4m3 : mq::kKStepF16;
    const mq::GemmPlan p = mq::plan_gemm(M, N, K, sms, fused, INT64_MAX, 0, kstep, fused ? 0 : pair_clusters);
    plan_out[0] = p.bn;
    plan_out[1] = p.pair;
    plan_out[2] = p.split;
    plan_out[3] = p.full_tiles;
    plan_out[4] = p.tiles;
    plan_out[5] = p.units;
    plan_out[6] = p.grid;
    plan_out[7] = p.ws_bytes;
    plan_out[8] = p.kb_align;
    *count = mq::schedule_units(p, M, N, K, kstep, units, cap);
    return MQ_OK;
}

int mq_debug_cvt_f16(uint32_t first, int64_t count, void *out, void *stream)
{
    if (!out)
        return fail(MQ_ERR_INVALID, "out is NULL");
    if (count < 0 || (count & 1) || (first & 1u) || count > (int64_t(1) << 32) - int64_t(first))
        return fail(MQ_ERR_SHAPE, "first=%u count=%lld: need even first and count, first + count <= 2^32", first,
                    (long long)count);
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0)
        return fail(MQ_ERR_ALIGN, "out=%p is not 4-byte aligned", out);
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    if (count == 0)
        return MQ_OK;
    cudaError_t e = mq::launch_debug_cvt_f16(first, count, static_cast<uint16_t *>(out),
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "f16 conversion launch");
    return MQ_OK;
}

int mq_weight_e4m3_info(mq_handle w, int64_t *ldk8, const void **codes, const float **scales)
{
    int rc = check_handle(w);
    if (rc)
        return rc;
    if (ldk8) *ldk8 = w->ldk8;
    if (codes) *codes = w->w8;
    if (scales) *scales = w->w8_scale;
    return MQ_OK;
}

int mq_quantize_e4m3(const void *x, int64_t rows, int64_t K, int64_t ld, void *dst, int64_t ldo, float *scales,
                     void *stream)
{
    if (!x || !dst || !scales)
        return fail(MQ_ERR_INVALID, "%s is NULL", !x ? "x" : (!dst ? "dst" : "scales"));
    if (rows < 1 || K < 16 || K % 16 != 0 || ld < K || ld % 8 != 0 || ldo < K || ldo % 16 != 0)
        return fail(MQ_ERR_SHAPE,
                    "rows=%lld K=%lld ld=%lld ldo=%lld: need rows >= 1, K %% 16 == 0, ld >= K, ld %% 8 == 0, "
                    "ldo >= K, ldo %% 16 == 0",
                    (long long)rows, (long long)K, (long long)ld, (long long)ldo);
    if (!aligned16(x) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(scales) & 3u))
        return fail(MQ_ERR_ALIGN, "x and dst must be 16-byte aligned, scales 4-byte aligned");
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    cudaError_t e = mq::launch_quant_e4m3(static_cast<const __half *>(x), rows, K, ld, static_cast<uint8_t *>(dst),
                                          ldo, scales, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "e4m3 quantization launch");
    return MQ_OK;
}

namespace {

// Plan, workspace and launch of one e4m3 GEMM launch: one weight, or a group
// of weights sharing K and the quantized X (every member's N a multiple of
// 128), stacked along N as in run_gemm_group.
int run_e4m3_group(const void *x8, const float *x_scale, const mq_handle *ws, float *const *ys, int count, int64_t M,
                   cudaStream_t s)
{
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    const mq_handle w = ws[0];
    int64_t n_total = 0;
    for (int g = 0; g < count; ++g)
        n_total += ws[g]->N;
    const bool splitk_on = env_int("MQ_SPLITK", 1) != 0;
    const int pc = pair_clusters(M, n_total, w->K, d->sms, 0, mq::kKStepE4m3, true);
    const int64_t want =
        splitk_on ? mq::plan_ws_bytes_wanted(M, n_total, w->K, d->sms, false, 0, mq::kKStepE4m3, pc) : 0;
    if (want > d->ws_bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(s, &cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaStreamIsCapturing");
        if (cs == cudaStreamCaptureStatusNone) {
            std::lock_guard<std::mutex> lk(g_mu);
            rc = grow_workspace(*d, want);
            if (rc)
                return rc;
        }
    }
    mq::GemmPlan plan =
        mq::plan_gemm(M, n_total, w->K, d->sms, false, splitk_on ? d->ws_bytes : 0, 0, mq::kKStepE4m3, pc);
    plan.two_sm = two_sm_on(plan);
    CUtensorMap tm_x;
    CUresult cr = mq::encode_u8_2d(&tm_x, x8, M, w->K, w->K, 128, plan.pair ? plan.bn / 2 : plan.bn);
    if (cr != CUDA_SUCCESS)
        return fail(MQ_ERR_CUDA, "tensor map for x8 (M=%lld, K=%lld): CUresult %d", (long long)M, (long long)w->K,
                    (int)cr);
    mq::GemmArgs a{};
    a.y = ys[0];
    a.ws = d->ws;
    a.status = d->status;
    a.M = M;
    a.N = n_total;
    a.K = w->K;
    a.m_tiles = static_cast<int>((M + plan.bn - 1) / plan.bn);
    a.kblocks = static_cast<int>((w->K + mq::kKStepE4m3 - 1) / mq::kKStepE4m3);
    a.full_tiles = plan.full_tiles;
    a.split = plan.split;
    a.units = plan.units;
    a.kb_align = plan.kb_align;
    a.qtype = w->type;
    a.pair = plan.pair;
    a.x_scale = x_scale;
    a.stall_producer = env_int("MQ_INJECT_PRODUCER_STALL", 0) != 0 ? 1 : 0;   // failure injection (tests)
    a.groups = count;
    mq::WMaps maps{};
    int nt = 0;
    for (int g = 0; g < count; ++g) {
        a.g_tile0[g] = nt;
        a.g_y[g] = ys[g];
        a.g_N[g] = ws[g]->N;
        a.g_wscale[g] = ws[g]->w8_scale;
        maps.m[g] = ws[g]->tm_w8;
        nt += static_cast<int>((ws[g]->N + 127) / 128);
    }
    a.g_tile0[count] = nt;
    a.n_tiles = nt;
    mq::set_output_maps(maps, a);
    const int64_t tr = trace_begin(s, MQ_TRACE_GEMM_CACHED, w->type, M, n_total, w->K);
    cudaError_t e = mq::launch_gemm_e4m3(maps, tm_x, a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "e4m3 GEMM launch");
    trace_mark(tr, 1, s);
    e = mq::launch_splitk_reduce(a, plan, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "split-K reduce launch");
    trace_mark(tr, 2, s, plan.split > 1 && plan.tiles > plan.full_tiles);
    return MQ_OK;
}

}  // namespace

int mq_gemm_e4m3(const void *x8, const float *x_scale, mq_handle w, float *y, int64_t M, void *stream)
{
    return mq_gemm_e4m3_grouped(x8, x_scale, &w, 1, &y, M, stream);
}

int mq_gemm_e4m3_grouped(const void *x8, const float *x_scale, const mq_handle *w, int count, float *const *y,
                         int64_t M, void *stream)
{
    if (!w || !y)
        return fail(MQ_ERR_INVALID, "%s is NULL", w ? "y" : "w");
    if (!x_scale)
        return fail(MQ_ERR_INVALID, "x_scale is NULL");
    if (count < 1 || count > mq::kMaxGroup)
        return fail(MQ_ERR_INVALID, "count=%d: need 1 <= count <= %d", count, mq::kMaxGroup);
    bool one_launch = true;
    for (int g = 0; g < count; ++g) {
        int rc = check_gemm_args(x8, w[g], y[g], M);
        if (rc)
            return rc;
        if (!w[g]->w8)
            return fail(MQ_ERR_NO_CACHE, "member %d was registered without MQ_REG_E4M3: it has no e4m3 copy", g);
        if (w[g]->K != w[0]->K)
            return fail(MQ_ERR_SHAPE, "member %d has K=%lld, member 0 has K=%lld: a group shares X", g,
                        (long long)w[g]->K, (long long)w[0]->K);
        if (w[g]->device != w[0]->device)
            return fail(MQ_ERR_INVALID, "member %d is registered on device %d, member 0 on %d", g, w[g]->device,
                        w[0]->device);
        if (w[g]->N % 128 != 0)
            one_launch = false;
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (one_launch || count == 1)
        return run_e4m3_group(x8, x_scale, w, y, count, M, s);
    for (int g = 0; g < count; ++g) {
        int rc = run_e4m3_group(x8, x_scale, &w[g], &y[g], 1, M, s);
        if (rc)
            return rc;
    }
    return MQ_OK;
}

int64_t mq_get_m_gate(void) { return current_gate(); }

int mq_set_m_gate(int64_t m)
{
    if (m < 1)
        return fail(MQ_ERR_INVALID, "gate %lld: need >= 1", (long long)m);
    g_gate.store(m);
    return MQ_OK;
}

int mq_reserve_workspace(int64_t bytes)
{
    if (bytes < 0)
        return fail(MQ_ERR_INVALID, "bytes=%lld < 0", (long long)bytes);
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    return grow_workspace(*d, bytes);
}

int mq_trace_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (on)
        g_trace_n = 0;
    g_trace_on = on != 0;
    return MQ_OK;
}

int64_t mq_trace_count(void)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    return g_trace_n;
}

int mq_trace_read(int64_t i, mq_trace_record *out)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!out || i < 0 || i >= g_trace_n)
        return fail(MQ_ERR_INVALID, "trace record %lld does not exist (count %lld)", (long long)i,
                    (long long)g_trace_n);
    TraceRec &t = g_trace[i];
    cudaError_t e = cudaEventSynchronize(t.ev[2]);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaEventSynchronize(trace)");
    float a = 0.f, b = 0.f;
    e = cudaEventElapsedTime(&a, t.ev[0], t.ev[1]);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaEventElapsedTime(trace)");
    if (t.aux) {
        e = cudaEventElapsedTime(&b, t.ev[1], t.ev[2]);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaEventElapsedTime(trace)");
    }
    *out = t.r;
    out->ms_main = a;
    out->ms_aux = b;
    return MQ_OK;
}

int mq_stream_status(void *stream)
{
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc)
        return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    unsigned st = 0;
    e = cudaMemcpy(&st, d->status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the device status word");
    st |= mq::noalloc_take_status();
    if (st != 0) {
        cudaMemset(d->status, 0, sizeof st);
        return fail(MQ_ERR_DEVICE, "device status 0x%x:%s%s", st, (st & 1u) ? " pipeline wait timed out" : "",
                    (st & 2u) ? " kernel rejected its arguments" : "");
    }
    return MQ_OK;
}

}  // extern "C"

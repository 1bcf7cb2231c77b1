// ssd_api.cu -- the C ABI of libssd: validation, path choice, scratch memory,
// launches.  Every entry point only enqueues on the caller's stream (except
// the host-buffer variant, which synchronises it at the end).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

std::atomic<uint64_t> g_launches{0};

size_t elem_size(int dtype) { return dtype == SSD_DTYPE_BF16 ? 2 : 4; }

bool mul_ok(int64_t a, int64_t b, int64_t *out)
{
    if (a < 0 || b < 0)
        return false;
    if (a != 0 && b > INT64_MAX / a)
        return false;
    *out = a * b;
    return true;
}

struct Sizes {
    int64_t x, dt, bc, par, state;  // bytes
};

ssd_status_t check_dims(const ssd_dims_t *d, Sizes *sz)
{
    if (!d)
        return SSD_ERR_NULL_PTR;
    if (d->reserved != 0 || d->batch < 0 || d->seqlen < 0 || d->nheads < 1 || d->headdim < 1 ||
        d->dstate < 1 || d->ngroups < 1 || d->chunk < 1 || d->nheads % d->ngroups != 0)
        return SSD_ERR_INVALID_DIMS;
    if (d->dtype != SSD_DTYPE_F32 && d->dtype != SSD_DTYPE_BF16)
        return SSD_ERR_UNSUPPORTED_DTYPE;
    const uint32_t path = d->flags & SSD_PATH_MASK;
    if ((d->flags & ~(SSD_PATH_MASK | SSD_SCHEDULE_REQUEST_MASK | SSD_DIAG_STALL_HANDOFF)) != 0 ||
        path > SSD_PATH_DECODE)
        return SSD_ERR_INVALID_DIMS;
    int64_t bl, blh, t;
    const int64_t es = (int64_t)elem_size(d->dtype);
    if (!mul_ok(d->batch, d->seqlen, &bl) || !mul_ok(bl, d->nheads, &blh) ||
        !mul_ok(blh, d->headdim, &t) || !mul_ok(t, es, &sz->x) || !mul_ok(blh, 4, &sz->dt))
        return SSD_ERR_INVALID_DIMS;
    if (!mul_ok(bl, d->ngroups, &t) || !mul_ok(t, d->dstate, &t) || !mul_ok(t, es, &sz->bc))
        return SSD_ERR_INVALID_DIMS;
    sz->par = (int64_t)d->nheads * 4;
    if (!mul_ok(d->batch, d->nheads, &t) || !mul_ok(t, d->headdim, &t) ||
        !mul_ok(t, d->dstate, &t) || !mul_ok(t, 4, &sz->state))
        return SSD_ERR_INVALID_DIMS;
    if (sz->x > (INT64_C(1) << 46) || sz->state > (INT64_C(1) << 46) || d->seqlen >= (INT64_C(1) << 31))
        return SSD_ERR_INVALID_DIMS;
    return SSD_OK;
}

ScanArgs make_args(const void *x, const float *dt_raw, const float *dt_bias, const float *A_log,
                   const void *B, const void *C, const float *D, const float *init_state, void *y,
                   float *final_state, const ssd_dims_t *d)
{
    ScanArgs a;
    a.x = x;
    a.dt_raw = dt_raw;
    a.dt_bias = dt_bias;
    a.A_log = A_log;
    a.B = B;
    a.C = C;
    a.D = D;
    a.init_state = init_state;
    a.y = y;
    a.final_state = final_state;
    a.batch = d->batch;
    a.seqlen = d->seqlen;
    a.nheads = d->nheads;
    a.headdim = d->headdim;
    a.dstate = d->dstate;
    a.ngroups = d->ngroups;
    a.chunk = d->chunk;
    a.dtype = d->dtype;
    a.diag_stall = (d->flags & SSD_DIAG_STALL_HANDOFF) != 0;
    a.sched_req = (int)((d->flags & SSD_SCHEDULE_REQUEST_MASK) >> SSD_SCHEDULE_SHIFT);
    return a;
}

bool overlaps(const void *p, int64_t pn, const void *q, int64_t qn)
{
    if (!p || !q || pn <= 0 || qn <= 0)
        return false;
    const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
    return a < b + (uintptr_t)qn && b < a + (uintptr_t)pn;
}

bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

bool device_is_gb300_class()
{
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return false;
    return major == 10 && minor == 3;
}

// Why the chunked path refuses dims it does not support: its operands are bf16
// only, so another dtype is a dtype error; anything else is a shape error.
ssd_status_t chunk_refusal(const ScanArgs &a)
{
    return a.dtype != SSD_DTYPE_BF16 ? SSD_ERR_UNSUPPORTED_DTYPE : SSD_ERR_UNSUPPORTED;
}

// Unique id of the CUDA context current on this thread, or 0 when there is none
// or the driver cannot say.  The driver never reuses an id within a process, so
// the per-device caches below, keyed on it, notice a cudaDeviceReset or a
// re-created primary context and set themselves up again instead of handing out
// a pool, stream or address of a context that no longer exists.
uint64_t current_context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Resolves the path for validated dims.  Returns SSD_PATH_* or -status.
int32_t resolve_path(const ScanArgs &a, uint32_t requested, bool probe_device)
{
    const bool seq_ok = seq_supported(a.headdim, a.dstate);
    const bool decode_ok = decode_supported(a);
    if (requested == SSD_PATH_DECODE)
        return decode_ok ? (int32_t)SSD_PATH_DECODE : -(int32_t)SSD_ERR_UNSUPPORTED;
    if (requested == SSD_PATH_AUTO && decode_ok)
        return SSD_PATH_DECODE;
    const bool chunk_ok = chunk_supported(a) && (!probe_device || device_is_gb300_class());
    if (requested == SSD_PATH_SEQUENTIAL)
        return seq_ok ? (int32_t)SSD_PATH_SEQUENTIAL : -(int32_t)SSD_ERR_UNSUPPORTED;
    if (requested == SSD_PATH_CHUNKED)
        return chunk_ok ? (int32_t)SSD_PATH_CHUNKED : -(int32_t)chunk_refusal(a);
    if (chunk_ok)
        return SSD_PATH_CHUNKED;
    if (seq_ok)
        return SSD_PATH_SEQUENTIAL;
    return -(int32_t)SSD_ERR_UNSUPPORTED;
}

// Library-owned stream-ordered memory pool per device (kept cached so that
// repeated calls do not go back to the driver; set up again when the device's
// context has changed since).
cudaMemPool_t scratch_pool(int dev)
{
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    static uint64_t pool_ctx[64] = {};
    if (dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    const uint64_t ctx = current_context_id();
    if (!pools[dev] || ctx == 0 || ctx != pool_ctx[dev]) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess)
            return nullptr;
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[dev] = p;
        pool_ctx[dev] = current_context_id();   // the context exists now
    }
    return pools[dev];
}

// The host-buffer path pipelines pieces of whole batch rows through three
// library-owned streams per device (copies in, kernels, copies out).
constexpr int kHostPieces = 8;                          // most pieces per call
constexpr int64_t kHostPipelineMinBytes = 32ll << 20;   // smaller calls run as one piece

struct HostStreams {
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
};

HostStreams host_streams(int dev)
{
    static std::mutex mu;
    static HostStreams streams[64];
    static uint64_t streams_ctx[64] = {};
    if (dev < 0 || dev >= 64)
        return HostStreams{};
    std::lock_guard<std::mutex> lk(mu);
    HostStreams &h = streams[dev];
    const uint64_t ctx = current_context_id();
    if (!h.in || ctx == 0 || ctx != streams_ctx[dev]) {
        HostStreams n;
        if (cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&n.comp, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking) != cudaSuccess)
            return HostStreams{};
        h = n;
        streams_ctx[dev] = current_context_id();
    }
    return h;
}

// The paths that need no scratch: the sequential scan and the decode step.
ssd_status_t launch_direct(const ScanArgs &a, int32_t path, cudaStream_t st)
{
    const cudaError_t e = path == SSD_PATH_DECODE ? decode_launch(a, st) : seq_launch(a, st);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t run_device(const ScanArgs &a, uint32_t requested, cudaStream_t st)
{
    const int32_t path = resolve_path(a, requested, true);
    if (path < 0)
        return (ssd_status_t)(-path);
    if (path != SSD_PATH_CHUNKED)
        return launch_direct(a, path, st);
    const size_t ws_bytes = chunk_workspace_bytes(a);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(dev);
    if (!pool)
        return SSD_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, ws_bytes, pool, st) != cudaSuccess)
        return SSD_ERR_CUDA;
    const ssd_status_t s = chunk_launch(a, ws, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && s == SSD_OK)
        return SSD_ERR_CUDA;
    return s;
}

ssd_status_t validate(const void *x, const float *dt_raw, const float *dt_bias, const float *A_log,
                      const void *B, const void *C, const float *D, const float *init_state,
                      const void *y, const float *final_state, const ssd_dims_t *dims, Sizes *sz)
{
    ssd_status_t s = check_dims(dims, sz);
    if (s != SSD_OK)
        return s;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!x || !dt_raw || !dt_bias || !A_log || !B || !C || !D || !y))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state};
    for (const void *p : ptrs)
        if (!aligned16(p))
            return SSD_ERR_MISALIGNED;
    if (work) {
        const void *ins[] = {x, dt_raw, dt_bias, A_log, B, C, D, init_state};
        const int64_t inb[] = {sz->x, sz->dt, sz->par, sz->par, sz->bc, sz->bc, sz->par, sz->state};
        for (int i = 0; i < 8; ++i) {
            if (overlaps(y, sz->x, ins[i], inb[i]))
                return SSD_ERR_ALIASING;
            if (overlaps(final_state, sz->state, ins[i], inb[i]) && !(i == 7 && final_state == init_state))
                return SSD_ERR_ALIASING;
        }
        if (overlaps(final_state, sz->state, y, sz->x))
            return SSD_ERR_ALIASING;
    } else if (init_state && final_state && init_state != final_state &&
               overlaps(final_state, sz->state, init_state, sz->state)) {
        return SSD_ERR_ALIASING;
    }
    return SSD_OK;
}

// ---- allocation-free variant of the chunked path ------------------------
//
// Some callers cannot let a library allocate device memory during a call:
// processes that reserve the whole device up front in an arena of their own
// (a serving stack that sizes weights, caches and activations at start-up)
// leave a library pool nothing to grow into, so a first-call allocation fails
// with out-of-memory; and drivers or virtualised devices without stream-ordered
// memory pools (cudaDevAttrMemoryPoolsSupported == 0) cannot serve
// cudaMallocFromPoolAsync at all.  For them ssd_scan_fwd_noalloc runs the
// chunked kernel with its scratch (abort word, handoff flags, chunk-handoff
// states) in this fixed module-scope array instead of a pool allocation.
//
// Limit: 32 MiB.  The kernel needs 256 B for the abort word, 64 B of flags
// per unit, and, when a batch-row x head-pair chain is split into several
// units, 64 KiB of handoff state per chain: about 20 MiB for batch 8 x 80
// heads at L = 4096, so roughly 500 split chains fit.  Larger needs are
// rejected with SSD_ERR_SCRATCH_LIMIT before anything is enqueued.
//
// Nothing in the array has to start at zero: every flag and the abort word
// are compared against a per-call tag that is never zero and never repeats
// within a process, so values left by an earlier call never match.
//
// The array is one per device and shared by every call: two calls whose
// kernels overlap in time on the same device (different streams, or threads
// without ordering between them) race on it and give wrong results or
// time out.  Calls ordered on one stream are safe.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (the host-side name
// of the array is not a device address).  Looked up with that device current on
// the first call, and again whenever the device's context has changed since (a
// cudaDeviceReset unloads the module, and the array may come back elsewhere);
// cached otherwise.  Null on failure.
void *noalloc_scratch(int dev)
{
    static std::mutex mu;
    static void *addr[64] = {};
    static uint64_t addr_ctx[64] = {};
    if (dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    const uint64_t ctx = current_context_id();
    if (!addr[dev] || ctx == 0 || ctx != addr_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            addr[dev] = nullptr;
            return nullptr;
        }
        addr[dev] = p;
        addr_ctx[dev] = current_context_id();   // the lookup made the context current
    }
    return addr[dev];
}

}  // namespace

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status_t ssd_scan_fwd(const void *x, const float *dt_raw, const float *dt_bias,
                          const float *A_log, const void *B, const void *C, const float *D,
                          const float *init_state, void *y, float *final_state,
                          const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_scan_fwd");
    Sizes sz;
    ssd_status_t s = validate(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims, &sz);
    if (s != SSD_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->batch == 0)
        return SSD_OK;
    if (dims->seqlen == 0) {
        // no steps: the final state is the initial state (zero when none)
        if (!final_state || sz.state == 0)
            return SSD_OK;
        cudaError_t e = init_state ? (init_state == final_state
                                          ? cudaSuccess
                                          : cudaMemcpyAsync(final_state, init_state, (size_t)sz.state,
                                                            cudaMemcpyDeviceToDevice, st))
                                   : cudaMemsetAsync(final_state, 0, (size_t)sz.state, st);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    const ScanArgs a = make_args(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims);
    return run_device(a, dims->flags & SSD_PATH_MASK, st);
}

ssd_status_t ssd_scan_fwd_host(const void *x, const float *dt_raw, const float *dt_bias,
                               const float *A_log, const void *B, const void *C,
                               const float *D, const float *init_state, void *y,
                               float *final_state, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_scan_fwd_host");
    Sizes sz;
    ssd_status_t s = validate(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims, &sz);
    if (s != SSD_OK)
        return s;
    if (dims->batch == 0 || (dims->seqlen == 0 && !final_state))
        return SSD_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->seqlen == 0) {
        if (init_state)
            std::memmove(final_state, init_state, (size_t)sz.state);
        else
            std::memset(final_state, 0, (size_t)sz.state);
        return SSD_OK;
    }
    auto up = [](int64_t v) { return (v + 255) & ~(int64_t)255; };
    const int64_t off_x = 0, off_dt = off_x + up(sz.x), off_bias = off_dt + up(sz.dt),
                  off_alog = off_bias + up(sz.par), off_B = off_alog + up(sz.par),
                  off_C = off_B + up(sz.bc), off_D = off_C + up(sz.bc), off_h0 = off_D + up(sz.par),
                  off_y = off_h0 + (init_state ? up(sz.state) : 0),
                  off_hf = off_y + up(sz.x), total = off_hf + (final_state ? up(sz.state) : 0);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(dev);
    const HostStreams hs = host_streams(dev);
    if (!pool || !hs.in)
        return SSD_ERR_CUDA;
    char *buf = nullptr;
    if (cudaMallocFromPoolAsync((void **)&buf, (size_t)total, pool, st) != cudaSuccess)
        return SSD_ERR_CUDA;

    // Pieces of whole batch rows go through three streams: copies in, kernels,
    // copies out, so the two copy directions and the scan overlap.  All kernels
    // stay on one stream (the persistent chunked kernel never shares the GPU
    // with another of its launches).  Each piece takes the schedule the whole
    // batch would (ranges and pieces give the same bits; a batch that would
    // take the split schedule runs as one piece), so the result is bitwise the
    // one ssd_scan_fwd gives.
    const int64_t Bt = dims->batch;
    const ScanArgs whole = make_args(buf + off_x, (const float *)(buf + off_dt), (const float *)(buf + off_bias),
                                     (const float *)(buf + off_alog), buf + off_B, buf + off_C,
                                     (const float *)(buf + off_D),
                                     init_state ? (const float *)(buf + off_h0) : nullptr, buf + off_y,
                                     final_state ? (float *)(buf + off_hf) : nullptr, dims);
    const uint32_t req = dims->flags & SSD_PATH_MASK;
    const int32_t path = resolve_path(whole, req, true);
    if (path < 0) {
        cudaFreeAsync(buf, st);
        cudaStreamSynchronize(st);
        return (ssd_status_t)(-path);
    }
    int sched = path == SSD_PATH_CHUNKED ? chunk_schedule(whole) : SSD_SCHEDULE_NONE;
    int pieces = (int)std::min<int64_t>(Bt, kHostPieces);
    if (sched == SSD_SCHEDULE_SPLIT || total < kHostPipelineMinBytes)
        pieces = 1;
    const int64_t xr = sz.x / Bt, dtr = sz.dt / Bt, bcr = sz.bc / Bt, str = sz.state / Bt;   // bytes per row

    cudaEvent_t start = nullptr, in_done[kHostPieces] = {}, comp_done[kHostPieces] = {}, end_in = nullptr,
                end_comp = nullptr, end_out = nullptr;
    bool ok = cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&end_in, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&end_comp, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&end_out, cudaEventDisableTiming) == cudaSuccess;
    for (int k = 0; ok && k < pieces; ++k)
        ok = cudaEventCreateWithFlags(&in_done[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&comp_done[k], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventRecord(start, st) == cudaSuccess && cudaStreamWaitEvent(hs.in, start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(hs.comp, start, 0) == cudaSuccess && cudaStreamWaitEvent(hs.out, start, 0) == cudaSuccess;
    auto h2d = [&](int64_t off, const void *src, int64_t n) {
        if (ok && src && n > 0)
            ok = cudaMemcpyAsync(buf + off, src, (size_t)n, cudaMemcpyHostToDevice, hs.in) == cudaSuccess;
    };
    auto d2h = [&](void *dst, int64_t off, int64_t n) {
        if (ok && dst && n > 0)
            ok = cudaMemcpyAsync(dst, buf + off, (size_t)n, cudaMemcpyDeviceToHost, hs.out) == cudaSuccess;
    };
    h2d(off_bias, dt_bias, sz.par);
    h2d(off_alog, A_log, sz.par);
    h2d(off_D, D, sz.par);
    ssd_status_t rs = ok ? SSD_OK : SSD_ERR_CUDA;
    int64_t b0 = 0;
    for (int k = 0; k < pieces && rs == SSD_OK; ++k) {
        const int64_t rows = Bt / pieces + (k < Bt % pieces ? 1 : 0);
        const char *hx = static_cast<const char *>(x), *hB = static_cast<const char *>(B);
        const char *hC = static_cast<const char *>(C);
        h2d(off_x + b0 * xr, hx + b0 * xr, rows * xr);
        h2d(off_dt + b0 * dtr, reinterpret_cast<const char *>(dt_raw) + b0 * dtr, rows * dtr);
        h2d(off_B + b0 * bcr, hB + b0 * bcr, rows * bcr);
        h2d(off_C + b0 * bcr, hC + b0 * bcr, rows * bcr);
        if (init_state)
            h2d(off_h0 + b0 * str, reinterpret_cast<const char *>(init_state) + b0 * str, rows * str);
        ok = ok && cudaEventRecord(in_done[k], hs.in) == cudaSuccess &&
             cudaStreamWaitEvent(hs.comp, in_done[k], 0) == cudaSuccess;
        if (!ok) {
            rs = SSD_ERR_CUDA;
            break;
        }
        ssd_dims_t pd = *dims;
        pd.batch = rows;
        if (pieces > 1 && sched != SSD_SCHEDULE_NONE)
            pd.flags = (pd.flags & ~SSD_SCHEDULE_REQUEST_MASK) | ((uint32_t)sched << SSD_SCHEDULE_SHIFT);
        const ScanArgs a = make_args(buf + off_x + b0 * xr, (const float *)(buf + off_dt + b0 * dtr),
                                     (const float *)(buf + off_bias), (const float *)(buf + off_alog),
                                     buf + off_B + b0 * bcr, buf + off_C + b0 * bcr, (const float *)(buf + off_D),
                                     init_state ? (const float *)(buf + off_h0 + b0 * str) : nullptr,
                                     buf + off_y + b0 * xr,
                                     final_state ? (float *)(buf + off_hf + b0 * str) : nullptr, &pd);
        rs = run_device(a, req, hs.comp);
        if (rs != SSD_OK)
            break;
        ok = cudaEventRecord(comp_done[k], hs.comp) == cudaSuccess &&
             cudaStreamWaitEvent(hs.out, comp_done[k], 0) == cudaSuccess;
        d2h(static_cast<char *>(y) + b0 * xr, off_y + b0 * xr, rows * xr);
        if (final_state)
            d2h(reinterpret_cast<char *>(final_state) + b0 * str, off_hf + b0 * str, rows * str);
        if (!ok)
            rs = SSD_ERR_CUDA;
        b0 += rows;
    }
    // join the worker streams back into the caller's stream before the buffer goes
    const bool joined = end_in && end_comp && end_out && cudaEventRecord(end_in, hs.in) == cudaSuccess &&
                        cudaEventRecord(end_comp, hs.comp) == cudaSuccess &&
                        cudaEventRecord(end_out, hs.out) == cudaSuccess &&
                        cudaStreamWaitEvent(st, end_in, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(st, end_comp, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(st, end_out, 0) == cudaSuccess;
    if (!joined) {   // fall back to waiting on the host
        cudaStreamSynchronize(hs.in);
        cudaStreamSynchronize(hs.comp);
        cudaStreamSynchronize(hs.out);
        if (rs == SSD_OK)
            rs = SSD_ERR_CUDA;
    }
    cudaFreeAsync(buf, st);
    if (cudaStreamSynchronize(st) != cudaSuccess && rs == SSD_OK)
        rs = SSD_ERR_CUDA;
    for (cudaEvent_t e : {start, end_in, end_comp, end_out})
        if (e)
            cudaEventDestroy(e);
    for (int k = 0; k < pieces; ++k) {
        if (in_done[k])
            cudaEventDestroy(in_done[k]);
        if (comp_done[k])
            cudaEventDestroy(comp_done[k]);
    }
    return rs;
}

ssd_status_t ssd_scan_fwd_noalloc(const void *x, const float *dt_raw, const float *dt_bias,
                                  const float *A_log, const void *B, const void *C,
                                  const float *D, const float *init_state, void *y,
                                  float *final_state, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_scan_fwd_noalloc");
    Sizes sz;
    ssd_status_t s = validate(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims, &sz);
    if (s != SSD_OK)
        return s;
    // empty work: ssd_scan_fwd launches nothing and allocates nothing here
    if (dims->batch == 0 || dims->seqlen == 0)
        return ssd_scan_fwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims,
                            stream);
    // the chunked kernel is the only path here: another explicit request is refused
    const uint32_t req = dims->flags & SSD_PATH_MASK;
    if (req != SSD_PATH_AUTO && req != SSD_PATH_CHUNKED)
        return SSD_ERR_UNSUPPORTED;
    ScanArgs a = make_args(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims);
    if (a.sched_req == SSD_SCHEDULE_SPLIT)
        return SSD_ERR_UNSUPPORTED;
    a.scratch_cap = kNoAllocScratchBytes;
    const int32_t path = resolve_path(a, SSD_PATH_CHUNKED, true);
    if (path < 0)
        return (ssd_status_t)(-path);
    if (chunk_workspace_bytes(a) > kNoAllocScratchBytes)
        return SSD_ERR_SCRATCH_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    void *ws = noalloc_scratch(dev);
    if (!ws)
        return SSD_ERR_CUDA;
    return chunk_launch(a, ws, static_cast<cudaStream_t>(stream));
}

ssd_status_t ssd_scan_fwd_workspace_size(const ssd_dims_t *dims, uint64_t *bytes)
{
    if (!bytes)
        return SSD_ERR_NULL_PTR;
    Sizes sz;
    const ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    *bytes = 0;
    if (dims->batch == 0 || dims->seqlen == 0)
        return SSD_OK;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, dims);
    const int32_t path = resolve_path(a, dims->flags & SSD_PATH_MASK, true);
    if (path < 0)
        return (ssd_status_t)(-path);
    if (path == SSD_PATH_CHUNKED)
        *bytes = chunk_workspace_bytes(a);
    return SSD_OK;
}

ssd_status_t ssd_scan_fwd_ws(const void *x, const float *dt_raw, const float *dt_bias,
                             const float *A_log, const void *B, const void *C, const float *D,
                             const float *init_state, void *y, float *final_state, void *workspace,
                             uint64_t workspace_bytes, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_scan_fwd_ws");
    Sizes sz;
    ssd_status_t s = validate(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims, &sz);
    if (s != SSD_OK)
        return s;
    if (!aligned16(workspace))
        return SSD_ERR_MISALIGNED;
    if (workspace && workspace_bytes > 0) {
        const void *args[] = {x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state};
        const int64_t argb[] = {sz.x, sz.dt, sz.par, sz.par, sz.bc, sz.bc, sz.par, sz.state, sz.x, sz.state};
        const int64_t wb = workspace_bytes > (uint64_t)INT64_MAX ? INT64_MAX : (int64_t)workspace_bytes;
        for (int i = 0; i < 10; ++i)
            if (overlaps(workspace, wb, args[i], argb[i]))
                return SSD_ERR_ALIASING;
    }
    // empty work needs no scratch: ssd_scan_fwd allocates nothing here
    if (dims->batch == 0 || dims->seqlen == 0)
        return ssd_scan_fwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims,
                            stream);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ScanArgs a = make_args(x, dt_raw, dt_bias, A_log, B, C, D, init_state, y, final_state, dims);
    const int32_t path = resolve_path(a, dims->flags & SSD_PATH_MASK, true);
    if (path < 0)
        return (ssd_status_t)(-path);
    if (path != SSD_PATH_CHUNKED)
        return launch_direct(a, path, st);
    const size_t need = chunk_workspace_bytes(a);
    if (workspace_bytes < need)
        return SSD_ERR_SCRATCH_LIMIT;
    if (!workspace)
        return SSD_ERR_NULL_PTR;
    return chunk_launch(a, workspace, st);
}

int32_t ssd_select_path(const ssd_dims_t *dims)
{
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return -(int32_t)s;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, dims);
    return resolve_path(a, dims->flags & SSD_PATH_MASK, true);
}

int32_t ssd_launches_per_call(const ssd_dims_t *dims)
{
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return -(int32_t)s;
    if (dims->batch == 0 || dims->seqlen == 0)
        return 0;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, dims);
    const int32_t path = resolve_path(a, dims->flags & SSD_PATH_MASK, true);
    if (path < 0)
        return path;
    return path == SSD_PATH_CHUNKED ? chunk_launches(a) : 1;
}

int32_t ssd_chunk_schedule(const ssd_dims_t *dims)
{
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return -(int32_t)s;
    if (dims->batch == 0 || dims->seqlen == 0)
        return SSD_SCHEDULE_NONE;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, dims);
    const int32_t path = resolve_path(a, dims->flags & SSD_PATH_MASK, true);
    if (path < 0)
        return path;
    return path == SSD_PATH_CHUNKED ? chunk_schedule(a) : SSD_SCHEDULE_NONE;
}

uint64_t ssd_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ssd_status_t ssd_get_device_error(void *stream, uint32_t *code)
{
    if (!code)
        return SSD_ERR_NULL_PTR;
    const ssd_status_t s = chunk_read_device_error(static_cast<cudaStream_t>(stream), code);
    if (s != SSD_OK)
        return s;
    uint32_t bwd = 0, cplx = 0;   // the backward's and the complex chunk form's kernels keep their own words
    ssd_status_t s2 = bwd_tc_read_device_error(&bwd);
    if (s2 == SSD_OK)
        s2 = complex_tc_read_device_error(&cplx);
    if (s2 != SSD_OK)
        return s2;
    if (*code == 0)
        *code = bwd ? bwd : cplx;
    return SSD_OK;
}

const char *ssd_status_string(ssd_status_t status)
{
    switch ((int32_t)status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_DIMS: return "invalid dimensions";
    case SSD_ERR_NULL_PTR: return "required pointer is null";
    case SSD_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SSD_ERR_UNSUPPORTED: return "dtype, shape or path not supported";
    case SSD_ERR_CUDA: return "CUDA call failed";
    case SSD_ERR_TIMEOUT: return "kernel exceeded a bounded wait";
    case SSD_ERR_ALIASING: return "output overlaps an input";
    case SSD_ERR_SCRATCH_LIMIT: return "scratch needed exceeds the buffer the call may use";
    case SSD_ERR_UNSUPPORTED_DTYPE: return "dtype not supported";
    default: return "unknown status";
    }
}

int32_t ssd_abi_version(void) { return SSD_ABI_VERSION; }

ssd_status_t ssd_complex_scan_fwd(const void *x, const float *dt_raw, const float *dt_bias, const float *A_polar,
                                  const void *B, const void *C, const float *D, const float *init_state, void *y,
                                  float *final_state, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_complex_scan_fwd");
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    if ((dims->flags & ~SSD_PATH_MASK) != 0)
        return SSD_ERR_INVALID_DIMS;
    const uint32_t path = dims->flags & SSD_PATH_MASK;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_SEQUENTIAL && path != SSD_PATH_CHUNKED)
        return SSD_ERR_UNSUPPORTED;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!x || !dt_raw || !dt_bias || !A_polar || !B || !C || !D || !y))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {x, dt_raw, dt_bias, A_polar, B, C, D, init_state, y, final_state};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    // outputs overlap no input (the state may be updated in place) and not each other
    const void *ins[] = {x, dt_raw, dt_bias, A_polar, B, C, D, init_state};
    const int64_t inb[] = {sz.x, sz.dt, sz.par, 2 * sz.par, sz.bc, sz.bc, sz.par, sz.state};
    const void *outs[] = {work ? y : nullptr, final_state};
    const int64_t outb[] = {sz.x, sz.state};
    for (int o = 0; o < 2; ++o)
        for (int i = 0; i < 8; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i]) && !(o == 1 && ins[i] == init_state && outs[o] == init_state))
                return SSD_ERR_ALIASING;
    if (overlaps(outs[0], outb[0], outs[1], outb[1]))
        return SSD_ERR_ALIASING;
    ComplexArgs ca;
    ca.x = x;
    ca.B = B;
    ca.C = C;
    ca.dt_raw = dt_raw;
    ca.dt_bias = dt_bias;
    ca.A_polar = A_polar;
    ca.D = D;
    ca.init_state = init_state;
    ca.y = y;
    ca.final_state = final_state;
    ca.batch = dims->batch;
    ca.seqlen = dims->seqlen;
    ca.nheads = dims->nheads;
    ca.headdim = dims->headdim;
    ca.dstate = dims->dstate;
    ca.ngroups = dims->ngroups;
    ca.dtype = dims->dtype;
    // the chunk form on the tensor cores where it applies (auto) or is asked for
    const bool tc = path != SSD_PATH_SEQUENTIAL && complex_tc_supported(ca);
    if (path == SSD_PATH_CHUNKED && !tc)
        return SSD_ERR_UNSUPPORTED;
    if (!tc && !complex_supported(ca))
        return SSD_ERR_UNSUPPORTED;
    if (dims->batch == 0)
        return SSD_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->seqlen == 0) {   // no steps: the state passes through (zero when not given)
        if (!final_state || final_state == init_state)
            return SSD_OK;
        const cudaError_t e = init_state ? cudaMemcpyAsync(final_state, init_state, (size_t)sz.state,
                                                           cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(final_state, 0, (size_t)sz.state, st);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    return (tc ? complex_tc_launch(ca, st) : complex_launch(ca, st)) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_trap_scan_fwd(const void *v, const void *k, const void *q, const float *dt, const float *a,
                               const float *trap, const float *D, const float *h0, const void *k0,
                               const void *v0, void *y, float *h_final, void *k_final, void *v_final,
                               const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_trap_scan_fwd");
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    const uint32_t path = dims->flags & SSD_PATH_MASK;
    if ((dims->flags & ~(SSD_PATH_MASK | SSD_SCHEDULE_REQUEST_MASK)) != 0)
        return SSD_ERR_INVALID_DIMS;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_SEQUENTIAL && path != SSD_PATH_CHUNKED)
        return SSD_ERR_UNSUPPORTED;
    const int64_t es = dims->dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const int64_t kst = dims->batch * dims->nheads * dims->dstate * es;   // k_state bytes
    const int64_t vst = dims->batch * dims->nheads * dims->headdim * es;  // v_state bytes
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!v || !k || !q || !dt || !a || !trap || !D || !y))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {v, k, q, dt, a, trap, D, h0, k0, v0, y, h_final, k_final, v_final};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    // outputs overlap no input (each state may be updated in place) and no other output
    const void *ins[] = {v, k, q, dt, a, trap, D, h0, k0, v0};
    const int64_t inb[] = {sz.x, sz.bc, sz.bc, sz.dt, sz.dt, sz.dt, sz.par, sz.state, kst, vst};
    const void *outs[] = {work ? y : nullptr, h_final, k_final, v_final};
    const int64_t outb[] = {sz.x, sz.state, kst, vst};
    const void *same[] = {nullptr, h0, k0, v0};   // the input each output may replace exactly
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 10; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i]) && !(outs[o] == same[o] && ins[i] == same[o]))
                return SSD_ERR_ALIASING;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlaps(outs[o], outb[o], outs[o2], outb[o2]))
                return SSD_ERR_ALIASING;
    }
    if (dims->batch == 0)
        return SSD_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->seqlen == 0) {
        // no steps: every carried state passes through unchanged (zero when not given)
        const void *src[] = {h0, k0, v0};
        void *dst[] = {h_final, k_final, v_final};
        const int64_t nb[] = {sz.state, kst, vst};
        for (int i = 0; i < 3; ++i) {
            if (!dst[i] || nb[i] == 0 || src[i] == dst[i])
                continue;
            const cudaError_t e = src[i] ? cudaMemcpyAsync(dst[i], src[i], (size_t)nb[i], cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(dst[i], 0, (size_t)nb[i], st);
            if (e != cudaSuccess)
                return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    TrapArgs ta;
    ta.v = v;
    ta.k = k;
    ta.q = q;
    ta.dt = dt;
    ta.a = a;
    ta.trap = trap;
    ta.D = D;
    ta.h0 = h0;
    ta.k0 = k0;
    ta.v0 = v0;
    ta.y = y;
    ta.h_final = h_final;
    ta.k_final = k_final;
    ta.v_final = v_final;
    ta.batch = dims->batch;
    ta.seqlen = dims->seqlen;
    ta.nheads = dims->nheads;
    ta.headdim = dims->headdim;
    ta.dstate = dims->dstate;
    ta.ngroups = dims->ngroups;
    ta.dtype = dims->dtype;
    // the chunked tcgen05 kernel in its trapezoidal mode, or the sequential kernel
    ScanArgs ca = make_args(v, nullptr, nullptr, nullptr, k, q, D, h0, y, h_final, dims);
    ca.trap = true;
    ca.tdt = dt;
    ca.ta = a;
    ca.ttrap = trap;
    ca.k0 = k0;
    ca.v0 = v0;
    const bool chunk_ok = chunk_supported(ca) && device_is_gb300_class();
    const bool seq_ok = trap_supported(ta);
    bool chunked;
    if (path == SSD_PATH_CHUNKED)
        chunked = true;
    else if (path == SSD_PATH_SEQUENTIAL)
        chunked = false;
    else   // one step is a stream of the state: the sequential kernel
        chunked = chunk_ok && (dims->seqlen > 1 || !seq_ok);
    if (chunked ? !chunk_ok : !seq_ok)
        return chunked && dims->dtype != SSD_DTYPE_BF16 ? SSD_ERR_UNSUPPORTED_DTYPE : SSD_ERR_UNSUPPORTED;
    if (!chunked)
        return trap_launch(ta, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(dev);
    if (!pool)
        return SSD_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, chunk_workspace_bytes(ca), pool, st) != cudaSuccess)
        return SSD_ERR_CUDA;
    ssd_status_t rs = chunk_launch(ca, ws, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && rs == SSD_OK)
        rs = SSD_ERR_CUDA;
    if (rs == SSD_OK && trap_carry_launch(ta, st) != cudaSuccess)
        rs = SSD_ERR_CUDA;
    return rs;
}

ssd_status_t ssd_conv1d_silu_fwd(const void *xbc, const float *weight, const float *bias,
                                 const void *conv_state, void *x, void *B, void *C, void *conv_state_out,
                                 int32_t kernel_size, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_conv1d_silu_fwd");
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    if (dims->flags != 0 || kernel_size < 1)
        return SSD_ERR_INVALID_DIMS;
    const int64_t es = dims->dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const int64_t Cc = (int64_t)dims->nheads * dims->headdim + 2 * (int64_t)dims->ngroups * dims->dstate;
    int64_t xbcb, stb;
    if (!mul_ok(dims->batch * dims->seqlen, Cc * es, &xbcb) || !mul_ok(dims->batch * (kernel_size - 1), Cc * es, &stb))
        return SSD_ERR_INVALID_DIMS;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!xbc || !weight || !x || !B || !C))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {xbc, weight, bias, conv_state, x, B, C, conv_state_out};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    const void *ins[] = {xbc, weight, bias, conv_state};
    const int64_t inb[] = {xbcb, Cc * kernel_size * 4, Cc * 4, stb};
    const void *outs[] = {work ? x : nullptr, work ? B : nullptr, work ? C : nullptr, conv_state_out};
    const int64_t outb[] = {sz.x, sz.bc, sz.bc, stb};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 4; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i]))
                return SSD_ERR_ALIASING;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlaps(outs[o], outb[o], outs[o2], outb[o2]))
                return SSD_ERR_ALIASING;
    }
    NeighborArgs na;
    na.xbc = xbc;
    na.w = weight;
    na.bias = bias;
    na.state_in = conv_state;
    na.x = x;
    na.B = B;
    na.C = C;
    na.state_out = conv_state_out;
    na.kernel_size = kernel_size;
    na.batch = dims->batch;
    na.seqlen = dims->seqlen;
    na.nheads = dims->nheads;
    na.headdim = dims->headdim;
    na.dstate = dims->dstate;
    na.ngroups = dims->ngroups;
    na.dtype = dims->dtype;
    if (!conv_supported(na))
        return SSD_ERR_UNSUPPORTED;
    if (dims->batch == 0)
        return SSD_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->seqlen == 0) {   // no steps: the conv state passes through (zero when not given)
        if (!conv_state_out || stb == 0)
            return SSD_OK;
        const cudaError_t e = conv_state ? cudaMemcpyAsync(conv_state_out, conv_state, (size_t)stb,
                                                           cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(conv_state_out, 0, (size_t)stb, st);
        return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    }
    return conv_launch(na, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_conv_scan_fwd(const void *xbc, const float *conv_weight, const float *conv_bias,
                               const void *conv_state, int32_t kernel_size, const float *dt_raw,
                               const float *dt_bias, const float *A_log, const float *D,
                               const float *init_state, void *y, float *final_state, void *conv_state_out,
                               const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_conv_scan_fwd");
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    if ((dims->flags & ~(SSD_PATH_MASK | SSD_SCHEDULE_REQUEST_MASK)) != 0 || kernel_size < 2 || kernel_size > 4)
        return SSD_ERR_INVALID_DIMS;
    const uint32_t path = dims->flags & SSD_PATH_MASK;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_CHUNKED)
        return SSD_ERR_UNSUPPORTED;
    if (dims->dtype != SSD_DTYPE_BF16)
        return SSD_ERR_UNSUPPORTED_DTYPE;
    const int64_t HP = (int64_t)dims->nheads * dims->headdim, GN = (int64_t)dims->ngroups * dims->dstate;
    const int64_t Cc = HP + 2 * GN;
    if (HP % 8 != 0 || GN % 8 != 0)
        return SSD_ERR_UNSUPPORTED;
    int64_t xbcb, stb;
    if (!mul_ok(dims->batch * dims->seqlen, Cc * 2, &xbcb) || !mul_ok(dims->batch * (kernel_size - 1), Cc * 2, &stb))
        return SSD_ERR_INVALID_DIMS;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!xbc || !conv_weight || !dt_raw || !dt_bias || !A_log || !D || !y))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {xbc, conv_weight, conv_bias, conv_state, dt_raw, dt_bias, A_log, D,
                          init_state, y, final_state, conv_state_out};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    // outputs overlap no input (the scan state may be updated in place) and not each other
    const void *ins[] = {xbc, conv_weight, conv_bias, conv_state, dt_raw, dt_bias, A_log, D, init_state};
    const int64_t inb[] = {xbcb, Cc * kernel_size * 4, Cc * 4, stb, sz.dt, sz.par, sz.par, sz.par, sz.state};
    const void *outs[] = {work ? y : nullptr, final_state, conv_state_out};
    const int64_t outb[] = {sz.x, sz.state, stb};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 9; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i]) && !(o == 1 && i == 8 && outs[o] == ins[i]))
                return SSD_ERR_ALIASING;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(outs[o], outb[o], outs[o2], outb[o2]))
                return SSD_ERR_ALIASING;
    }
    ScanArgs a = make_args(nullptr, dt_raw, dt_bias, A_log, nullptr, nullptr, D, init_state, y, final_state, dims);
    a.conv = true;
    a.xbc = xbc;
    a.conv_w = conv_weight;
    a.conv_b = conv_bias;
    a.conv_state = conv_state;
    a.conv_k = kernel_size;
    a.conv_cc = (int)Cc;
    if (!chunk_supported(a))
        return SSD_ERR_UNSUPPORTED;
    if (dims->batch == 0)
        return SSD_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->seqlen == 0) {   // no steps: both states pass through (zero when not given)
        const void *src[] = {init_state, conv_state};
        void *dst[] = {final_state, conv_state_out};
        const int64_t nb[] = {sz.state, stb};
        for (int i = 0; i < 2; ++i) {
            if (!dst[i] || nb[i] == 0 || src[i] == dst[i])
                continue;
            const cudaError_t e = src[i] ? cudaMemcpyAsync(dst[i], src[i], (size_t)nb[i], cudaMemcpyDeviceToDevice, st)
                                         : cudaMemsetAsync(dst[i], 0, (size_t)nb[i], st);
            if (e != cudaSuccess)
                return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    if (!device_is_gb300_class())
        return SSD_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(dev);
    if (!pool)
        return SSD_ERR_CUDA;
    // scratch: the convolved B and C, then the chunked path's own
    const size_t bc_bytes = ((size_t)sz.bc + 255) & ~(size_t)255;
    const size_t ws_bytes = chunk_workspace_bytes(a);
    char *buf = nullptr;
    if (cudaMallocFromPoolAsync((void **)&buf, 2 * bc_bytes + ws_bytes, pool, st) != cudaSuccess)
        return SSD_ERR_CUDA;
    NeighborArgs na;
    na.xbc = xbc;
    na.w = conv_weight;
    na.bias = conv_bias;
    na.state_in = conv_state;
    na.B = buf;
    na.C = buf + bc_bytes;
    na.state_out = conv_state_out;
    na.kernel_size = kernel_size;
    na.batch = dims->batch;
    na.seqlen = dims->seqlen;
    na.nheads = dims->nheads;
    na.headdim = dims->headdim;
    na.dstate = dims->dstate;
    na.ngroups = dims->ngroups;
    na.dtype = dims->dtype;
    ssd_status_t rs = conv_bc_launch(na, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    if (rs == SSD_OK) {
        a.B = na.B;
        a.C = na.C;
        rs = chunk_launch(a, buf + 2 * bc_bytes, st);
    }
    if (cudaFreeAsync(buf, st) != cudaSuccess && rs == SSD_OK)
        rs = SSD_ERR_CUDA;
    return rs;
}

ssd_status_t ssd_gated_rmsnorm_fwd(const void *y, const void *z, const float *weight, float eps, void *out,
                                   const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_gated_rmsnorm_fwd");
    Sizes sz;
    ssd_status_t s = check_dims(dims, &sz);
    if (s != SSD_OK)
        return s;
    if (dims->flags != 0 || !(eps >= 0.f))
        return SSD_ERR_INVALID_DIMS;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!y || !z || !weight || !out))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {y, z, weight, out};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    if (work && (overlaps(out, sz.x, y, sz.x) || overlaps(out, sz.x, z, sz.x) ||
                 overlaps(out, sz.x, weight, (int64_t)dims->nheads * dims->headdim * 4)))
        return SSD_ERR_ALIASING;
    NeighborArgs na;
    na.y = y;
    na.z = z;
    na.w = weight;
    na.out = out;
    na.eps = eps;
    na.batch = dims->batch;
    na.seqlen = dims->seqlen;
    na.nheads = dims->nheads;
    na.headdim = dims->headdim;
    na.dtype = dims->dtype;
    if (!gnorm_supported(na))
        return SSD_ERR_UNSUPPORTED;
    if (!work)
        return SSD_OK;
    return gnorm_launch(na, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_scan_bwd(const void *x, const float *dt_raw, const float *dt_bias, const float *A_log,
                          const void *B, const void *C, const float *D, const float *init_state, const void *dy,
                          const float *d_final, float *dx, float *ddt_raw, float *ddt_bias, float *dA_log,
                          float *dB, float *dC, float *dD, float *d_init, const ssd_dims_t *dims, void *stream)
{
    SSD_NVTX_RANGE("ssd_scan_bwd");
    Sizes sz;
    if (!dims)
        return SSD_ERR_NULL_PTR;
    ssd_dims_t dchk = *dims;   // (the backward's own flags are checked here, the rest by check_dims)
    dchk.flags &= ~(SSD_BWD_FP32_FORM | SSD_BWD_SPLIT_STATES);
    ssd_status_t s = check_dims(&dchk, &sz);
    if (s != SSD_OK)
        return s;
    if ((dims->flags & ~(SSD_PATH_MASK | SSD_BWD_FP32_FORM | SSD_BWD_SPLIT_STATES)) != 0)
        return SSD_ERR_INVALID_DIMS;
    const uint32_t path = dims->flags & SSD_PATH_MASK;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_SEQUENTIAL && path != SSD_PATH_CHUNKED)
        return SSD_ERR_UNSUPPORTED;
    const bool work = dims->batch > 0 && dims->seqlen > 0;
    if (work && (!x || !dt_raw || !dt_bias || !A_log || !B || !C || !D || !dy || !dx || !ddt_raw || !ddt_bias ||
                 !dA_log || !dB || !dC || !dD))
        return SSD_ERR_NULL_PTR;
    const void *ptrs[] = {x, dt_raw, dt_bias, A_log, B, C, D, init_state, dy, d_final,
                          dx, ddt_raw, ddt_bias, dA_log, dB, dC, dD, d_init};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr))
            return SSD_ERR_MISALIGNED;
    // fp32 gradients: dx [B,L,H,P], ddt_raw [B,L,H], dB/dC [B,L,G,N], per-head [H], d_init [B,H,P,N]
    const int64_t es = dims->dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const int64_t x32 = sz.x / es * 4, bc32 = sz.bc / es * 4;
    const void *ins[] = {x, dt_raw, dt_bias, A_log, B, C, D, init_state, dy, d_final};
    const int64_t inb[] = {sz.x, sz.dt, sz.par, sz.par, sz.bc, sz.bc, sz.par, sz.state, sz.x, sz.state};
    const void *outs[] = {dx, ddt_raw, ddt_bias, dA_log, dB, dC, dD, d_init};
    const int64_t outb[] = {x32, sz.dt, sz.par, sz.par, bc32, bc32, sz.par, sz.state};
    if (work)
        for (int o = 0; o < 8; ++o) {
            for (int i = 0; i < 10; ++i)
                if (overlaps(outs[o], outb[o], ins[i], inb[i]))
                    return SSD_ERR_ALIASING;
            for (int o2 = o + 1; o2 < 8; ++o2)
                if (overlaps(outs[o], outb[o], outs[o2], outb[o2]))
                    return SSD_ERR_ALIASING;
        }
    BwdArgs ba;
    ba.x = x;
    ba.B = B;
    ba.C = C;
    ba.dy = dy;
    ba.dt_raw = dt_raw;
    ba.dt_bias = dt_bias;
    ba.A_log = A_log;
    ba.D = D;
    ba.init_state = init_state;
    ba.d_final = d_final;
    ba.dx = dx;
    ba.ddt_raw = ddt_raw;
    ba.ddt_bias = ddt_bias;
    ba.dA_log = dA_log;
    ba.dB = dB;
    ba.dC = dC;
    ba.dD = dD;
    ba.d_init = d_init;
    ba.batch = dims->batch;
    ba.seqlen = dims->seqlen;
    ba.nheads = dims->nheads;
    ba.headdim = dims->headdim;
    ba.dstate = dims->dstate;
    ba.ngroups = dims->ngroups;
    ba.dtype = dims->dtype;
    ba.path = path;
    ba.fp32_form = (dims->flags & SSD_BWD_FP32_FORM) != 0;
    ba.split_states = (dims->flags & SSD_BWD_SPLIT_STATES) != 0;
    if (path == SSD_PATH_AUTO)
        ba.path = bwd_chunk_supported(ba) ? SSD_PATH_CHUNKED : SSD_PATH_SEQUENTIAL;
    if (!bwd_supported(ba))
        return SSD_ERR_UNSUPPORTED;
    if (!work)
        return SSD_OK;   // (empty work: nothing is written)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(dev);
    if (!pool)
        return SSD_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bwd_workspace_bytes(ba), pool, st) != cudaSuccess)
        return SSD_ERR_CUDA;
    ssd_status_t rs = bwd_launch(ba, ws, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
    if (cudaFreeAsync(ws, st) != cudaSuccess && rs == SSD_OK)
        rs = SSD_ERR_CUDA;
    return rs;
}

}  // extern "C"

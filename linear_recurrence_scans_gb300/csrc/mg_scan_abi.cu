// The C entry points of mg_scan.h: argument validation (all of it before any
// launch), workspace bookkeeping and dispatch to the launchers.
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "common.cuh"

namespace mg {

static thread_local char g_detail[512];

mg_status fail(mg_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return st;
}

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 40;

struct Buf {
    const void *p;
    size_t bytes;
    const char *name;
    bool output;
    bool optional = false;   // NULL allowed (the buffer is then not used)
};

// NULL, alignment and overlap checks.  Outputs may overlap nothing.
mg_status check_bufs(const char *fn, std::initializer_list<Buf> bufs)
{
    for (const Buf &b : bufs) {
        if (b.p == nullptr && b.optional) continue;
        if (b.p == nullptr) return fail(MG_ERR_INVALID_ARG, "%s: %s is NULL", fn, b.name);
        if (reinterpret_cast<uintptr_t>(b.p) % 16 != 0)
            return fail(MG_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, b.name);
    }
    for (const Buf &o : bufs) {
        if (!o.output || o.p == nullptr) continue;
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(o.p), o1 = o0 + o.bytes;
        for (const Buf &x : bufs) {
            if (&x == &o || x.p == nullptr) continue;
            const uintptr_t x0 = reinterpret_cast<uintptr_t>(x.p), x1 = x0 + x.bytes;
            if (o0 < x1 && x0 < o1)
                return fail(MG_ERR_INVALID_ARG, "%s: output %s overlaps %s", fn, o.name, x.name);
        }
    }
    return MG_OK;
}

mg_status check_dims(const char *fn, std::initializer_list<int64_t> dims)
{
    int64_t prod = 1;
    for (int64_t d : dims) {
        if (d < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative size %lld", fn, (long long)d);
        if (d > kMaxDim) return fail(MG_ERR_UNSUPPORTED, "%s: size %lld too large", fn, (long long)d);
        if (d > 0 && prod > (int64_t(1) << 58) / d)
            return fail(MG_ERR_UNSUPPORTED, "%s: tensor too large", fn);
        prod *= (d > 0 ? d : 1);
    }
    return MG_OK;
}

// The channel-wise kernels index channels with 32-bit integers (a tile's
// first channel plus the lane's offset): D must stay clear of 2^31.
constexpr int64_t kMaxChannels = (int64_t(1) << 31) - (int64_t(1) << 16);

mg_status check_channels(const char *fn, int64_t D)
{
    if (D > kMaxChannels)
        return fail(MG_ERR_UNSUPPORTED, "%s: D = %lld channels exceeds %lld", fn, (long long)D,
                    (long long)kMaxChannels);
    return MG_OK;
}

mg_status check_ws(const char *fn, const void *ws, size_t ws_bytes, size_t need)
{
    if (ws == nullptr) return fail(MG_ERR_INVALID_ARG, "%s: workspace is NULL", fn);
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return fail(MG_ERR_INVALID_ARG, "%s: workspace is not 256-byte aligned", fn);
    if (ws_bytes < need)
        return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
    return MG_OK;
}

bool valid_kv(int x) { return x == 1 || x == 2 || x == 4 || x == 8 || x == 16; }

// Default launch options (bounded waits of 2 s, no stalled tile).
LaunchOpts default_opts() { return LaunchOpts{}; }

// ------------------------------------------------ static scratch (no-alloc)
// mg_linear_scan_fwd_noalloc keeps its look-back workspace in this array
// instead of a caller buffer.  Every device that loads the library holds it
// (kNoAllocScratchBytes) until the process exits.  Host code must not use the
// symbol as an address: the device address is obtained once per device with
// cudaGetSymbolAddress and cached below.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set-up on the
// first call per device, with that device current).
mg_status noalloc_scratch(const char *fn, void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MG_ERR_LAUNCH, "%s: cudaGetDevice: %s", fn, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MG_ERR_UNSUPPORTED, "%s: device ordinal %d beyond %d", fn, dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(MG_ERR_LAUNCH, "%s: cudaGetSymbolAddress of the static scratch: %s", fn,
                        cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MG_OK;
}

// Read and clear the error record of the workspace `ws` (synchronises
// `stream`).  The record is Control::error, error_tile and error_epoch (16
// contiguous bytes).
mg_status read_status(const char *fn, void *ws, cudaStream_t stream)
{
    static_assert(offsetof(Control, error_tile) == offsetof(Control, error) + 4 &&
                      offsetof(Control, error_epoch) == offsetof(Control, error) + 8,
                  "the error record is contiguous");
    unsigned int words[2] = {0, 0};  // Control::error, Control::error_tile
    Control *ctl = static_cast<Control *>(ws);
    cudaError_t e = cudaMemcpyAsync(words, &ctl->error, sizeof(words), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    if (words[0] == 0) return MG_OK;
    e = cudaMemsetAsync(&ctl->error, 0, 16, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    if (words[0] & kErrBadSeqlens)
        return fail(MG_ERR_INVALID_ARG,
                    "cu_seqlens was not non-decreasing from 0 to the packed length; the outputs "
                    "of that launch are unspecified");
    if (words[0] & kErrBadTicket)
        return fail(MG_ERR_INVALID_ARG,
                    "the workspace was not zero-filled before its first use (or is shared by "
                    "overlapping calls); the outputs of that launch are unspecified");
    return fail(MG_ERR_TIMEOUT,
                "a chunk look-back wait gave up (first tile %u); the outputs of that launch are "
                "unspecified", words[1] ? words[1] - 1 : 0u);
}

#define MG_TRY(expr)                      \
    do {                                  \
        const mg_status st__ = (expr);    \
        if (st__ != MG_OK) return st__;   \
    } while (0)

}  // namespace
}  // namespace mg

using namespace mg;

extern "C" {

int mg_abi_version(void) { return MG_SCAN_ABI_VERSION; }

const char *mg_strerror(mg_status status)
{
    switch (status) {
    case MG_OK: return "ok";
    case MG_ERR_INVALID_ARG: return "invalid argument";
    case MG_ERR_UNSUPPORTED: return "unsupported by the kernels";
    case MG_ERR_LAUNCH: return "kernel launch failed";
    case MG_ERR_TIMEOUT: return "a look-back wait timed out on the device";
    }
    return "unknown status";
}

const char *mg_last_error_detail(void) { return g_detail; }

size_t mg_linear_scan_workspace_size(int64_t B, int64_t T, int64_t D)
{
    if (B < 0 || T < 0 || D < 0) return 0;
    if (B == 0 || T == 0 || D == 0) return kControlBytes;
    return linear_ws_bytes(B, T, D);
}

size_t mg_log_scan_workspace_size(int64_t B, int64_t T, int64_t D)
{
    if (B < 0 || T < 0 || D < 0) return 0;
    if (B == 0 || T == 0 || D == 0) return kControlBytes;
    return log_ws_bytes(B, T, D);
}

size_t mg_affine_scan_workspace_size(int64_t B, int64_t T, int64_t n, int k, int v)
{
    if (B < 0 || T < 0 || n < 0 || !valid_kv(k) || !valid_kv(v)) return 0;
    if (B == 0 || T == 0 || n == 0) return kControlBytes;
    return affine_ws_bytes(B, T, n, k, v);
}

mg_status mg_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream)
{
    g_detail[0] = 0;
    if (ws == nullptr) return fail(MG_ERR_INVALID_ARG, "mg_workspace_init: workspace is NULL");
    const cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "mg_workspace_init: %s", cudaGetErrorString(e));
    return MG_OK;
}

mg_status mg_workspace_status(void *ws, cudaStream_t stream)
{
    g_detail[0] = 0;
    if (ws == nullptr) return fail(MG_ERR_INVALID_ARG, "mg_workspace_status: workspace is NULL");
    return read_status("mg_workspace_status", ws, stream);
}


mg_status mg_linear_scan_fwd(const void *a, const void *b, mg_dtype in_dt, float *A, float *Bc,
                             int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes,
                             cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_fwd";
    g_detail[0] = 0;
    if (in_dt != MG_F32 && in_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(in_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = in_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {b, n * isz, "b", false},
                           {A, n * 4, "A", true},
                           {Bc, n * 4, "Bc", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_linear_fwd(a, b, in_dt, A, Bc, B, T, D, ws, ws_bytes, stream, default_opts());
}

mg_status mg_linear_scan_bwd(const void *a, mg_dtype a_dt, const float *A, const float *Bc,
                             const float *gA, const float *gBc, float *da, float *db, int64_t B,
                             int64_t T, int64_t D, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_bwd";
    g_detail[0] = 0;
    if (a_dt != MG_F32 && a_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(a_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = a_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {A, n * 4, "A", false},
                           {Bc, n * 4, "Bc", false},
                           {gA, n * 4, "gA", false},
                           {gBc, n * 4, "gBc", false},
                           {da, n * 4, "da", true},
                           {db, n * 4, "db", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_linear_bwd(a, a_dt, A, Bc, gA, gBc, da, db, B, T, D, ws, ws_bytes, stream,
                             default_opts());
}

mg_status mg_linear_scan_bwd_bf16_grads(const void *a, mg_dtype a_dt, const float *A,
                                        const float *Bc, const float *gA, const float *gBc,
                                        void *da, void *db, int64_t B, int64_t T, int64_t D,
                                        void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_bwd_bf16_grads";
    g_detail[0] = 0;
    if (a_dt != MG_F32 && a_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(a_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = a_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {A, n * 4, "A", false},
                           {Bc, n * 4, "Bc", false},
                           {gA, n * 4, "gA", false},
                           {gBc, n * 4, "gBc", false},
                           {da, n * 2, "da", true},
                           {db, n * 2, "db", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_linear_bwd_bf16_grads(a, a_dt, A, Bc, gA, gBc, static_cast<bf16_t *>(da),
                                        static_cast<bf16_t *>(db), B, T, D, ws, ws_bytes, stream,
                                        default_opts());
}

mg_status mg_linear_scan_h0_fwd(const void *a, const void *b, mg_dtype in_dt, const float *h0,
                                float *A, float *H, int64_t B, int64_t T, int64_t D, void *ws,
                                size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_h0_fwd";
    g_detail[0] = 0;
    if (in_dt != MG_F32 && in_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(in_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = in_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {b, n * isz, "b", false},
                           {h0, size_t(B) * D * 4, "h0", false},
                           {A, n * 4, "A", true},
                           {H, n * 4, "H", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_linear_h0_fwd(a, b, in_dt, h0, A, H, B, T, D, ws, ws_bytes, stream, default_opts());
}

mg_status mg_linear_scan_h0_bwd(const void *a, mg_dtype a_dt, const float *h0, const float *A,
                                const float *H, const float *gA, const float *gH, float *da,
                                float *db, float *dh0, int64_t B, int64_t T, int64_t D, void *ws,
                                size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_h0_bwd";
    g_detail[0] = 0;
    if (a_dt != MG_F32 && a_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(a_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = a_dt == MG_F32 ? 4 : 2, nh = size_t(B) * D;
    if (T == 0) {  // L does not depend on h0: its gradient is zero
        MG_TRY(check_bufs(fn, {{dh0, nh * 4, "dh0", true}}));
        const cudaError_t e = cudaMemsetAsync(dh0, 0, nh * 4, stream);
        return e == cudaSuccess ? MG_OK : fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    }
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {h0, nh * 4, "h0", false},
                           {A, n * 4, "A", false},
                           {H, n * 4, "H", false},
                           {gA, n * 4, "gA", false},
                           {gH, n * 4, "gH", false},
                           {da, n * 4, "da", true},
                           {db, n * 4, "db", true},
                           {dh0, nh * 4, "dh0", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_linear_h0_bwd(a, a_dt, h0, A, H, gA, gH, da, db, dh0, B, T, D, ws, ws_bytes,
                                stream, default_opts());
}

size_t mg_linear_scan_varlen_workspace_size(int64_t Ttot, int64_t D)
{
    if (Ttot < 0 || D < 0) return 0;
    if (Ttot == 0 || D == 0) return kControlBytes;
    return varlen_ws_bytes(Ttot, D);
}

// cu_seqlens: nseq + 1 int64 offsets, 8-byte aligned; nseq >= 1 when Ttot > 0.
static mg_status check_varlen(const char *fn, const int64_t *cu, int64_t nseq, int64_t Ttot)
{
    if (nseq < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative nseq", fn);
    if (nseq > (int64_t(1) << 31) - 2) return fail(MG_ERR_UNSUPPORTED, "%s: nseq too large", fn);
    if (Ttot > 0 && nseq == 0)
        return fail(MG_ERR_INVALID_ARG, "%s: %lld packed rows but no sequences", fn, (long long)Ttot);
    if (cu == nullptr) return fail(MG_ERR_INVALID_ARG, "%s: cu_seqlens is NULL", fn);
    if (reinterpret_cast<uintptr_t>(cu) % 8 != 0)
        return fail(MG_ERR_INVALID_ARG, "%s: cu_seqlens is not 8-byte aligned", fn);
    return MG_OK;
}

mg_status mg_linear_scan_varlen_fwd(const void *a, const void *b, mg_dtype in_dt,
                                    const int64_t *cu_seqlens, int64_t nseq, const float *h0,
                                    float *A, float *H, int64_t Ttot, int64_t D, void *ws,
                                    size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_varlen_fwd";
    g_detail[0] = 0;
    if (in_dt != MG_F32 && in_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(in_dt));
    if (nseq < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative nseq", fn);
    MG_TRY(check_dims(fn, {Ttot, D}));
    MG_TRY(check_channels(fn, D));
    if (Ttot == 0 || D == 0) return MG_OK;
    MG_TRY(check_varlen(fn, cu_seqlens, nseq, Ttot));
    const size_t n = size_t(Ttot) * D, isz = in_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, varlen_ws_bytes(Ttot, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {b, n * isz, "b", false},
                           {h0, size_t(nseq) * D * 4, "h0", false, true},
                           {A, n * 4, "A", true},
                           {H, n * 4, "H", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_varlen_fwd(a, b, in_dt, cu_seqlens, nseq, h0, A, H, Ttot, D, ws, ws_bytes,
                             stream, default_opts());
}

mg_status mg_linear_scan_varlen_bwd(const void *a, mg_dtype a_dt, const int64_t *cu_seqlens,
                                    int64_t nseq, const float *h0, const float *A, const float *H,
                                    const float *gA, const float *gH, float *da, float *db,
                                    float *dh0, int64_t Ttot, int64_t D, void *ws,
                                    size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_varlen_bwd";
    g_detail[0] = 0;
    if (a_dt != MG_F32 && a_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(a_dt));
    if (nseq < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative nseq", fn);
    MG_TRY(check_dims(fn, {Ttot, D}));
    MG_TRY(check_channels(fn, D));
    if ((h0 == nullptr) != (dh0 == nullptr))
        return fail(MG_ERR_INVALID_ARG, "%s: h0 and dh0 must be given together (or both NULL)", fn);
    if (D == 0) return MG_OK;
    const size_t nh = size_t(nseq) * D;
    if (dh0 != nullptr && nh > 0) {   // empty sequences keep dh0 = 0
        MG_TRY(check_bufs(fn, {{dh0, nh * 4, "dh0", true}}));
        const cudaError_t e = cudaMemsetAsync(dh0, 0, nh * 4, stream);
        if (e != cudaSuccess) return fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    }
    if (Ttot == 0) return MG_OK;
    MG_TRY(check_varlen(fn, cu_seqlens, nseq, Ttot));
    const size_t n = size_t(Ttot) * D, isz = a_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, varlen_ws_bytes(Ttot, D)));
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {h0, nh * 4, "h0", false, true},
                           {A, n * 4, "A", false},
                           {H, n * 4, "H", false},
                           {gA, n * 4, "gA", false},
                           {gH, n * 4, "gH", false},
                           {da, n * 4, "da", true},
                           {db, n * 4, "db", true},
                           {dh0, nh * 4, "dh0", true, true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_varlen_bwd(a, a_dt, cu_seqlens, nseq, h0, A, H, gA, gH, da, db, dh0, Ttot, D, ws,
                             ws_bytes, stream, default_opts());
}

// perm, sgn, p2p: host (R, k) arrays; every perm[r] a permutation of
// 0..k-1 and p2p[r] its inverse.  Fills the per-lane tables of the kernels.
static mg_status angle_tables(const char *fn, const int32_t *perm, const float *sgn,
                              const int32_t *p2p, int R, int k, AngleTables &tb)
{
    if (k != 2 && k != 4 && k != 8 && k != 16 && k != 32)
        return fail(MG_ERR_UNSUPPORTED, "%s: k = %d outside {2, 4, 8, 16, 32}", fn, k);
    if (R < 1 || R > kAngleMaxR)
        return fail(MG_ERR_UNSUPPORTED, "%s: R = %d outside [1, %d]", fn, R, kAngleMaxR);
    if (perm == nullptr || sgn == nullptr || p2p == nullptr)
        return fail(MG_ERR_INVALID_ARG, "%s: perm, sgn and p2p are required (host arrays)", fn);
    memset(&tb, 0, sizeof(tb));
    tb.R = R;
    for (int r = 0; r < R; ++r) {
        bool seen[kAngleMaxK] = {};
        for (int pos = 0; pos < k; ++pos) {
            const int j = perm[r * k + pos];
            if (j < 0 || j >= k || seen[j])
                return fail(MG_ERR_INVALID_ARG, "%s: perm[%d] is not a permutation of 0..%d", fn, r, k - 1);
            seen[j] = true;
            if (p2p[r * k + j] != pos)
                return fail(MG_ERR_INVALID_ARG, "%s: p2p[%d] is not the inverse of perm[%d]", fn, r, r);
        }
        for (int j = 0; j < k; ++j) {
            const int pos = p2p[r * k + j];
            tb.pair[r][j] = static_cast<signed char>(pos >> 1);
            tb.role[r][j] = static_cast<signed char>(pos & 1);
            tb.partner[r][j] = static_cast<signed char>(perm[r * k + (pos ^ 1)]);
            tb.sgn[r][j] = sgn[r * k + j];
        }
    }
    return MG_OK;
}

mg_status mg_angle_scan_fwd(const float *theta, const float *scale, const float *gamma,
                            const float *b, const float *h0, const int32_t *perm, const float *sgn,
                            const int32_t *p2p, int has_scale, int has_decay, float *h, int64_t B,
                            int64_t T, int64_t n, int R, int k, cudaStream_t stream)
{
    const char *fn = "mg_angle_scan_fwd";
    g_detail[0] = 0;
    AngleTables tb;
    MG_TRY(angle_tables(fn, perm, sgn, p2p, R, k, tb));
    MG_TRY(check_dims(fn, {B, T, n, k}));
    if (B * n > (int64_t(1) << 40) / k) return fail(MG_ERR_UNSUPPORTED, "%s: too many sequences", fn);
    if (T >= (int64_t(1) << 31) || n * int64_t(R) * k >= (int64_t(1) << 31))
        return fail(MG_ERR_UNSUPPORTED, "%s: T and n*R*k must stay below 2^31", fn);
    if (B == 0 || T == 0 || n == 0) return MG_OK;
    const size_t st = size_t(B) * T * n;
    MG_TRY(check_bufs(fn, {{theta, st * R * (k / 2) * 4, "theta", false},
                           {scale, st * 4, "scale", false, !has_scale},
                           {gamma, st * 4, "gamma", false, !has_decay},
                           {b, st * k * 4, "b", false},
                           {h0, size_t(B) * n * k * 4, "h0", false},
                           {h, st * k * 4, "h", true}}));
    return launch_angle(false, theta, scale, gamma, b, h0, nullptr, nullptr, h, nullptr, nullptr,
                        nullptr, nullptr, nullptr, B, T, n, k, has_scale != 0, has_decay != 0, tb,
                        stream);
}

mg_status mg_angle_scan_bwd(const float *theta, const float *scale, const float *gamma,
                            const float *h0, const float *out, const float *grad_out,
                            const int32_t *perm, const float *sgn, const int32_t *p2p,
                            int has_scale, int has_decay, float *dtheta, float *dscale,
                            float *dgamma, float *db, float *dh0, int64_t B, int64_t T, int64_t n,
                            int R, int k, cudaStream_t stream)
{
    const char *fn = "mg_angle_scan_bwd";
    g_detail[0] = 0;
    AngleTables tb;
    MG_TRY(angle_tables(fn, perm, sgn, p2p, R, k, tb));
    MG_TRY(check_dims(fn, {B, T, n, k}));
    if (B * n > (int64_t(1) << 40) / k) return fail(MG_ERR_UNSUPPORTED, "%s: too many sequences", fn);
    if (T >= (int64_t(1) << 31) || n * int64_t(R) * k >= (int64_t(1) << 31))
        return fail(MG_ERR_UNSUPPORTED, "%s: T and n*R*k must stay below 2^31", fn);
    if (B == 0 || n == 0) return MG_OK;
    const size_t nh = size_t(B) * n * k * 4;
    if (T == 0) {   // L does not depend on h0: its gradient is zero
        MG_TRY(check_bufs(fn, {{dh0, nh, "dh0", true}}));
        const cudaError_t e = cudaMemsetAsync(dh0, 0, nh, stream);
        return e == cudaSuccess ? MG_OK : fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    }
    const size_t st = size_t(B) * T * n;
    MG_TRY(check_bufs(fn, {{theta, st * R * (k / 2) * 4, "theta", false},
                           {scale, st * 4, "scale", false, !has_scale},
                           {gamma, st * 4, "gamma", false, !has_decay},
                           {h0, nh, "h0", false},
                           {out, st * k * 4, "out", false},
                           {grad_out, st * k * 4, "grad_out", false},
                           {dtheta, st * R * (k / 2) * 4, "dtheta", true},
                           {dscale, st * 4, "dscale", true},
                           {dgamma, st * 4, "dgamma", true},
                           {db, st * k * 4, "db", true},
                           {dh0, nh, "dh0", true}}));
    return launch_angle(true, theta, scale, gamma, nullptr, h0, out, grad_out, nullptr, dtheta,
                        dscale, dgamma, db, dh0, B, T, n, k, has_scale != 0, has_decay != 0, tb,
                        stream);
}

size_t mg_mingru_scan_workspace_size(int64_t B, int64_t T, int64_t D)
{
    if (B < 0 || T < 0 || D < 0) return 0;
    if (B == 0 || T == 0 || D == 0) return kControlBytes;
    return mingru_ws_bytes(B, T, D);
}

mg_status mg_mingru_scan_fwd(const void *x1, const void *x2, mg_dtype x_dt, float *A, float *Bc,
                             int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes,
                             cudaStream_t stream)
{
    const char *fn = "mg_mingru_scan_fwd";
    g_detail[0] = 0;
    if (x_dt != MG_F32 && x_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(x_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, isz = x_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, mingru_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{x1, n * isz, "x1", false},
                           {x2, n * isz, "x2", false},
                           {A, n * 4, "A", true, true},
                           {Bc, n * 4, "Bc", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_mingru_fwd(x1, x2, x_dt, A, Bc, B, T, D, ws, ws_bytes, stream, default_opts());
}

mg_status mg_mingru_scan_bwd(const void *x1, const void *x2, mg_dtype x_dt, const float *A,
                             const float *Bc, const float *gA, const float *gBc, void *dx1,
                             void *dx2, mg_dtype grad_dt, int64_t B, int64_t T, int64_t D,
                             void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_mingru_scan_bwd";
    g_detail[0] = 0;
    if (x_dt != MG_F32 && x_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(x_dt));
    if (grad_dt != MG_F32 && grad_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: gradient dtype %d not supported", fn, int(grad_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    if ((gA == nullptr) != (A == nullptr))
        return fail(MG_ERR_INVALID_ARG, "%s: A and gA must be given together (or both NULL)", fn);
    const size_t n = size_t(B) * T * D, isz = x_dt == MG_F32 ? 4 : 2;
    const size_t gsz = grad_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_ws(fn, ws, ws_bytes, mingru_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{x1, n * isz, "x1", false},
                           {x2, n * isz, "x2", false},
                           {A, n * 4, "A", false, true},
                           {Bc, n * 4, "Bc", false},
                           {gA, n * 4, "gA", false, true},
                           {gBc, n * 4, "gBc", false},
                           {dx1, n * gsz, "dx1", true},
                           {dx2, n * gsz, "dx2", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_mingru_bwd(x1, x2, x_dt, A, Bc, gA, gBc, dx1, dx2, grad_dt, B, T, D, ws,
                             ws_bytes, stream, default_opts());
}

mg_status mg_log_scan_fwd(const float *log_coeffs, const float *log_values, float *h, int64_t B,
                          int64_t T, int64_t D, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_log_scan_fwd";
    g_detail[0] = 0;
    MG_TRY(check_dims(fn, {B, T + 1, D}));
    MG_TRY(check_channels(fn, D));
    if (T < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative size", fn);
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, nv = size_t(B) * (T + 1) * D;
    MG_TRY(check_ws(fn, ws, ws_bytes, log_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{log_coeffs, n * 4, "log_coeffs", false},
                           {log_values, nv * 4, "log_values", false},
                           {h, n * 4, "h", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_log_fwd(log_coeffs, log_values, h, B, T, D, ws, ws_bytes, stream, default_opts());
}

mg_status mg_log_scan_bwd(const float *log_coeffs, const float *log_values, const float *h,
                          const float *gh, float *dlog_coeffs, float *dlog_values, int64_t B,
                          int64_t T, int64_t D, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_log_scan_bwd";
    g_detail[0] = 0;
    MG_TRY(check_dims(fn, {B, T + 1, D}));
    MG_TRY(check_channels(fn, D));
    if (T < 0) return fail(MG_ERR_INVALID_ARG, "%s: negative size", fn);
    if (B == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D, nv = size_t(B) * (T + 1) * D;
    if (T == 0) {  // L does not depend on h_0: its gradient is zero
        MG_TRY(check_bufs(fn, {{dlog_values, nv * 4, "dlog_values", true}}));
        const cudaError_t e = cudaMemsetAsync(dlog_values, 0, nv * 4, stream);
        return e == cudaSuccess ? MG_OK : fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    }
    MG_TRY(check_ws(fn, ws, ws_bytes, log_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{log_coeffs, n * 4, "log_coeffs", false},
                           {log_values, nv * 4, "log_values", false},
                           {h, n * 4, "h", false},
                           {gh, n * 4, "gh", false},
                           {dlog_coeffs, n * 4, "dlog_coeffs", true},
                           {dlog_values, nv * 4, "dlog_values", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_log_bwd(log_coeffs, log_values, h, gh, dlog_coeffs, dlog_values, B, T, D, ws,
                          ws_bytes, stream, default_opts());
}

mg_status mg_affine_scan_fwd(const float *A, const float *Bm, float *Abar, float *Bbar, int64_t B,
                             int64_t T, int64_t n, int k, int v, void *ws, size_t ws_bytes,
                             cudaStream_t stream)
{
    const char *fn = "mg_affine_scan_fwd";
    g_detail[0] = 0;
    if (!valid_kv(k) || !valid_kv(v))
        return fail(MG_ERR_UNSUPPORTED, "%s: k=%d v=%d outside {1,2,4,8,16}", fn, k, v);
    MG_TRY(check_dims(fn, {B, T, n, k, k > v ? k : v}));
    if (B == 0 || T == 0 || n == 0) return MG_OK;
    const size_t s = size_t(B) * T * n;
    MG_TRY(check_ws(fn, ws, ws_bytes, affine_ws_bytes(B, T, n, k, v)));
    MG_TRY(check_bufs(fn, {{A, s * k * k * 4, "A", false},
                           {Bm, s * k * v * 4, "Bm", false},
                           {Abar, s * k * k * 4, "Abar", true},
                           {Bbar, s * k * v * 4, "Bbar", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_affine_fwd(A, Bm, nullptr, Abar, Bbar, B, T, n, k, v, ws, ws_bytes, stream,
                             default_opts());
}

mg_status mg_affine_scan_h0_fwd(const float *A, const float *Bm, const float *H0, float *Abar,
                                float *Bbar, int64_t B, int64_t T, int64_t n, int k, int v,
                                void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_affine_scan_h0_fwd";
    g_detail[0] = 0;
    if (!valid_kv(k) || !valid_kv(v))
        return fail(MG_ERR_UNSUPPORTED, "%s: k=%d v=%d outside {1,2,4,8,16}", fn, k, v);
    MG_TRY(check_dims(fn, {B, T, n, k, k > v ? k : v}));
    if (B == 0 || T == 0 || n == 0) return MG_OK;
    const size_t s = size_t(B) * T * n;
    MG_TRY(check_ws(fn, ws, ws_bytes, affine_ws_bytes(B, T, n, k, v)));
    MG_TRY(check_bufs(fn, {{A, s * k * k * 4, "A", false},
                           {Bm, s * k * v * 4, "Bm", false},
                           {H0, size_t(B) * n * k * v * 4, "H0", false},
                           {Abar, s * k * k * 4, "Abar", true},
                           {Bbar, s * k * v * 4, "Bbar", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_affine_fwd(A, Bm, H0, Abar, Bbar, B, T, n, k, v, ws, ws_bytes, stream,
                             default_opts());
}

mg_status mg_affine_scan_h0_bwd(const float *A, const float *H0, const float *Abar,
                                const float *Bbar, const float *gAbar, const float *gBbar,
                                float *dA, float *dB, float *dH0, int64_t B, int64_t T, int64_t n,
                                int k, int v, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_affine_scan_h0_bwd";
    g_detail[0] = 0;
    if (!valid_kv(k) || !valid_kv(v))
        return fail(MG_ERR_UNSUPPORTED, "%s: k=%d v=%d outside {1,2,4,8,16}", fn, k, v);
    MG_TRY(check_dims(fn, {B, T, n, k, k > v ? k : v}));
    if (B == 0 || n == 0) return MG_OK;
    const size_t s = size_t(B) * T * n, nh = size_t(B) * n * k * v;
    if (T == 0) {  // L does not depend on H0: its gradient is zero
        MG_TRY(check_bufs(fn, {{dH0, nh * 4, "dH0", true}}));
        const cudaError_t e = cudaMemsetAsync(dH0, 0, nh * 4, stream);
        return e == cudaSuccess ? MG_OK : fail(MG_ERR_LAUNCH, "%s: %s", fn, cudaGetErrorString(e));
    }
    MG_TRY(check_ws(fn, ws, ws_bytes, affine_ws_bytes(B, T, n, k, v)));
    MG_TRY(check_bufs(fn, {{A, s * k * k * 4, "A", false},
                           {H0, nh * 4, "H0", false},
                           {Abar, s * k * k * 4, "Abar", false},
                           {Bbar, s * k * v * 4, "Bbar", false},
                           {gAbar, s * k * k * 4, "gAbar", false},
                           {gBbar, s * k * v * 4, "gBbar", false},
                           {dA, s * k * k * 4, "dA", true},
                           {dB, s * k * v * 4, "dB", true},
                           {dH0, nh * 4, "dH0", true},
                           {ws, ws_bytes, "workspace", true}}));
    MG_TRY(launch_affine_bwd(A, Abar, Bbar, gAbar, gBbar, dA, dB, B, T, n, k, v, ws, ws_bytes,
                             stream, default_opts()));
    return launch_affine_h0_grad(A, H0, dB, dA, dH0, B, T, n, k, v, stream);
}

mg_status mg_affine_scan_bwd(const float *A, const float *Abar, const float *Bbar,
                             const float *gAbar, const float *gBbar, float *dA, float *dB,
                             int64_t B, int64_t T, int64_t n, int k, int v, void *ws,
                             size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "mg_affine_scan_bwd";
    g_detail[0] = 0;
    if (!valid_kv(k) || !valid_kv(v))
        return fail(MG_ERR_UNSUPPORTED, "%s: k=%d v=%d outside {1,2,4,8,16}", fn, k, v);
    MG_TRY(check_dims(fn, {B, T, n, k, k > v ? k : v}));
    if (B == 0 || T == 0 || n == 0) return MG_OK;
    const size_t s = size_t(B) * T * n;
    MG_TRY(check_ws(fn, ws, ws_bytes, affine_ws_bytes(B, T, n, k, v)));
    MG_TRY(check_bufs(fn, {{A, s * k * k * 4, "A", false},
                           {Abar, s * k * k * 4, "Abar", false},
                           {Bbar, s * k * v * 4, "Bbar", false},
                           {gAbar, s * k * k * 4, "gAbar", false},
                           {gBbar, s * k * v * 4, "gBbar", false},
                           {dA, s * k * k * 4, "dA", true},
                           {dB, s * k * v * 4, "dB", true},
                           {ws, ws_bytes, "workspace", true}}));
    return launch_affine_bwd(A, Abar, Bbar, gAbar, gBbar, dA, dB, B, T, n, k, v, ws, ws_bytes,
                             stream, default_opts());
}

mg_status mg_testing_linear_scan_fwd_stall(const float *a, const float *b, float *A, float *Bc,
                                           int64_t B, int64_t T, int64_t D, void *ws,
                                           size_t ws_bytes, int64_t stall_tile,
                                           uint64_t wait_limit_ns, cudaStream_t stream)
{
    const char *fn = "mg_testing_linear_scan_fwd_stall";
    g_detail[0] = 0;
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const size_t n = size_t(B) * T * D;
    MG_TRY(check_ws(fn, ws, ws_bytes, linear_ws_bytes(B, T, D)));
    MG_TRY(check_bufs(fn, {{a, n * 4, "a", false},
                           {b, n * 4, "b", false},
                           {A, n * 4, "A", true},
                           {Bc, n * 4, "Bc", true},
                           {ws, ws_bytes, "workspace", true}}));
    if (wait_limit_ns == 0 || wait_limit_ns > 10000000000ull)
        return fail(MG_ERR_INVALID_ARG, "%s: wait_limit_ns must be in (0, 1e10]", fn);
    LaunchOpts o = default_opts();
    o.wait_limit_ns = wait_limit_ns;
    o.stall_tile = stall_tile;
    return launch_linear_fwd(a, b, MG_F32, A, Bc, B, T, D, ws, ws_bytes, stream, o);
}

size_t mg_linear_scan_fwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

mg_status mg_linear_scan_fwd_noalloc(const void *a, const void *b, mg_dtype in_dt, float *A,
                                     float *Bc, int64_t B, int64_t T, int64_t D,
                                     cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_fwd_noalloc";
    g_detail[0] = 0;
    if (in_dt != MG_F32 && in_dt != MG_BF16)
        return fail(MG_ERR_UNSUPPORTED, "%s: input dtype %d not supported", fn, int(in_dt));
    MG_TRY(check_dims(fn, {B, T, D}));
    MG_TRY(check_channels(fn, D));
    if (B == 0 || T == 0 || D == 0) return MG_OK;
    const LaunchOpts o = default_opts();
    const size_t need = linear_fwd_ws_bytes(in_dt, B, T, D);
    if (need > kNoAllocScratchBytes)
        return fail(MG_ERR_INVALID_ARG,
                    "%s: (B,T,D) = (%lld,%lld,%lld) needs %zu bytes of scratch; the static scratch "
                    "holds %zu (use mg_linear_scan_fwd with a caller workspace)",
                    fn, (long long)B, (long long)T, (long long)D, need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    MG_TRY(noalloc_scratch(fn, &scratch));
    const size_t n = size_t(B) * T * D, isz = in_dt == MG_F32 ? 4 : 2;
    MG_TRY(check_bufs(fn, {{a, n * isz, "a", false},
                           {b, n * isz, "b", false},
                           {A, n * 4, "A", true},
                           {Bc, n * 4, "Bc", true}}));
    // The array keeps the previous call's contents.  Only the ticket and done
    // counters must start at zero (every completed launch leaves them so;
    // clearing them here also covers a launch that never started).  The
    // launch epoch is kept: it makes the previous calls' flags stale, and it
    // keeps the error record of earlier calls (read by
    // mg_linear_scan_fwd_noalloc_status) from being taken for this call's.
    static_assert(offsetof(Control, ticket) == 0 && offsetof(Control, done) == 4,
                  "the counters open the control block");
    const cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * sizeof(unsigned int), stream);
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "%s: clearing the scratch counters: %s", fn,
                    cudaGetErrorString(e));
    return launch_linear_fwd(a, b, in_dt, A, Bc, B, T, D, scratch, kNoAllocScratchBytes, stream, o);
}

mg_status mg_linear_scan_fwd_noalloc_status(cudaStream_t stream)
{
    const char *fn = "mg_linear_scan_fwd_noalloc_status";
    g_detail[0] = 0;
    void *scratch = nullptr;
    MG_TRY(noalloc_scratch(fn, &scratch));
    return read_status(fn, scratch, stream);
}

}  // extern "C"

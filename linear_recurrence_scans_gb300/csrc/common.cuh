// Internal declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lookback.cuh"
#include "mg_scan.h"

namespace mg {

// ---------------------------------------------------------------- host side

// Record a failure detail for mg_last_error_detail() and return `st`.
mg_status fail(mg_status st, const char *fmt, ...);

// Options a launcher takes beyond the op's own arguments.
struct LaunchOpts {
    unsigned long long wait_limit_ns = 2000000000ull;  // 2 s of %globaltimer
    unsigned int max_polls = 1u << 24;
    long long stall_tile = -1;                         // testing only
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace bytes for a tiled scan with `n_tiles` records of `record_bytes`.
inline size_t tiled_ws_bytes(size_t n_tiles, size_t record_bytes)
{
    return kControlBytes + align_up(n_tiles * sizeof(unsigned long long), 256) +
           n_tiles * record_bytes;
}

// Build the device-side look-back view of a workspace for `n_tiles` records.
inline Lookback make_lookback(void *ws, size_t n_tiles, const LaunchOpts &o)
{
    Lookback lb;
    char *base = static_cast<char *>(ws);
    lb.ctl = reinterpret_cast<Control *>(base);
    lb.flags = reinterpret_cast<unsigned long long *>(base + kControlBytes);
    lb.data = reinterpret_cast<float *>(
        base + kControlBytes + align_up(n_tiles * sizeof(unsigned long long), 256));
    lb.wait_limit_ns = o.wait_limit_ns;
    lb.max_polls = o.max_polls;
    lb.stall_tile = o.stall_tile;
    return lb;
}

struct bf16_t;  // bf16 storage type (raw bits), defined below

// Launchers (defined in channel_scan.cu / affine_scan.cu).  They assume the
// arguments were validated by the C entry points and B, T, D > 0.
// Workspace bytes each launch needs (each mirrors its launcher's choice of
// kernel shape).
size_t linear_fwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D);
size_t linear_bwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D);
size_t linear_ws_bytes(int64_t B, int64_t T, int64_t D);  // both, both dtypes
size_t log_ws_bytes(int64_t B, int64_t T, int64_t D);
size_t affine_ws_bytes(int64_t B, int64_t T, int64_t n, int k, int v);

mg_status launch_linear_fwd(const void *a, const void *b, mg_dtype dt, float *A, float *Bc,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes,
                            cudaStream_t s, const LaunchOpts &o);
mg_status launch_linear_bwd(const void *a, mg_dtype dt, const float *A, const float *Bc,
                            const float *gA, const float *gBc, float *da, float *db,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes,
                            cudaStream_t s, const LaunchOpts &o);
size_t linear_bwd16_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D);
size_t linear_h0_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D);
size_t varlen_ws_bytes(int64_t Ttot, int64_t D);
mg_status launch_varlen_fwd(const void *a, const void *b, mg_dtype dt, const int64_t *cu,
                            int64_t nseq, const float *h0, float *A, float *H, int64_t Ttot,
                            int64_t D, void *ws, size_t ws_bytes, cudaStream_t s,
                            const LaunchOpts &o);
mg_status launch_varlen_bwd(const void *a, mg_dtype dt, const int64_t *cu, int64_t nseq,
                            const float *h0, const float *A, const float *H, const float *gA,
                            const float *gH, float *da, float *db, float *dh0, int64_t Ttot,
                            int64_t D, void *ws, size_t ws_bytes, cudaStream_t s,
                            const LaunchOpts &o);
mg_status launch_linear_h0_fwd(const void *a, const void *b, mg_dtype dt, const float *h0,
                               float *A, float *H, int64_t B, int64_t T, int64_t D, void *ws,
                               size_t ws_bytes, cudaStream_t s, const LaunchOpts &o);
mg_status launch_linear_h0_bwd(const void *a, mg_dtype dt, const float *h0, const float *A,
                               const float *H, const float *gA, const float *gH, float *da,
                               float *db, float *dh0, int64_t B, int64_t T, int64_t D, void *ws,
                               size_t ws_bytes, cudaStream_t s, const LaunchOpts &o);
mg_status launch_linear_bwd_bf16_grads(const void *a, mg_dtype dt, const float *A, const float *Bc,
                                       const float *gA, const float *gBc, bf16_t *da,
                                       bf16_t *db, int64_t B, int64_t T, int64_t D,
                                       void *ws, size_t ws_bytes, cudaStream_t s,
                                       const LaunchOpts &o);
// The angle-fused scan's layer tables (filled on the host from perm, sgn and
// p2p; passed to the kernels by value): per layer and coordinate, the pair
// index, the role in the pair (0: first), the partner coordinate, the sign.
constexpr int kAngleMaxR = 8;
constexpr int kAngleMaxK = 32;
struct AngleTables {
    signed char pair[kAngleMaxR][kAngleMaxK];
    signed char role[kAngleMaxR][kAngleMaxK];
    signed char partner[kAngleMaxR][kAngleMaxK];
    float sgn[kAngleMaxR][kAngleMaxK];
    int R;
};
mg_status launch_angle(bool bwd, const float *theta, const float *scale, const float *gamma,
                       const float *b, const float *h0, const float *out, const float *grad_out,
                       float *h, float *dtheta, float *dscale, float *dgamma, float *db, float *dh0,
                       int64_t B, int64_t T, int64_t n, int k, int has_scale, int has_decay,
                       const AngleTables &tb, cudaStream_t s);
size_t mingru_ws_bytes(int64_t B, int64_t T, int64_t D);
mg_status launch_mingru_fwd(const void *x1, const void *x2, mg_dtype dt, float *A, float *Bc,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes,
                            cudaStream_t s, const LaunchOpts &o);
mg_status launch_mingru_bwd(const void *x1, const void *x2, mg_dtype dt, const float *A,
                            const float *Bc, const float *gA, const float *gBc, void *dx1,
                            void *dx2, mg_dtype grad_dt, int64_t B, int64_t T, int64_t D,
                            void *ws, size_t ws_bytes, cudaStream_t s, const LaunchOpts &o);
mg_status launch_log_bwd(const float *lc, const float *lv, const float *h, const float *gh,
                         float *dlc, float *dlv, int64_t B, int64_t T, int64_t D, void *ws,
                         size_t wsb, cudaStream_t s, const LaunchOpts &o);
mg_status launch_log_fwd(const float *lc, const float *lv, float *h, int64_t B, int64_t T,
                         int64_t D, void *ws, size_t ws_bytes, cudaStream_t s,
                         const LaunchOpts &o);
mg_status launch_affine_fwd(const float *A, const float *Bm, const float *H0, float *Abar,
                            float *Bbar, int64_t B, int64_t T, int64_t n, int k, int v, void *ws,
                            size_t ws_bytes, cudaStream_t s, const LaunchOpts &o);
mg_status launch_affine_h0_grad(const float *A, const float *H0, const float *dB, float *dA,
                                float *dH0, int64_t B, int64_t T, int64_t n, int k, int v,
                                cudaStream_t s);
mg_status launch_affine_bwd(const float *A, const float *Abar, const float *Bbar,
                            const float *gAbar, const float *gBbar, float *dA, float *dB,
                            int64_t B, int64_t T, int64_t n, int k, int v, void *ws,
                            size_t ws_bytes, cudaStream_t s, const LaunchOpts &o);

// ------------------------------------------------------------- device side

// bf16 storage type (raw bits); widening to float32 is exact.
struct bf16_t {
    unsigned short bits;
};

__device__ __forceinline__ float bf16_bits_to_float(unsigned int bits16)
{
    return __uint_as_float(bits16 << 16);
}

// Load VEC consecutive elements starting at p (aligned to VEC elements) and
// widen them to float32.
template <int VEC>
__device__ __forceinline__ void load_vec(const float *p, float (&o)[VEC])
{
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const float4 x = *reinterpret_cast<const float4 *>(p + 4 * q);
            o[4 * q + 0] = x.x;
            o[4 * q + 1] = x.y;
            o[4 * q + 2] = x.z;
            o[4 * q + 3] = x.w;
        }
    } else if constexpr (VEC == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        o[0] = x.x;
        o[1] = x.y;
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = p[v];
    }
}

template <int VEC>
__device__ __forceinline__ void load_vec(const bf16_t *p, float (&o)[VEC])
{
    if constexpr (VEC % 8 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 8; ++q) {
            const uint4 x = *reinterpret_cast<const uint4 *>(p + 8 * q);
            const unsigned w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[8 * q + 2 * e + 0] = __uint_as_float(w[e] << 16);
                o[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
    } else if constexpr (VEC == 4) {
        const uint2 x = *reinterpret_cast<const uint2 *>(p);
        o[0] = __uint_as_float(x.x << 16);
        o[1] = __uint_as_float(x.x & 0xffff0000u);
        o[2] = __uint_as_float(x.y << 16);
        o[3] = __uint_as_float(x.y & 0xffff0000u);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = bf16_bits_to_float(p[v].bits);
    }
}

// VEC consecutive input elements of type T kept in registers as loaded:
// bf16 stays packed (two per 32-bit word, one for VEC = 1) until each value
// is used, so a load is never tied to the instructions that widen it and
// the registers it needs are halved.  v-th value: x[v]; fill(c) sets every
// value to c (c exactly representable in T).
template <typename T, int VEC>
struct Raw;

template <int VEC>
struct Raw<float, VEC> {
    float w[VEC];
    __device__ __forceinline__ void load(const float *p) { load_vec<VEC>(p, w); }
    __device__ __forceinline__ float operator[](int v) const { return w[v]; }
    __device__ __forceinline__ void fill(float c)
    {
#pragma unroll
        for (int v = 0; v < VEC; ++v) w[v] = c;
    }
};

template <int VEC>
struct Raw<bf16_t, VEC> {
    static constexpr int NW = VEC == 1 ? 1 : VEC / 2;
    static_assert(VEC == 1 || VEC % 2 == 0, "packed bf16 pairs");
    unsigned w[NW];
    __device__ __forceinline__ void load(const bf16_t *p)
    {
        if constexpr (VEC % 8 == 0) {
#pragma unroll
            for (int q = 0; q < VEC / 8; ++q) {
                const uint4 x = *reinterpret_cast<const uint4 *>(p + 8 * q);
                w[4 * q + 0] = x.x;
                w[4 * q + 1] = x.y;
                w[4 * q + 2] = x.z;
                w[4 * q + 3] = x.w;
            }
        } else if constexpr (VEC == 4) {
            const uint2 x = *reinterpret_cast<const uint2 *>(p);
            w[0] = x.x;
            w[1] = x.y;
        } else if constexpr (VEC == 2) {
            w[0] = *reinterpret_cast<const unsigned *>(p);
        } else {
            w[0] = p[0].bits;
        }
    }
    __device__ __forceinline__ float operator[](int v) const
    {
        if constexpr (VEC == 1) return __uint_as_float(w[0] << 16);
        return (v & 1) ? __uint_as_float(w[v >> 1] & 0xffff0000u) : __uint_as_float(w[v >> 1] << 16);
    }
    __device__ __forceinline__ void fill(float c)
    {
        const unsigned h = __float_as_uint(c) >> 16;
#pragma unroll
        for (int q = 0; q < NW; ++q) w[q] = VEC == 1 ? h : (h | (h << 16));
    }
};

// Store VEC consecutive float32 values at p (aligned to VEC elements).
template <int VEC>
__device__ __forceinline__ void store_vec(float *p, const float (&x)[VEC])
{
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q)
            *reinterpret_cast<float4 *>(p + 4 * q) =
                make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) p[v] = x[v];
    }
}

// Store VEC consecutive values at p rounded to bf16 (round to nearest even).
__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi)
{
    const unsigned l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const unsigned h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

template <int VEC>
__device__ __forceinline__ void store_vec(bf16_t *p, const float (&x)[VEC])
{
    if constexpr (VEC % 8 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 8; ++q)
            *reinterpret_cast<uint4 *>(p + 8 * q) =
                make_uint4(pack_bf16x2(x[8 * q], x[8 * q + 1]), pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                           pack_bf16x2(x[8 * q + 4], x[8 * q + 5]), pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
    } else if constexpr (VEC == 4) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    } else if constexpr (VEC == 2) {
        *reinterpret_cast<unsigned *>(p) = pack_bf16x2(x[0], x[1]);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) p[v].bits = __bfloat16_as_ushort(__float2bfloat16_rn(x[v]));
    }
}

// Output stores of the scan epilogues.  With MG_STREAM_OUT (default on)
// they carry the streaming cache hint (st.global.cs, evicted first): the
// outputs are not read again by the kernel, so they do not displace the
// inputs that its second pass re-reads from L2.
#ifndef MG_STREAM_OUT
#define MG_STREAM_OUT 1
#endif
template <int VEC>
__device__ __forceinline__ void store_out(float *p, const float (&x)[VEC])
{
    if constexpr (MG_STREAM_OUT != 0 && VEC % 4 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q)
            __stcs(reinterpret_cast<float4 *>(p + 4 * q),
                   make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
    } else if constexpr (MG_STREAM_OUT != 0) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) __stcs(p + v, x[v]);
    } else {
        store_vec<VEC>(p, x);
    }
}

template <int VEC>
__device__ __forceinline__ void store_out(bf16_t *p, const float (&x)[VEC])
{
    if constexpr (MG_STREAM_OUT != 0 && VEC % 8 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 8; ++q)
            __stcs(reinterpret_cast<uint4 *>(p + 8 * q),
                   make_uint4(pack_bf16x2(x[8 * q], x[8 * q + 1]), pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                              pack_bf16x2(x[8 * q + 4], x[8 * q + 5]), pack_bf16x2(x[8 * q + 6], x[8 * q + 7])));
    } else if constexpr (MG_STREAM_OUT != 0 && VEC == 4) {
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3])));
    } else {
        store_vec<VEC>(p, x);
    }
}

// L2-only (.cg) variants for look-back records written by one CTA and read
// by another.
template <int VEC>
__device__ __forceinline__ void store_vec_cg(float *p, const float (&x)[VEC])
{
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q)
            __stcg(reinterpret_cast<float4 *>(p + 4 * q),
                   make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) __stcg(p + v, x[v]);
    }
}

template <int VEC>
__device__ __forceinline__ void load_vec_cg(const float *p, float (&o)[VEC])
{
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(p + 4 * q));
            o[4 * q + 0] = x.x;
            o[4 * q + 1] = x.y;
            o[4 * q + 2] = x.z;
            o[4 * q + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = __ldcg(p + v);
    }
}

// ------------------------------------------------------ log-space helpers
// 2^x by the PTX instruction ex2.approx (relative error near 2^-22).  The ftz
// form flushes subnormal results to zero (used for weights in [0, 1] whose
// tiny values cannot matter); the plain form keeps subnormal results.
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float ex2_sub(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2eF = 1.4426950408889634f;

// log(xs e^u + ys e^ym) returned as (m, s), the value being s e^m (natural
// logs; xs, ys >= 0 and finite).  m is the larger exponent, so one weight is
// 1 and the other e^-|u - ym|.  Both exponents -inf (both terms zero) make the
// gap NaN: the weight is then taken as 1 and m stays -inf, still the value 0.
__device__ __forceinline__ void log_add(float u, float xs, float ym, float ys, float &m, float &s)
{
    const float gap = u - ym;
    const float w = ex2_ftz(fminf(-fabsf(gap) * kLog2eF, 0.f));
    const bool ge = gap >= 0.f;
    m = ge ? u : ym;
    s = ge ? fmaf(ys, w, xs) : fmaf(xs, w, ys);
}

// ------------------------------------------------- TMA bulk copies (1D)
// One-dimensional bulk copies global -> shared completed on an mbarrier (the
// Hopper/Blackwell async copy engine; no tensor map needed).  Addresses and
// sizes must be multiples of 16 bytes.

__device__ __forceinline__ unsigned smem_addr(const void *p)
{
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(smem_addr(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" : : : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, unsigned bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
        : : "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, unsigned parity)
{
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ void tma_load_1d(void *dst, const void *src, unsigned bytes,
                                            unsigned long long *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        : : "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Per-thread asynchronous 16-byte copies global -> shared (LDGSTS), grouped
// per thread: commit closes a group, wait<N> returns once at most N of this
// thread's groups are still in flight.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" : : "r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" : : : "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" : : "n"(N) : "memory");
}

// Bounded wait for phase `parity` of `bar`; false if it gave up (the caller
// records the error; the copies themselves always complete).
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, unsigned parity,
                                                  unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > limit_ns) break;
    }
    return false;
}

}  // namespace mg

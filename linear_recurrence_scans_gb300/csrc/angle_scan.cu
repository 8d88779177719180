// The angle-fused scan (Kernel 4 of the page "minGRU - Triton kernels",
// sections "angle_scan_fwd", "angle_scan_bwd", "angle_scan_impl").
//
// Shapes as on the page: theta (B,T,n,R,half), scale and gamma (B,T,n),
// b (B,T,n,k), h0 (B,n,k), perm/sgn/p2p (R,k), half = k/2; output h (B,T,n,k).
// The page does not say how theta, perm, sgn and p2p form the transition;
// the reading implemented (and written out in the test oracle) is
//   h_t = s_t g_t Q_t h_{t-1} + b_t,   h_0 = h0,
//   Q_t = L_{R-1} ... L_0,  L_r: rotate each pair (perm[r][2i], perm[r][2i+1])
//   by theta_{t,r,i}, then scale coordinate j by sgn[r][j],
// with s_t = scale_t under has_scale (else 1), g_t = gamma_t under has_decay
// (else 1), and p2p[r] the inverse permutation of perm[r].
//
// One lane owns one coordinate j of one sequence (k lanes per sequence, k a
// power of two up to 32, so a sequence lies inside one warp).  A rotation
// needs the partner coordinate of the pair, which another lane of the same
// warp holds: one shuffle per layer.  The lane's pair index, role in the
// pair, partner and sign per layer come from p2p and perm, which are small
// host arrays passed by value (validated on the host).  Time runs
// sequentially per sequence; sequences are independent, so the data
// parallelism is B * n * k lanes.  sin and cos are the hardware
// approximations (__sincosf: absolute error near 2^-21 for angles within
// [-pi, pi]); each step's rotation error is that small, and the scale and
// decay factors (|s g| <= 1 in the module) damp old errors.
//
// Staging.  A block holds NSEQ = 256 / k consecutive sequences.  The inputs
// of one step for all of them (their theta rows, b or grad_out rows, h_{t-1}
// rows for the backward, scale and gamma) are copied into a shared-memory
// ring by every thread of the block, one float per 4-byte asynchronous copy
// (cp.async), so consecutive threads copy consecutive floats of each
// sequence's rows and the block's requests for one step cover a few
// contiguous runs of memory.  The ring holds NG groups of G steps; the block
// waits for a group, runs its G steps from shared memory, and refills the
// group's slots NG groups ahead, so the loads of a step are issued about
// NG*G steps before its use.
//
// Backward (exact, from the stored states): reverse time, lam_t =
// grad_out_t + A_{t+1}^T lam_{t+1}; db_t = lam_t; the layers are recomputed
// forward from h_{t-1} (the stored output, or h0) keeping each layer's
// input; dscale_t, dgamma_t from the group sum of lam_t . Q_t h_{t-1}; the
// gradient is carried back through the signs and the transposed rotations,
// giving dtheta per pair (the pair's first lane stores it) and
// A_t^T lam_t for the next step; dh0 = A_1^T lam_1.
#include <cmath>

#include "common.cuh"

namespace mg {

namespace {

constexpr int kAngleThreads = 256;
constexpr int kAngleG = 4;        // steps per group (one block barrier per group)
constexpr int kAngleNG = 4;       // groups in flight
constexpr int kAngleSteps = kAngleG * kAngleNG;   // ring slots
constexpr int kAngleJobs = 7;     // copies per thread per step, at most

struct AngleGeom {
    int64_t B, T, n;
    int has_scale, has_decay;
};

// The lane's role in each layer r < RR, unpacked once before the time loop:
// the partner lane (absolute lane index in the warp), the offset of the
// pair's angle in the sequence's theta row (r * half + pair index), the
// sign sgn[r][j], and q = +1 for the pair's second coordinate, -1 for its
// first (the sign of the partner's term in the rotation).
template <int RR>
struct LaneTables {
    int partner[RR], thoff[RR];
    float sgn[RR], q[RR];
};

template <int RR, int HALF>
__device__ __forceinline__ void lane_tables(const AngleTables &tb, int j, int gbase,
                                            LaneTables<RR> &lt)
{
#pragma unroll
    for (int r = 0; r < RR; ++r) {
        const bool on = r < tb.R;
        lt.partner[r] = gbase + (on ? tb.partner[r][j] : j);
        lt.thoff[r] = r * HALF + (on ? tb.pair[r][j] : 0);
        lt.sgn[r] = on ? tb.sgn[r][j] : 1.f;
        lt.q[r] = (on && tb.role[r][j]) ? 1.f : -1.f;
    }
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" : : "r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

// Shared layout of one step of a block (floats): theta rows [NSEQ][R*half]
// at 0, vec rows [NSEQ][k] at o_vec (b forward, grad_out backward), h_{t-1}
// rows [NSEQ][k] at o_hp (backward), scale [NSEQ] at o_s, gamma [NSEQ] at
// o_g; `floats` in all, rounded up to a multiple of 4.
struct StepLayout {
    int o_vec, o_hp, o_s, o_g, floats;
};

__host__ __device__ inline StepLayout step_layout(int nseq, int R, int k, bool bwd)
{
    StepLayout L;
    L.o_vec = nseq * R * (k / 2);
    L.o_hp = L.o_vec + nseq * k;
    L.o_s = L.o_hp + (bwd ? nseq * k : 0);
    L.o_g = L.o_s + nseq;
    L.floats = (L.o_g + nseq + 3) / 4 * 4;
    return L;
}

// The copies this thread makes for every step: copy i (i < kAngleJobs) is
// float e = threadIdx.x + i * 256 of the step's layout, from `src[i]` at
// t = 0 advancing by `stride[i]` floats per step; bit i of `live` says the
// copy exists (a float of the layout, of a sequence of the batch), bit i of
// `prev` that it reads h_{t-1} (nothing to read at t = 0).  A step holds at
// most 128 R + 2*256 + 2*NSEQ <= 1792 floats (R <= 8, NSEQ <= 128), so
// seven copies per thread cover it.
struct CopyJobs {
    const float *src[kAngleJobs];
    int stride[kAngleJobs];   // n * (floats per (b, t, n)) < 2^31 (checked on the host)
    unsigned live, prev;
};

__device__ __forceinline__ void make_jobs(const float *theta, const float *scale,
                                          const float *gamma, const float *vec, const float *hp,
                                          const AngleGeom &g, const StepLayout &L, int nseq,
                                          int64_t seq0, int R, int k, CopyJobs &cj)
{
    const int half = k / 2;
    const int rh = R * half;
    const int total = L.o_g + nseq;
    const int64_t nall = g.B * g.n;
    cj.live = 0u;
    cj.prev = 0u;
#pragma unroll
    for (int i = 0; i < kAngleJobs; ++i) {
        const int e = threadIdx.x + i * kAngleThreads;
        int sl = 0, off = 0;
        const float *base = theta;
        int64_t per = rh;   // floats of this stream per (b, t, n)
        bool prev = false, on = e < total;
        if (e < L.o_vec) {
            sl = e / rh; off = e % rh;
        } else if (e < L.o_hp) {
            sl = (e - L.o_vec) / k; off = (e - L.o_vec) % k; base = vec; per = k;
        } else if (e < L.o_s) {
            sl = (e - L.o_hp) / k; off = (e - L.o_hp) % k; base = hp; per = k; prev = true;
        } else if (e < L.o_g) {
            sl = e - L.o_s; base = scale; per = 1; on = on && g.has_scale;
        } else {
            sl = e - L.o_g; base = gamma; per = 1; on = on && g.has_decay;
        }
        const int64_t seq = seq0 + sl;
        on = on && seq < nall;
        const int64_t sq = on ? seq : 0;
        const int64_t st0 = (sq / g.n) * g.T * g.n + sq % g.n;   // step index of (b, 0, n)
        // h_{t-1} rows: the source of step t is row t - 1 (only used for t >= 1)
        cj.src[i] = on ? base + (prev ? st0 - g.n : st0) * per + off : theta;
        cj.stride[i] = int(g.n * per);
        cj.live |= unsigned(on) << i;
        cj.prev |= unsigned(prev) << i;
    }
}

// Issue this thread's copies of step t (t < 2^31) into `slot`.
__device__ __forceinline__ void issue_step(const CopyJobs &cj, float *slot, int t)
{
#pragma unroll
    for (int i = 0; i < kAngleJobs; ++i) {
        if (!((cj.live >> i) & 1u) || (((cj.prev >> i) & 1u) && t == 0)) continue;
        cp_async4(slot + threadIdx.x + i * kAngleThreads, cj.src[i] + int64_t(t) * cj.stride[i]);
    }
}

template <int K, int RR>
__global__ void __launch_bounds__(kAngleThreads)
    angle_fwd_kernel(const float *theta, const float *scale, const float *gamma, const float *b,
                     const float *h0, float *h, const AngleGeom g, const AngleTables tb)
{
    constexpr int NSEQ = kAngleThreads / K, HALF = K / 2;
    extern __shared__ float4 angle_smem[];
    float *const ring = reinterpret_cast<float *>(angle_smem);
    const int R = tb.R;
    const StepLayout L = step_layout(NSEQ, R, K, false);
    const int64_t seq0 = int64_t(blockIdx.x) * NSEQ;
    const int sl = threadIdx.x / K, j = threadIdx.x % K;
    const int lane = threadIdx.x & 31;
    const int64_t seq = seq0 + sl;
    const bool act = seq < g.B * g.n;
    LaneTables<RR> lt;
    lane_tables<RR, HALF>(tb, j, lane - j, lt);
    CopyJobs cj;
    make_jobs(theta, scale, gamma, b, nullptr, g, L, NSEQ, seq0, R, K, cj);
    const int64_t sq = act ? seq : 0;
    const int64_t st0 = (sq / g.n) * g.T * g.n + sq % g.n;   // step index of (b, 0, n)
    const int64_t ngroups = (g.T + kAngleG - 1) / kAngleG;
    auto issue_group = [&](int64_t gi) {
        for (int u = 0; u < kAngleG; ++u) {
            const int64_t t = gi * kAngleG + u;
            if (gi < ngroups && t < g.T)
                issue_step(cj, ring + int((t % kAngleSteps) * L.floats), int(t));
        }
        cp_async_commit();
    };
    for (int gi = 0; gi < kAngleNG; ++gi) issue_group(gi);

    float x = act ? __ldg(h0 + sq * K + j) : 0.f;
    float *const h_lane = h + st0 * K + j;   // h of step t at h_lane[t * n * K]
    const int nK = int(g.n * K);
    for (int64_t gi = 0; gi < ngroups; ++gi) {
        cp_async_wait<kAngleNG - 1>();
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kAngleG; ++u) {
            const int64_t t = gi * kAngleG + u;
            if (t >= g.T) break;
            const float *sp = ring + int((t % kAngleSteps) * L.floats);
            const float *th = sp + sl * R * HALF;
#pragma unroll
            for (int r = 0; r < RR; ++r) {
                if (r >= R) break;
                float sn, cs;
                __sincosf(th[lt.thoff[r]], &sn, &cs);
                const float v = __shfl_sync(0xffffffffu, x, lt.partner[r]);
                x = fmaf(cs, x, lt.q[r] * sn * v) * lt.sgn[r];
            }
            const float f = (g.has_scale ? sp[L.o_s + sl] : 1.f) * (g.has_decay ? sp[L.o_g + sl] : 1.f);
            x = fmaf(f, x, sp[L.o_vec + sl * K + j]);
            if (act) h_lane[int64_t(int(t)) * nK] = x;
        }
        __syncthreads();   // every thread is done with the group's slots
        issue_group(gi + kAngleNG);
    }
    cp_async_wait<0>();
}

template <int K, int RR>
__global__ void __launch_bounds__(kAngleThreads)
    angle_bwd_kernel(const float *theta, const float *scale, const float *gamma, const float *h0,
                     const float *out, const float *grad_out, float *dtheta, float *dscale,
                     float *dgamma, float *db, float *dh0, const AngleGeom g, const AngleTables tb)
{
    constexpr int NSEQ = kAngleThreads / K, HALF = K / 2;
    extern __shared__ float4 angle_smem[];
    float *const ring = reinterpret_cast<float *>(angle_smem);
    const int R = tb.R;
    const StepLayout L = step_layout(NSEQ, R, K, true);
    const int64_t seq0 = int64_t(blockIdx.x) * NSEQ;
    const int sl = threadIdx.x / K, j = threadIdx.x % K;
    const int lane = threadIdx.x & 31;
    const int64_t seq = seq0 + sl;
    const bool act = seq < g.B * g.n;
    LaneTables<RR> lt;
    lane_tables<RR, HALF>(tb, j, lane - j, lt);
    CopyJobs cj;
    make_jobs(theta, scale, gamma, grad_out, out, g, L, NSEQ, seq0, R, K, cj);
    const int64_t sq = act ? seq : 0;
    const int64_t st0 = (sq / g.n) * g.T * g.n + sq % g.n;   // step index of (b, 0, n)
    const int64_t ngroups = (g.T + kAngleG - 1) / kAngleG;
    // processing index q = T-1-t (reverse time) names the ring slot
    auto issue_group = [&](int64_t gi) {
        for (int u = 0; u < kAngleG; ++u) {
            const int64_t q = gi * kAngleG + u;
            if (gi < ngroups && q < g.T)
                issue_step(cj, ring + int((q % kAngleSteps) * L.floats), int(g.T - 1 - q));
        }
        cp_async_commit();
    };
    for (int gi = 0; gi < kAngleNG; ++gi) issue_group(gi);

    const float h0j = act ? __ldg(h0 + sq * K + j) : 0.f;
    float carry = 0.f;   // A_{t+1}^T lam_{t+1}
    for (int64_t gi = 0; gi < ngroups; ++gi) {
        cp_async_wait<kAngleNG - 1>();
        __syncthreads();
#pragma unroll 1
        for (int u = 0; u < kAngleG; ++u) {
            const int64_t q = gi * kAngleG + u;
            if (q >= g.T) break;
            const int64_t t = g.T - 1 - q;
            const int64_t st = st0 + t * g.n;
            const float *sp = ring + int((q % kAngleSteps) * L.floats);
            const float *th = sp + sl * R * HALF;
            const float s_t = g.has_scale ? sp[L.o_s + sl] : 1.f;
            const float g_t = g.has_decay ? sp[L.o_g + sl] : 1.f;
            const float lam = sp[L.o_vec + sl * K + j] + carry;
            // the layers forward from h_{t-1}, keeping each layer's input
            float xs[RR + 1], sn[RR], cs[RR];
            xs[0] = t > 0 ? sp[L.o_hp + sl * K + j] : h0j;
#pragma unroll
            for (int r = 0; r < RR; ++r) {
                if (r < R) {
                    __sincosf(th[lt.thoff[r]], &sn[r], &cs[r]);
                    const float v = __shfl_sync(0xffffffffu, xs[r], lt.partner[r]);
                    xs[r + 1] = fmaf(cs[r], xs[r], lt.q[r] * sn[r] * v) * lt.sgn[r];
                } else {
                    xs[r + 1] = xs[r];
                    sn[r] = 0.f;
                    cs[r] = 1.f;
                }
            }
            // lam . Q h_{t-1} over the sequence's K lanes (layers past R copy
            // their input, so the last entry is Q h_{t-1})
            float dot = lam * xs[RR];
#pragma unroll
            for (int off = K / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            float uu = s_t * g_t * lam;
#pragma unroll
            for (int r = RR - 1; r >= 0; --r) {
                if (r >= R) continue;
                const float up = uu * lt.sgn[r];   // gradient after the signs
                const float v = __shfl_sync(0xffffffffu, up, lt.partner[r]);
                const float xq = __shfl_sync(0xffffffffu, xs[r], lt.partner[r]);
                if (act && lt.q[r] < 0.f) {   // the pair's first lane: dtheta
                    const float dth = up * (-sn[r] * xs[r] - cs[r] * xq) + v * (cs[r] * xs[r] - sn[r] * xq);
                    dtheta[st * R * HALF + lt.thoff[r]] = dth;
                }
                uu = fmaf(cs[r], up, -lt.q[r] * sn[r] * v);
            }
            if (act) {
                db[st * K + j] = lam;
                if (j == 0) {
                    dscale[st] = g.has_scale ? g_t * dot : 0.f;
                    dgamma[st] = g.has_decay ? s_t * dot : 0.f;
                }
            }
            carry = uu;
        }
        __syncthreads();   // every thread is done with the group's slots
        issue_group(gi + kAngleNG);
    }
    cp_async_wait<0>();
    if (act) dh0[sq * K + j] = carry;
}

template <int K, int RR>
mg_status angle_launch(bool bwd, const float *theta, const float *scale, const float *gamma,
                       const float *b, const float *h0, const float *out, const float *grad_out,
                       float *h, float *dtheta, float *dscale, float *dgamma, float *db, float *dh0,
                       const AngleGeom &g, const AngleTables &tb, cudaStream_t s)
{
    constexpr int NSEQ = kAngleThreads / K;
    const StepLayout L = step_layout(NSEQ, tb.R, K, bwd);
    const size_t smem = size_t(kAngleSteps) * L.floats * sizeof(float);
    const unsigned blocks = unsigned((g.B * g.n + NSEQ - 1) / NSEQ);
    cudaError_t e;
    if (bwd) {
        e = cudaFuncSetAttribute(angle_bwd_kernel<K, RR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e == cudaSuccess)
            angle_bwd_kernel<K, RR><<<blocks, kAngleThreads, smem, s>>>(
                theta, scale, gamma, h0, out, grad_out, dtheta, dscale, dgamma, db, dh0, g, tb);
    } else {
        e = cudaFuncSetAttribute(angle_fwd_kernel<K, RR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e == cudaSuccess)
            angle_fwd_kernel<K, RR><<<blocks, kAngleThreads, smem, s>>>(theta, scale, gamma, b, h0, h,
                                                                        g, tb);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", bwd ? "mg_angle_scan_bwd" : "mg_angle_scan_fwd",
                    cudaGetErrorString(e));
    return MG_OK;
}

}  // namespace

mg_status launch_angle(bool bwd, const float *theta, const float *scale, const float *gamma,
                       const float *b, const float *h0, const float *out, const float *grad_out,
                       float *h, float *dtheta, float *dscale, float *dgamma, float *db, float *dh0,
                       int64_t B, int64_t T, int64_t n, int k, int has_scale, int has_decay,
                       const AngleTables &tb, cudaStream_t s)
{
    const AngleGeom g{B, T, n, has_scale, has_decay};
    // layer arrays sized to the next power of two >= R (layers past R are
    // skipped at run time)
    const int rr = tb.R <= 1 ? 1 : tb.R <= 2 ? 2 : tb.R <= 4 ? 4 : 8;
#define MG_ANGLE_CALL(KK, RRR)                                                                  \
    return angle_launch<KK, RRR>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta,    \
                                 dscale, dgamma, db, dh0, g, tb, s)
#define MG_ANGLE_K(KK)                                                                          \
    switch (rr) {                                                                               \
    case 1: MG_ANGLE_CALL(KK, 1);                                                              \
    case 2: MG_ANGLE_CALL(KK, 2);                                                              \
    case 4: MG_ANGLE_CALL(KK, 4);                                                              \
    default: MG_ANGLE_CALL(KK, 8);                                                             \
    }
    switch (k) {
    case 2: MG_ANGLE_K(2);
    case 4: MG_ANGLE_K(4);
    case 8: MG_ANGLE_K(8);
    case 16: MG_ANGLE_K(16);
    case 32: MG_ANGLE_K(32);
    default: break;
    }
#undef MG_ANGLE_K
#undef MG_ANGLE_CALL
    return fail(MG_ERR_UNSUPPORTED, "angle scan: k = %d outside {2, 4, 8, 16, 32}", k);
}

}  // namespace mg

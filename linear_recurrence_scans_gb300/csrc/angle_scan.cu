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
// sequentially per sequence; U steps of inputs are loaded ahead of their
// use so the loads of a warp overlap its arithmetic.  Sequences are
// independent, so the data parallelism is B * n * k lanes.  sin and cos are
// the hardware approximations (__sincosf: absolute error near 2^-21 for
// angles within [-pi, pi]); each step's rotation error is that small, and
// the scale and decay factors (|s g| <= 1 in the module) damp old errors.
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

constexpr int kAngleU = 4;        // steps of inputs loaded ahead
constexpr int kAngleThreads = 256;

struct AngleGeom {
    int64_t B, T, n;
    int has_scale, has_decay;
};

template <int K>
struct LaneTables {
    int pair[kAngleMaxR], role[kAngleMaxR], partner[kAngleMaxR];
    float sgn[kAngleMaxR];
};

template <int K>
__device__ __forceinline__ void lane_tables(const AngleTables &tb, int j, int gbase,
                                            LaneTables<K> &lt)
{
#pragma unroll
    for (int r = 0; r < kAngleMaxR; ++r) {
        const bool on = r < tb.R;
        lt.pair[r] = on ? tb.pair[r][j] : 0;
        lt.role[r] = on ? tb.role[r][j] : 0;
        lt.partner[r] = gbase + (on ? tb.partner[r][j] : j);
        lt.sgn[r] = on ? tb.sgn[r][j] : 1.f;
    }
}

// Inputs of one step for this lane.
struct StepIn {
    float th[kAngleMaxR];
    float f;      // s_t g_t
    float s, g;   // s_t, g_t (the backward needs them apart)
    float x;      // b_t[j] (forward) or grad_out_t[j] (backward)
    float hp;     // h_{t-1}[j] (backward only)
};

template <int K>
__device__ __forceinline__ void load_step(const float *theta, const float *scale, const float *gamma,
                                          const float *vec, const float *hprev, const AngleGeom &g,
                                          const LaneTables<K> &lt, int R, int64_t seq, int64_t t,
                                          int j, bool bwd, StepIn &in)
{
    constexpr int HALF = K / 2;
    const int64_t bb = seq / g.n, nn = seq % g.n;
    const int64_t st = (bb * g.T + t) * g.n + nn;   // step index (b, t, n)
#pragma unroll
    for (int r = 0; r < kAngleMaxR; ++r)
        in.th[r] = r < R ? __ldg(theta + (st * R + r) * HALF + lt.pair[r]) : 0.f;
    in.s = g.has_scale ? __ldg(scale + st) : 1.f;
    in.g = g.has_decay ? __ldg(gamma + st) : 1.f;
    in.f = in.s * in.g;
    in.x = __ldg(vec + st * K + j);
    if (bwd) in.hp = t > 0 ? __ldg(hprev + (st - g.n) * K + j) : 0.f;
}

template <int K>
__global__ void __launch_bounds__(kAngleThreads)
    angle_fwd_kernel(const float *theta, const float *scale, const float *gamma, const float *b,
                     const float *h0, float *h, const AngleGeom g, const AngleTables tb)
{
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int j = int(gid % K);
    const int64_t seq = gid / K;
    const int lane = threadIdx.x & 31;
    const int gbase = lane - j;   // first lane of this sequence's group
    const bool act = seq < g.B * g.n;
    const int R = tb.R;
    LaneTables<K> lt;
    lane_tables<K>(tb, j, gbase, lt);
    const int64_t sq = act ? seq : 0;   // inactive lanes shadow sequence 0 (no stores)
    float x = __ldg(h0 + sq * K + j);
    StepIn in[kAngleU];
    for (int64_t t0 = 0; t0 < g.T; t0 += kAngleU) {
#pragma unroll
        for (int u = 0; u < kAngleU; ++u)
            if (t0 + u < g.T) load_step<K>(theta, scale, gamma, b, nullptr, g, lt, R, sq, t0 + u, j, false, in[u]);
#pragma unroll
        for (int u = 0; u < kAngleU; ++u) {
            if (t0 + u >= g.T) break;
#pragma unroll
            for (int r = 0; r < kAngleMaxR; ++r) {
                if (r >= R) break;
                float s, c;
                __sincosf(in[u].th[r], &s, &c);
                const float v = __shfl_sync(0xffffffffu, x, lt.partner[r]);
                x = fmaf(c, x, (lt.role[r] ? s : -s) * v) * lt.sgn[r];
            }
            x = fmaf(in[u].f, x, in[u].x);
            if (act) {
                const int64_t bb = seq / g.n, nn = seq % g.n;
                h[((bb * g.T + t0 + u) * g.n + nn) * K + j] = x;
            }
        }
    }
}

template <int K>
__global__ void __launch_bounds__(kAngleThreads)
    angle_bwd_kernel(const float *theta, const float *scale, const float *gamma, const float *h0,
                     const float *out, const float *grad_out, float *dtheta, float *dscale,
                     float *dgamma, float *db, float *dh0, const AngleGeom g, const AngleTables tb)
{
    constexpr int HALF = K / 2;
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int j = int(gid % K);
    const int64_t seq = gid / K;
    const int lane = threadIdx.x & 31;
    const int gbase = lane - j;
    const bool act = seq < g.B * g.n;
    const int R = tb.R;
    LaneTables<K> lt;
    lane_tables<K>(tb, j, gbase, lt);
    const int64_t sq = act ? seq : 0;
    const int64_t bb = sq / g.n, nn = sq % g.n;
    const float h0j = __ldg(h0 + sq * K + j);
    float carry = 0.f;   // A_{t+1}^T lam_{t+1}
    StepIn in[kAngleU];
    for (int64_t te = g.T; te > 0; te -= kAngleU) {   // steps te-1 down to te-U
#pragma unroll
        for (int u = 0; u < kAngleU; ++u)
            if (te - 1 - u >= 0)
                load_step<K>(theta, scale, gamma, grad_out, out, g, lt, R, sq, te - 1 - u, j, true, in[u]);
#pragma unroll
        for (int u = 0; u < kAngleU; ++u) {
            const int64_t t = te - 1 - u;
            if (t < 0) break;
            const int64_t st = (bb * g.T + t) * g.n + nn;
            const float lam = in[u].x + carry;
            // the layers forward from h_{t-1}, keeping each layer's input
            float xs[kAngleMaxR + 1], sn[kAngleMaxR], cs[kAngleMaxR];
            xs[0] = t > 0 ? in[u].hp : h0j;
#pragma unroll
            for (int r = 0; r < kAngleMaxR; ++r) {
                if (r < R) {
                    __sincosf(in[u].th[r], &sn[r], &cs[r]);
                    const float v = __shfl_sync(0xffffffffu, xs[r], lt.partner[r]);
                    xs[r + 1] = fmaf(cs[r], xs[r], (lt.role[r] ? sn[r] : -sn[r]) * v) * lt.sgn[r];
                } else {
                    xs[r + 1] = xs[r];
                    sn[r] = 0.f;
                    cs[r] = 1.f;
                }
            }
            // lam . Q h_{t-1} over the sequence's K lanes (layers past R copy
            // their input, so the last entry is Q h_{t-1})
            float dot = lam * xs[kAngleMaxR];
#pragma unroll
            for (int off = K / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            float uu = in[u].f * lam;
#pragma unroll
            for (int r = kAngleMaxR - 1; r >= 0; --r) {
                if (r >= R) continue;
                const float up = uu * lt.sgn[r];   // gradient after the signs
                const float v = __shfl_sync(0xffffffffu, up, lt.partner[r]);
                const float xq = __shfl_sync(0xffffffffu, xs[r], lt.partner[r]);
                if (act && lt.role[r] == 0) {   // the pair's first lane: dtheta
                    const float dth = up * (-sn[r] * xs[r] - cs[r] * xq) + v * (cs[r] * xs[r] - sn[r] * xq);
                    dtheta[(st * R + r) * HALF + lt.pair[r]] = dth;
                }
                uu = fmaf(cs[r], up, (lt.role[r] ? -sn[r] : sn[r]) * v);
            }
            if (act) {
                db[st * K + j] = lam;
                if (j == 0) {
                    dscale[st] = g.has_scale ? in[u].g * dot : 0.f;
                    dgamma[st] = g.has_decay ? in[u].s * dot : 0.f;
                }
            }
            carry = uu;
        }
    }
    if (act) dh0[sq * K + j] = carry;
}

template <int K>
mg_status angle_launch(bool bwd, const float *theta, const float *scale, const float *gamma,
                       const float *b, const float *h0, const float *out, const float *grad_out,
                       float *h, float *dtheta, float *dscale, float *dgamma, float *db, float *dh0,
                       const AngleGeom &g, const AngleTables &tb, cudaStream_t s)
{
    const int64_t lanes = g.B * g.n * K;
    const unsigned blocks = unsigned((lanes + kAngleThreads - 1) / kAngleThreads);
    if (bwd)
        angle_bwd_kernel<K><<<blocks, kAngleThreads, 0, s>>>(theta, scale, gamma, h0, out, grad_out,
                                                             dtheta, dscale, dgamma, db, dh0, g, tb);
    else
        angle_fwd_kernel<K><<<blocks, kAngleThreads, 0, s>>>(theta, scale, gamma, b, h0, h, g, tb);
    const cudaError_t e = cudaGetLastError();
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
    switch (k) {
    case 2: return angle_launch<2>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta, dscale, dgamma, db, dh0, g, tb, s);
    case 4: return angle_launch<4>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta, dscale, dgamma, db, dh0, g, tb, s);
    case 8: return angle_launch<8>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta, dscale, dgamma, db, dh0, g, tb, s);
    case 16: return angle_launch<16>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta, dscale, dgamma, db, dh0, g, tb, s);
    case 32: return angle_launch<32>(bwd, theta, scale, gamma, b, h0, out, grad_out, h, dtheta, dscale, dgamma, db, dh0, g, tb, s);
    default: break;
    }
    return fail(MG_ERR_UNSUPPORTED, "angle scan: k = %d outside {2, 4, 8, 16, 32}", k);
}

}  // namespace mg

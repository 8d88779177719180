// The minGRU gate fused into the linear scan (forward and gradients).
//
// A minGRU layer turns two projections x1, x2 of its input into the scan's
// coefficient and value, z = sigmoid(x1), a = 1 - z, b = z g(x2) with
// g(x) = x + 0.5 (x >= 0) else sigmoid(x), and runs linear_scan_fwd of the
// page "minGRU - Triton kernels" on (a, b) (the op its scan dispatch calls).
// Computing the gate inside the scan removes the gate's own pass over HBM
// (writing a and b, then reading them back): the fused forward reads x1, x2
// and writes Bc (and A when asked), the fused backward reads x1, x2, Bc,
// gBc (and A, gA when asked) and writes dx1, dx2.
//
// Both run on the chunk engine (scan_engine.cuh) exactly as the linear scan
// and its adjoint do (channel_scan.cu); the ops below only form the elements
// from the gate in registers.  The forward keeps pass 1's elements in shared
// memory for pass 2; the backward evaluates the coefficient in pass 1 and
// the whole gate in pass 2.  Gradients:
//   da, db from the linear adjoint (mu, lam recurrences, reverse time)
//   dx1 = (db g(x2) - da) z (1 - z),   dx2 = db z g'(x2)
// with g'(0) = 1 (the branch x + 0.5 defines g at 0).
#include <cmath>
#include <type_traits>

#include "scan_engine.cuh"

#ifndef MG_MG_PEEK32
#define MG_MG_PEEK32 0
#endif

namespace mg {
namespace {

// --------------------------------------------------------------- the gate
// sigmoid(+-x) from one exponential of -|x| (never overflows): with
// e = exp(-|x|) and r = 1 / (1 + e), sigmoid(|x|) = r and sigmoid(-|x|) = e r,
// so 1 - sigmoid(x1) is formed as sigmoid(-x1), without the cancellation of
// 1 - z as z approaches 1.  The exponentials are the hardware 2^x (PTX
// ex2.approx, relative error about 2^-22, subnormal results kept), and the
// two reciprocals 1 / (1 + e1), 1 / (1 + e2) share one: with
// R = 1 / ((1 + e1)(1 + e2)), 1 / (1 + e1) = R (1 + e2) and
// 1 / (1 + e2) = R (1 + e1) (the product lies in (1, 4], no overflow).
struct Gate {
    float a;    // 1 - z
    float z;    // sigmoid(x1)
    float g;    // g(x2)
    float gp;   // g'(x2)
};

__device__ __forceinline__ Gate gate(float x1, float x2)
{
    const float e1 = ex2_sub(-fabsf(x1) * kLog2eF);
    const float e2 = ex2_sub(fminf(x2, 0.f) * kLog2eF);   // x2 < 0: sigmoid(x2) = e2 / (1 + e2)
    const float p1 = 1.f + e1, p2 = 1.f + e2;
    const float R = __fdividef(1.f, p1 * p2);
    const float r1 = R * p2, r2 = R * p1;
    const float er1 = e1 * r1, s2 = e2 * r2;
    Gate q;
    q.z = x1 >= 0.f ? r1 : er1;
    q.a = x1 >= 0.f ? er1 : r1;
    q.g = x2 >= 0.f ? x2 + 0.5f : s2;
    q.gp = x2 >= 0.f ? 1.f : s2 * r2;
    return q;
}

// 1 - sigmoid(x1) alone (the backward's coefficient a_{t+1}).
__device__ __forceinline__ float gate_a(float x1)
{
    const float e1 = ex2_sub(-fabsf(x1) * kLog2eF);
    const float r1 = __fdividef(1.f, 1.f + e1);
    return x1 >= 0.f ? e1 * r1 : r1;
}

// ------------------------------------------------------------- forward
// Element of step t: (a_t, b_t) from (x1_t, x2_t); state (A, h) as in the
// linear forward.  WA: A is written (otherwise only Bc).  Pass 1 keeps the
// elements in shared memory (the engine's stash), so pass 2 neither reads
// x1, x2 again nor evaluates the gate a second time.  Steps past T load
// x1 = -inf, x2 = 0, whose gate is exactly the identity element (a = 1,
// b = 0), so no step needs a bounds select.
template <typename Tin, int VEC_, int L_, bool WA>
struct MinFwd {
    static constexpr int NS = 2, VEC = VEC_, L = L_;
    static constexpr bool kReverse = false;
    // a prefix's running product is read only when A is written
    static constexpr unsigned kPrefixStates = WA ? 0b11u : 0b10u;
    // look-back peek: measured faster for bf16 inputs, slower for float32
    static constexpr bool kPeek = MG_MG_PEEK32 != 0 || !std::is_same_v<Tin, float>;
    static constexpr bool kStash = true;
    using S = St<NS, VEC>;
    struct Args {
        const Tin *x1;
        const Tin *x2;
        float *A;
        float *Bc;
    };
    struct Regs {
        Raw<Tin, VEC> x1[L];
        Raw<Tin, VEC> x2[L];
    };

    __device__ static int valid_steps(const ChanGeom &g, int64_t t0, bool act)
    {
        const int64_t rem = g.T - t0;
        return act ? int(rem < 0 ? 0 : (rem > L ? L : rem)) : 0;
    }
    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        const int nv = valid_steps(g, t0, act);
#pragma unroll
        for (int i = 0; i < L; ++i) {
            if (i < nv) {
                const int64_t off = (bb * g.T + t0 + i) * g.D + d;
                r.x1[i].load(p.x1 + off);
                r.x2[i].load(p.x2 + off);
            } else {
                r.x1[i].fill(-INFINITY);
                r.x2[i].fill(0.f);
            }
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const Gate q = gate(r.x1[i][v], r.x2[i][v]);
            e.v[0][v] = q.a;
            e.v[1][v] = q.z * q.g;
        }
        return e;
    }
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = 1.f;
            e.v[1][v] = 0.f;
        }
        return e;
    }
    __device__ static S initial(const Args &, const ChanGeom &, int64_t, int, bool)
    {
        return identity();
    }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            o.v[0][v] = y.v[0][v] * x.v[0][v];
            o.v[1][v] = fmaf(y.v[0][v], x.v[1][v], y.v[1][v]);
        }
        return o;
    }
    __device__ static void epilogue_stash(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                          int d, bool act, const StashView<MinFwd> &sv, S &st)
    {
        const int nv = valid_steps(g, t0, act);
#pragma unroll
        for (int i = 0; i < L; ++i) {
            if (i < nv) {
                const S e = sv.get(i);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    st.v[0][v] = e.v[0][v] * st.v[0][v];
                    st.v[1][v] = fmaf(e.v[0][v], st.v[1][v], e.v[1][v]);
                }
                const int64_t off = (bb * g.T + t0 + i) * g.D + d;
                if constexpr (WA) store_out<VEC>(p.A + off, st.v[0]);
                store_out<VEC>(p.Bc + off, st.v[1]);
            }
        }
    }
};

// ------------------------------------------------------------ backward
// Reverse time.  Element of step t: (c_t = a_{t+1}, [gA_t,] gBc_t), c = 0 at
// t = T-1; state (C, [mu,] lam).  GA: the loss has a gA term (then A is read
// for da = mu A_{t-1} + lam Bc_{t-1}); without it mu = 0 and A is not read.
// The gradients dx1, dx2 are stored as Tout.
template <typename Tin, typename Tout, int VEC_, int L_, bool GA>
struct MinBwd {
    static constexpr int NS = GA ? 3 : 2, VEC = VEC_, L = L_;
    static constexpr int LAM = NS - 1;   // state index of lam
    static constexpr bool kReverse = true;
    static constexpr unsigned kPrefixStates = (1u << NS) - 2u;   // a prefix's C feeds no output
    // look-back peek: measured faster for bf16 inputs, slower for float32
    static constexpr bool kPeek = MG_MG_PEEK32 != 0 || !std::is_same_v<Tin, float>;
    using S = St<NS, VEC>;
    struct Args {
        const Tin *x1;
        const Tin *x2;
        const float *A;     // read only when GA
        const float *Bc;
        const float *gA;    // read only when GA
        const float *gBc;
        Tout *dx1;
        Tout *dx2;
    };
    struct Regs {
        Raw<Tin, VEC> x1[L + 1];  // rows t0 .. t0+L (x1_{t+1} gives the coefficient of step t)
        float gA[GA ? L : 1][VEC];
        float gB[L][VEC];
        int nr;                   // rows t0 .. t0+nr-1 exist (nr <= L + 1)
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        const int64_t rem = g.T - t0;
        r.nr = act ? int(rem < 0 ? 0 : (rem > L + 1 ? L + 1 : rem)) : 0;
#pragma unroll
        for (int i = 0; i <= L; ++i) {
            const int64_t off = (bb * g.T + t0 + i) * g.D + d;
            if (i < r.nr) {
                r.x1[i].load(p.x1 + off);
            } else {
                // row T (the step after the last): x1 = +inf, a = 0, which ends
                // the adjoint recurrence; later rows: x1 = -inf, a = 1, whose
                // steps (zero gradients) are the identity
                r.x1[i].fill(act && t0 + i == g.T ? INFINITY : -INFINITY);
            }
            if (i < L) {
                if (i < r.nr) {
                    if constexpr (GA) load_vec<VEC>(p.gA + off, r.gA[i]);
                    load_vec<VEC>(p.gBc + off, r.gB[i]);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        if constexpr (GA) r.gA[i][v] = 0.f;
                        r.gB[i][v] = 0.f;
                    }
                }
            }
        }
    }
    // coefficient of step t0+i: a_{t+1} (0 at t = T-1 and 1 past T, from the
    // padding rows of load)
    __device__ static float coef(const Regs &r, int i, int v) { return gate_a(r.x1[i + 1][v]); }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = coef(r, i, v);
            if constexpr (GA) e.v[1][v] = r.gA[i][v];
            e.v[LAM][v] = r.gB[i][v];
        }
        return e;
    }
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = 1.f;
#pragma unroll
            for (int q = 1; q < NS; ++q) e.v[q][v] = 0.f;
        }
        return e;
    }
    __device__ static S initial(const Args &, const ChanGeom &, int64_t, int, bool)
    {
        return identity();
    }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            o.v[0][v] = y.v[0][v] * x.v[0][v];
#pragma unroll
            for (int q = 1; q < NS; ++q) o.v[q][v] = fmaf(y.v[0][v], x.v[q][v], y.v[q][v]);
        }
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        // this round's x2 rows and the forward outputs of the step before each
        // (A_0 = 1, Bc_0 = 0), all issued before any arithmetic
        Raw<Tin, VEC> x2[L];
        float Ap[GA ? L : 1][VEC], Bp[L][VEC];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            const int64_t off = (bb * g.T + t) * g.D + d;
            if (i < r.nr && i < L) {
                x2[i].load(p.x2 + off);
            } else {
                x2[i].fill(0.f);
            }
            if (i < r.nr && t > 0) {
                if constexpr (GA) load_vec<VEC>(p.A + off - g.D, Ap[i]);
                load_vec<VEC>(p.Bc + off - g.D, Bp[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    if constexpr (GA) Ap[i][v] = 1.f;
                    Bp[i][v] = 0.f;
                }
            }
        }
        float mu[VEC], lam[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            mu[v] = GA ? st.v[GA ? 1 : 0][v] : 0.f;
            lam[v] = st.v[LAM][v];
        }
#pragma unroll
        for (int i = L - 1; i >= 0; --i) {
            if (i < r.nr) {
                float o1[VEC], o2[VEC];
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float c = coef(r, i, v);
                    if constexpr (GA) mu[v] = fmaf(c, mu[v], r.gA[i][v]);
                    lam[v] = fmaf(c, lam[v], r.gB[i][v]);
                    const float da = GA ? fmaf(mu[v], Ap[GA ? i : 0][v], lam[v] * Bp[i][v])
                                        : lam[v] * Bp[i][v];
                    const Gate q = gate(r.x1[i][v], x2[i][v]);
                    const float zz = q.z * q.a;                  // z (1 - z)
                    o1[v] = fmaf(lam[v], q.g, -da) * zz;
                    o2[v] = lam[v] * q.z * q.gp;
                }
                const int64_t off = (bb * g.T + t0 + i) * g.D + d;
                store_out<VEC>(p.dx1 + off, o1);
                store_out<VEC>(p.dx2 + off, o2);
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            if constexpr (GA) st.v[1][v] = mu[v];
            st.v[LAM][v] = lam[v];
        }
    }
};

// Tiles (as the bf16 linear scans; overridable at build time).
#ifndef MG_MGF_TX
#define MG_MGF_TX 32
#endif
#ifndef MG_MGF_TY
#define MG_MGF_TY 8
#endif
#ifndef MG_MGF_L
#define MG_MGF_L 4
#endif
#ifndef MG_MGF_MB
#define MG_MGF_MB 3
#endif
#ifndef MG_MGF_R
#define MG_MGF_R 2
#endif
#ifndef MG_MGB_TX
#define MG_MGB_TX 32
#endif
#ifndef MG_MGB_TY
#define MG_MGB_TY 4
#endif
#ifndef MG_MGB_L
#define MG_MGB_L 4
#endif
#ifndef MG_MGB_MB
#define MG_MGB_MB 6
#endif
#ifndef MG_MGB_R
#define MG_MGB_R 4
#endif
constexpr int kSTX = 32, kSTY = 8;

template <typename Tin, bool WA>
using MgFwd = ChanPlan<MinFwd<Tin, 4, MG_MGF_L, WA>, MG_MGF_TX, MG_MGF_TY, MG_MGF_MB, MG_MGF_R>;
template <typename Tin, bool WA>
using MgFwdS = ChanPlan<MinFwd<Tin, 1, 8, WA>, kSTX, kSTY>;
// float32 inputs (8 bytes of x per element against bf16's 4) measured fastest
// on shorter tiles
#ifndef MG_MGB32_TY
#define MG_MGB32_TY 4
#endif
#ifndef MG_MGB32_MB
#define MG_MGB32_MB 3
#endif
#ifndef MG_MGB32_R
#define MG_MGB32_R 4
#endif
template <typename Tin, typename Tout, bool GA>
using MgBwd = std::conditional_t<
    std::is_same_v<Tin, float>,
    ChanPlan<MinBwd<Tin, Tout, 4, MG_MGB_L, GA>, MG_MGB_TX, MG_MGB32_TY, MG_MGB32_MB, MG_MGB32_R>,
    ChanPlan<MinBwd<Tin, Tout, 4, MG_MGB_L, GA>, MG_MGB_TX, MG_MGB_TY, MG_MGB_MB, MG_MGB_R>>;
template <typename Tin, typename Tout, bool GA>
using MgBwdS = ChanPlan<MinBwd<Tin, Tout, 1, 4, GA>, kSTX, kSTY>;

template <typename Tin, bool WA>
mg_status fwd_t(const void *x1, const void *x2, float *A, float *Bc, int64_t B, int64_t T,
                int64_t D, void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_mingru_scan_fwd";
    using P = const Tin *;
    if (D % 4 == 0) return MgFwd<Tin, WA>::launch({P(x1), P(x2), A, Bc}, B, T, D, ws, wsb, s, o, nm);
    return MgFwdS<Tin, WA>::launch({P(x1), P(x2), A, Bc}, B, T, D, ws, wsb, s, o, nm);
}

template <typename Tin, typename Tout, bool GA>
mg_status bwd_t(const void *x1, const void *x2, const float *A, const float *Bc, const float *gA,
                const float *gBc, void *dx1, void *dx2, int64_t B, int64_t T, int64_t D, void *ws,
                size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_mingru_scan_bwd";
    using P = const Tin *;
    using Q = Tout *;
    if (D % 4 == 0)
        return MgBwd<Tin, Tout, GA>::launch({P(x1), P(x2), A, Bc, gA, gBc, Q(dx1), Q(dx2)}, B, T,
                                            D, ws, wsb, s, o, nm);
    return MgBwdS<Tin, Tout, GA>::launch({P(x1), P(x2), A, Bc, gA, gBc, Q(dx1), Q(dx2)}, B, T, D,
                                         ws, wsb, s, o, nm);
}

}  // namespace

size_t mingru_ws_bytes(int64_t B, int64_t T, int64_t D)
{
    size_t m = 0;
    auto up = [&](size_t x) { m = x > m ? x : m; };
    if (D % 4 == 0) {
        up(MgFwd<float, true>::ws_bytes(B, T, D));
        up(MgBwd<float, float, true>::ws_bytes(B, T, D));
        up(MgFwd<bf16_t, true>::ws_bytes(B, T, D));
        up(MgBwd<bf16_t, float, true>::ws_bytes(B, T, D));
    } else {
        up(MgFwdS<float, true>::ws_bytes(B, T, D));
        up(MgBwdS<float, float, true>::ws_bytes(B, T, D));
    }
    return m;
}

mg_status launch_mingru_fwd(const void *x1, const void *x2, mg_dtype dt, float *A, float *Bc,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t wsb, cudaStream_t s,
                            const LaunchOpts &o)
{
    if (dt == MG_F32)
        return A ? fwd_t<float, true>(x1, x2, A, Bc, B, T, D, ws, wsb, s, o)
                 : fwd_t<float, false>(x1, x2, A, Bc, B, T, D, ws, wsb, s, o);
    return A ? fwd_t<bf16_t, true>(x1, x2, A, Bc, B, T, D, ws, wsb, s, o)
             : fwd_t<bf16_t, false>(x1, x2, A, Bc, B, T, D, ws, wsb, s, o);
}

mg_status launch_mingru_bwd(const void *x1, const void *x2, mg_dtype dt, const float *A,
                            const float *Bc, const float *gA, const float *gBc, void *dx1,
                            void *dx2, mg_dtype grad_dt, int64_t B, int64_t T, int64_t D, void *ws,
                            size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const bool ga = gA != nullptr;
#define MG_MBWD(TIN, TOUT)                                                                     \
    return ga ? bwd_t<TIN, TOUT, true>(x1, x2, A, Bc, gA, gBc, dx1, dx2, B, T, D, ws, wsb, s, o) \
              : bwd_t<TIN, TOUT, false>(x1, x2, A, Bc, gA, gBc, dx1, dx2, B, T, D, ws, wsb, s, o)
    if (dt == MG_F32) {
        if (grad_dt == MG_F32) MG_MBWD(float, float);
        MG_MBWD(float, bf16_t);
    }
    if (grad_dt == MG_F32) MG_MBWD(bf16_t, float);
    MG_MBWD(bf16_t, bf16_t);
#undef MG_MBWD
}

}  // namespace mg

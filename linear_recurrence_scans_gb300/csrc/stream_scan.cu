// The channel-wise ops on the persistent warp-specialised engine
// (stream_engine.cuh): linear_scan_fwd, linear_scan_bwd and
// parallel_scan_log_fwd of the page "minGRU - Triton kernels", for D a
// multiple of the 16-byte vector width (the other sizes take the
// one-channel-per-lane path of channel_scan.cu).
#include <cmath>

#include "stream_engine.cuh"

namespace mg {
namespace {


// ----------------------------------------------------------- linear forward
// Staged: 0 = a (row t), 1 = b (row t).  State (running product, h).
template <typename Tin, int VEC_, int NCW_, int L_, int NLB_, int SG_>
struct LinFwdT {
    static constexpr int NS = 2, VEC = VEC_, NCW = NCW_, L = L_, NARR = 2;
    static constexpr int NLB = NLB_, STAGES = SG_;
    static constexpr bool kReverse = false;
    using S = St<NS, VEC>;
    static constexpr int elt(int) { return int(sizeof(Tin)); }
    static constexpr int shift(int) { return 0; }
    struct Args {
        Staged src[NARR];
        float *A;
        float *Bc;
    };
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
    __device__ static S initial(const Args &, const ChanGeom &, int64_t, int, bool) { return identity(); }
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
    __device__ static S elem(const char *st, int i, int lane, int64_t t, const ChanGeom &g)
    {
        if (t >= g.T) return identity();
        S e;
        load_vec<VEC>(srow<LinFwdT, Tin>(st, 0, i, lane), e.v[0]);
        load_vec<VEC>(srow<LinFwdT, Tin>(st, 1, i, lane), e.v[1]);
        return e;
    }
    __device__ static void step2(const Args &p, const char *st, int i, int lane, int64_t t,
                                 const ChanGeom &g, int64_t bb, int d, bool act, S &state)
    {
        if (t >= g.T) return;
        float a[VEC], b[VEC];
        load_vec<VEC>(srow<LinFwdT, Tin>(st, 0, i, lane), a);
        load_vec<VEC>(srow<LinFwdT, Tin>(st, 1, i, lane), b);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            state.v[0][v] = a[v] * state.v[0][v];
            state.v[1][v] = fmaf(a[v], state.v[1][v], b[v]);
        }
        if (act) {
            const int64_t off = (bb * g.T + t) * g.D + d;
            store_vec<VEC>(p.A + off, state.v[0]);
            store_vec<VEC>(p.Bc + off, state.v[1]);
        }
    }
};

// ---------------------------------------------------------- linear backward
// Reverse time.  Staged: 0 = a (row t+1), 1 = gA (t), 2 = gBc (t),
// 3 = A (t-1), 4 = Bc (t-1).  State (C, mu, lam).
template <typename Tin, int NCW_, int L_, int NLB_, int SG_>
struct LinBwdT {
    static constexpr int NS = 3, VEC = 4, NCW = NCW_, L = L_, NARR = 5;
    static constexpr int NLB = NLB_, STAGES = SG_;
    static constexpr bool kReverse = true;
    using S = St<NS, VEC>;
    static constexpr int elt(int a) { return a == 0 ? int(sizeof(Tin)) : 4; }
    static constexpr int shift(int a) { return a == 0 ? 1 : (a >= 3 ? -1 : 0); }
    struct Args {
        Staged src[NARR];
        float *da;
        float *db;
    };
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = 1.f;
            e.v[1][v] = 0.f;
            e.v[2][v] = 0.f;
        }
        return e;
    }
    __device__ static S initial(const Args &, const ChanGeom &, int64_t, int, bool) { return identity(); }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            o.v[0][v] = y.v[0][v] * x.v[0][v];
            o.v[1][v] = fmaf(y.v[0][v], x.v[1][v], y.v[1][v]);
            o.v[2][v] = fmaf(y.v[0][v], x.v[2][v], y.v[2][v]);
        }
        return o;
    }
    __device__ static void coef(const char *st, int i, int lane, int64_t t, const ChanGeom &g,
                                float (&c)[VEC])
    {
        if (t + 1 < g.T) {
            load_vec<VEC>(srow<LinBwdT, Tin>(st, 0, i, lane), c);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) c[v] = 0.f;
        }
    }
    __device__ static S elem(const char *st, int i, int lane, int64_t t, const ChanGeom &g)
    {
        if (t >= g.T) return identity();
        S e;
        coef(st, i, lane, t, g, e.v[0]);
        load_vec<VEC>(srow<LinBwdT, float>(st, 1, i, lane), e.v[1]);
        load_vec<VEC>(srow<LinBwdT, float>(st, 2, i, lane), e.v[2]);
        return e;
    }
    __device__ static void step2(const Args &p, const char *st, int i, int lane, int64_t t,
                                 const ChanGeom &g, int64_t bb, int d, bool act, S &state)
    {
        if (t >= g.T) return;
        float c[VEC], gA[VEC], gB[VEC], Ap[VEC], Bp[VEC], da[VEC];
        coef(st, i, lane, t, g, c);
        load_vec<VEC>(srow<LinBwdT, float>(st, 1, i, lane), gA);
        load_vec<VEC>(srow<LinBwdT, float>(st, 2, i, lane), gB);
        if (t > 0) {
            load_vec<VEC>(srow<LinBwdT, float>(st, 3, i, lane), Ap);
            load_vec<VEC>(srow<LinBwdT, float>(st, 4, i, lane), Bp);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                Ap[v] = 1.f;
                Bp[v] = 0.f;
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            state.v[1][v] = fmaf(c[v], state.v[1][v], gA[v]);
            state.v[2][v] = fmaf(c[v], state.v[2][v], gB[v]);
            da[v] = fmaf(state.v[1][v], Ap[v], state.v[2][v] * Bp[v]);
        }
        if (act) {
            const int64_t off = (bb * g.T + t) * g.D + d;
            store_vec<VEC>(p.da + off, da);
            store_vec<VEC>(p.db + off, state.v[2]);
        }
    }
};

// ------------------------------------------------------- log-space forward
// Staged: 0 = log_coeffs (row t), 1 = log_values (row t+1 of T+1).  State
// (la, m, s) in natural logs, value = s * e^m.
template <int NCW_, int L_, int NLB_, int SG_>
struct LogFwdT {
    static constexpr int NS = 3, VEC = 4, NCW = NCW_, L = L_, NARR = 2;
    static constexpr int NLB = NLB_, STAGES = SG_;
    static constexpr bool kReverse = false;
    using S = St<NS, VEC>;
    static constexpr int elt(int) { return 4; }
    static constexpr int shift(int a) { return a; }
    struct Args {
        Staged src[NARR];
        float *h;
    };
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = 0.f;
            e.v[1][v] = -INFINITY;
            e.v[2][v] = 0.f;
        }
        return e;
    }
    __device__ static S initial(const Args &p, const ChanGeom &g, int64_t bb, int d, bool act)
    {
        S e = identity();
        if (act) {
            float l0[VEC];
            load_vec<VEC>(reinterpret_cast<const float *>(p.src[1].base) + (bb * (g.T + 1)) * g.D + d, l0);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                e.v[1][v] = l0[v];
                e.v[2][v] = 1.f;
            }
        }
        return e;
    }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            o.v[0][v] = x.v[0][v] + y.v[0][v];
            log_add(y.v[0][v] + x.v[1][v], x.v[2][v], y.v[1][v], y.v[2][v], o.v[1][v], o.v[2][v]);
        }
        return o;
    }
    __device__ static S elem(const char *st, int i, int lane, int64_t t, const ChanGeom &g)
    {
        if (t >= g.T) {
            S e;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                e.v[0][v] = 0.f;
                e.v[1][v] = -INFINITY;
                e.v[2][v] = 1.f;
            }
            return e;
        }
        S e;
        load_vec<VEC>(srow<LogFwdT, float>(st, 0, i, lane), e.v[0]);
        load_vec<VEC>(srow<LogFwdT, float>(st, 1, i, lane), e.v[1]);
#pragma unroll
        for (int v = 0; v < VEC; ++v) e.v[2][v] = 1.f;
        return e;
    }
    __device__ static void step2(const Args &p, const char *st, int i, int lane, int64_t t,
                                 const ChanGeom &g, int64_t bb, int d, bool act, S &state)
    {
        if (t >= g.T) return;
        float lc[VEC], lv[VEC], h[VEC];
        load_vec<VEC>(srow<LogFwdT, float>(st, 0, i, lane), lc);
        load_vec<VEC>(srow<LogFwdT, float>(st, 1, i, lane), lv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            log_add(lc[v] + state.v[1][v], state.v[2][v], lv[v], 1.f, state.v[1][v], state.v[2][v]);
            h[v] = state.v[2][v] * ex2_sub(state.v[1][v] * kLog2eF);
        }
        if (act) store_vec<VEC>(p.h + (bb * g.T + t) * g.D + d, h);
    }
};

// Tiles: NCW compute warps x L steps per warp, NLB concurrent look-backs per
// SM, a ring of SG staged tiles (SG - NLB - 1 of them loading ahead), sized
// to fit one SM's shared memory.
#ifndef MG_SF_NCW
#define MG_SF_NCW 4
#endif
#ifndef MG_SF_L
#define MG_SF_L 4
#endif
#ifndef MG_SF_NLB
#define MG_SF_NLB 3
#endif
#ifndef MG_SF_SG
#define MG_SF_SG 9
#endif
#ifndef MG_SF16_SG
#define MG_SF16_SG 7
#endif
#ifndef MG_SB_NCW
#define MG_SB_NCW 4
#endif
#ifndef MG_SB_L
#define MG_SB_L 2
#endif
#ifndef MG_SB_NLB
#define MG_SB_NLB 3
#endif
#ifndef MG_SB_SG
#define MG_SB_SG 7
#endif
#ifndef MG_SL_NCW
#define MG_SL_NCW 4
#endif
#ifndef MG_SL_L
#define MG_SL_L 4
#endif
#ifndef MG_SL_NLB
#define MG_SL_NLB 3
#endif
#ifndef MG_SL_SG
#define MG_SL_SG 8
#endif
using SFwdF32 = StreamPlan<LinFwdT<float, 4, MG_SF_NCW, MG_SF_L, MG_SF_NLB, MG_SF_SG>>;
using SFwdB16 = StreamPlan<LinFwdT<bf16_t, 8, MG_SF_NCW, MG_SF_L, MG_SF_NLB, MG_SF16_SG>>;
using SBwdF32 = StreamPlan<LinBwdT<float, MG_SB_NCW, MG_SB_L, MG_SB_NLB, MG_SB_SG>>;
using SBwdB16 = StreamPlan<LinBwdT<bf16_t, MG_SB_NCW, MG_SB_L, MG_SB_NLB, MG_SB_SG>>;
using SLog = StreamPlan<LogFwdT<MG_SL_NCW, MG_SL_L, MG_SL_NLB, MG_SL_SG>>;

Staged staged(const void *p, int64_t rows) { return Staged{static_cast<const char *>(p), rows}; }

}  // namespace

bool stream_linear_ok(mg_dtype dt, int64_t D) { return dt == MG_F32 ? D % 4 == 0 : D % 8 == 0; }
bool stream_log_ok(int64_t D) { return D % 4 == 0; }

size_t stream_linear_fwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    return dt == MG_F32 ? SFwdF32::ws_bytes(B, T, D) : SFwdB16::ws_bytes(B, T, D);
}

size_t stream_linear_bwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    return dt == MG_F32 ? SBwdF32::ws_bytes(B, T, D) : SBwdB16::ws_bytes(B, T, D);
}

size_t stream_log_ws_bytes(int64_t B, int64_t T, int64_t D) { return SLog::ws_bytes(B, T, D); }

mg_status stream_linear_fwd(const void *a, const void *b, mg_dtype dt, float *A, float *Bc,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t wsb, cudaStream_t s,
                            const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_fwd";
    if (dt == MG_F32)
        return SFwdF32::launch({{staged(a, T), staged(b, T)}, A, Bc}, B, T, D, ws, wsb, s, o, nm);
    return SFwdB16::launch({{staged(a, T), staged(b, T)}, A, Bc}, B, T, D, ws, wsb, s, o, nm);
}

mg_status stream_linear_bwd(const void *a, mg_dtype dt, const float *A, const float *Bc,
                            const float *gA, const float *gBc, float *da, float *db, int64_t B,
                            int64_t T, int64_t D, void *ws, size_t wsb, cudaStream_t s,
                            const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_bwd";
    const Staged src[5] = {staged(a, T), staged(gA, T), staged(gBc, T), staged(A, T), staged(Bc, T)};
    if (dt == MG_F32)
        return SBwdF32::launch({{src[0], src[1], src[2], src[3], src[4]}, da, db}, B, T, D, ws, wsb,
                               s, o, nm);
    return SBwdB16::launch({{src[0], src[1], src[2], src[3], src[4]}, da, db}, B, T, D, ws, wsb, s,
                           o, nm);
}

mg_status stream_log_fwd(const float *lc, const float *lv, float *h, int64_t B, int64_t T,
                         int64_t D, void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    return SLog::launch({{staged(lc, T), staged(lv, T + 1)}, h}, B, T, D, ws, wsb, s, o,
                        "mg_log_scan_fwd");
}

}  // namespace mg

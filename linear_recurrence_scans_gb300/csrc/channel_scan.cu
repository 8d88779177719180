// Channel-wise chunked scans on (B,T,D): linear_scan_fwd, linear_scan_bwd and
// parallel_scan_log_fwd of the page "minGRU - Triton kernels", and the
// adjoint of the log-space scan.
//
// All of them evaluate the same associative pair operator
//     (a1, b1) o (a2, b2) = (a2 a1, a2 b1 + b2)        (element 1 earlier)
// over time, independently for every channel (b, d), in one kernel shape
// (scan_engine.cuh):
//
//   * a CTA owns a tile of DC = TX*VEC channels by TY*L*R time steps, taken
//     by ticket (chunk-major, so predecessors have always started);
//   * each thread loads VEC channels (one 16-byte vector) for L consecutive
//     steps at a time straight into registers -- a warp row reads up to
//     32 x 16 contiguous bytes, fully coalesced -- and folds its R rounds of
//     L steps into its aggregate;
//   * the TY thread aggregates of a channel are folded through shared memory,
//     leaving each row its exclusive prefix within the tile;
//   * warp 0 finds the chunk's carry-in by decoupled look-back over the
//     previous chunks of the same channel tile (lookback.cuh);
//   * every thread composes carry o (its row's prefix) and re-runs its steps
//     from that state, re-reading them (now from L2) and writing the outputs,
//     so each input is read from HBM once and each output written once.
//
// The backward ops are the same engine run in reverse time on the adjoint
// recurrences; the log op carries log-space values as (m, s) with
// value = s * e^m so that one exp2 per combine suffices.
#include <cmath>

#include "scan_engine.cuh"

namespace mg {
namespace {

// ----------------------------------------------------------- linear forward
// Element of step t: (a_t, b_t).  State: (running product, h).  H0: the
// recurrence starts from h0[b, d] (a (B, D) float32 array) instead of 0; the
// state before step 1 is then (1, h0), and the second output is H_t.
template <typename Tin, int VEC_, int L_, bool H0 = false>
struct LinFwd {
    static constexpr int NS = 2, VEC = VEC_, L = L_;
    static constexpr bool kReverse = false;
    using S = St<NS, VEC>;
    struct Args {
        const Tin *a;
        const Tin *b;
        float *A;
        float *Bc;
        const float *h0;   // read only when H0
    };
    struct Regs {
        Raw<Tin, VEC> a[L];
        Raw<Tin, VEC> b[L];
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                r.a[i].load(p.a + off);
                r.b[i].load(p.b + off);
            } else {
                r.a[i].fill(1.f);
                r.b[i].fill(0.f);
            }
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = r.a[i][v];
            e.v[1][v] = r.b[i][v];
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
    __device__ static S initial(const Args &p, const ChanGeom &g, int64_t bb, int d, bool act)
    {
        S e = identity();
        if constexpr (H0) {
            if (act) load_vec<VEC>(p.h0 + bb * g.D + d, e.v[1]);
        }
        return e;
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
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        float P[VEC], H[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            P[v] = st.v[0][v];
            H[v] = st.v[1][v];
        }
#pragma unroll
        for (int i = 0; i < L; ++i) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                P[v] = r.a[i][v] * P[v];
                H[v] = fmaf(r.a[i][v], H[v], r.b[i][v]);
            }
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                store_out<VEC>(p.A + off, P);
                store_out<VEC>(p.Bc + off, H);
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            st.v[0][v] = P[v];
            st.v[1][v] = H[v];
        }
    }
};

// ---------------------------------------------------------- linear backward
// Reverse time.  Element of step t: (c_t = a_{t+1}, gA_t, gBc_t) with
// c_{T} = 0; state (C, mu, lam): mu_t = gA_t + c_t mu_{t+1}, same for lam.
// The gradients are stored as Tout (float32, or bf16 rounded to nearest).
// H0: the forward started from h0[b, d] (so H_0 = h0 in da_1), and
// dh0 = a_1 lam_1 is written to dh0[b, d] (both (B, D) float32).
template <typename Tin, int VEC_, int L_, typename Tout = float, bool H0 = false>
struct LinBwd {
    static constexpr int NS = 3, VEC = VEC_, L = L_;
    static constexpr bool kReverse = true;
    static constexpr unsigned kPrefixStates = 0b110u;   // a prefix's C feeds no output
    using S = St<NS, VEC>;
    struct Args {
        const Tin *a;
        const float *A;
        const float *Bc;
        const float *gA;
        const float *gBc;
        Tout *da;
        Tout *db;
        const float *h0;   // read only when H0
        float *dh0;        // written only when H0
    };
    struct Regs {
        Raw<Tin, VEC> c[L];
        float gA[L][VEC];
        float gB[L][VEC];
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                load_vec<VEC>(p.gA + off, r.gA[i]);
                load_vec<VEC>(p.gBc + off, r.gB[i]);
                if (t + 1 < g.T) {
                    r.c[i].load(p.a + off + g.D);
                } else {
                    r.c[i].fill(0.f);
                }
            } else {
                r.c[i].fill(1.f);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    r.gA[i][v] = 0.f;
                    r.gB[i][v] = 0.f;
                }
            }
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = r.c[i][v];
            e.v[1][v] = r.gA[i][v];
            e.v[2][v] = r.gB[i][v];
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
            e.v[2][v] = 0.f;
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
            o.v[2][v] = fmaf(y.v[0][v], x.v[2][v], y.v[2][v]);
        }
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        // A_{t-1}, Bc_{t-1} for the L steps (A_0 = 1, Bc_0 = 0 before the first step).
        float Ap[L][VEC], Bp[L][VEC];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T && t > 0) {
                const int64_t off = (bb * g.T + t - 1) * g.D + d;
                load_vec<VEC>(p.A + off, Ap[i]);
                load_vec<VEC>(p.Bc + off, Bp[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    Ap[i][v] = 1.f;
                    Bp[i][v] = 0.f;
                }
                if constexpr (H0) {
                    if (act && t == 0) load_vec<VEC>(p.h0 + bb * g.D + d, Bp[i]);
                }
            }
        }
        float mu[VEC], lam[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            mu[v] = st.v[1][v];
            lam[v] = st.v[2][v];
        }
#pragma unroll
        for (int i = L - 1; i >= 0; --i) {
            float da[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                mu[v] = fmaf(r.c[i][v], mu[v], r.gA[i][v]);
                lam[v] = fmaf(r.c[i][v], lam[v], r.gB[i][v]);
                da[v] = fmaf(mu[v], Ap[i][v], lam[v] * Bp[i][v]);
            }
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                store_out<VEC>(p.da + off, da);
                store_out<VEC>(p.db + off, lam);
                if constexpr (H0) {
                    if (t == 0) {  // dh0 = a_1 lam_1
                        Raw<Tin, VEC> a0;
                        a0.load(p.a + off);
                        float dh[VEC];
#pragma unroll
                        for (int v = 0; v < VEC; ++v) dh[v] = a0[v] * lam[v];
                        store_out<VEC>(p.dh0 + bb * g.D + d, dh);
                    }
                }
            }
        }
        // (the running coefficient product is not needed past the outputs)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            st.v[1][v] = mu[v];
            st.v[2][v] = lam[v];
        }
    }
};

// ------------------------------------------------------- log-space forward
// Element of step t: (lc_t, lv_t) in natural logs.  State (la, m, s): la =
// sum of log-coefficients, the log value being m + log(s).  Combine (x
// earlier): la = x.la + y.la and the value log(e^(y.la + LB_x) + e^(LB_y)),
// one log_add (one exp2) per combine.
template <int VEC_, int L_>
struct LogFwd {
    static constexpr int NS = 3, VEC = VEC_, L = L_;
    static constexpr bool kReverse = false;
    static constexpr unsigned kPrefixStates = 0b110u;   // a prefix's la feeds no output
    using S = St<NS, VEC>;
    struct Args {
        const float *lc;
        const float *lv;
        float *h;
    };
    struct Regs {
        float lc[L][VEC];
        float lv[L][VEC];
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                load_vec<VEC>(p.lc + (bb * g.T + t) * g.D + d, r.lc[i]);
                load_vec<VEC>(p.lv + (bb * (g.T + 1) + t + 1) * g.D + d, r.lv[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    r.lc[i][v] = 0.f;
                    r.lv[i][v] = -INFINITY;
                }
            }
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = r.lc[i][v];
            e.v[1][v] = r.lv[i][v];
            e.v[2][v] = 1.f;
        }
        return e;
    }
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
    // State before step 1: log h_0 = log_values[b, 0, d].
    __device__ static S initial(const Args &p, const ChanGeom &g, int64_t bb, int d, bool act)
    {
        S e = identity();
        if (act) {
            float l0[VEC];
            load_vec<VEC>(p.lv + (bb * (g.T + 1)) * g.D + d, l0);
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
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        float m[VEC], s[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            m[v] = st.v[1][v];
            s[v] = st.v[2][v];
        }
#pragma unroll
        for (int i = 0; i < L; ++i) {
            float h[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                log_add(r.lc[i][v] + m[v], s[v], r.lv[i][v], 1.f, m[v], s[v]);
                h[v] = s[v] * ex2_sub(m[v] * kLog2eF);
            }
            const int64_t t = t0 + i;
            if (act && t < g.T) store_out<VEC>(p.h + (bb * g.T + t) * g.D + d, h);
        }
        // (the summed log-coefficient is not needed past the outputs)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            st.v[1][v] = m[v];
            st.v[2][v] = s[v];
        }
    }
};

// ------------------------------------------------------ log-space adjoint
// Gradient of the log-space scan for L = sum_t gh_t h_t (the forward's
// recurrence h_t = a_t h_{t-1} + b_t, a_t = exp(lc_t), b_t = exp(lv_t)).
// Reverse time, element of step t: (c_t = a_{t+1}, gh_t) with c_T = 0; state
// (C, mu): mu_t = gh_t + a_{t+1} mu_{t+1}.  Epilogue: dlc_t = mu_t a_t h_{t-1}
// (h_0 = exp(lv_0)), dlv_t = mu_t b_t, and dlv_0 = a_1 mu_1 h_0 = dlc_1.
// A round loads L + 1 rows of lc, so a_t and a_{t+1} share the exponentials.
template <int VEC_, int L_>
struct LogBwd {
    static constexpr int NS = 2, VEC = VEC_, L = L_;
    static constexpr bool kReverse = true;
    static constexpr unsigned kPrefixStates = 0b10u;    // a prefix's C feeds no output
    using S = St<NS, VEC>;
    struct Args {
        const float *lc;
        const float *lv;
        const float *h;
        const float *gh;
        float *dlc;
        float *dlv;
    };
    struct Regs {
        float ea[L + 1][VEC];  // exp(lc) of steps t0 .. t0+L (0 past T)
        float g[L][VEC];
        int nval;              // steps of the round that are < T
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        const int64_t rem = g.T - t0;
        r.nval = act ? int(rem < 0 ? 0 : (rem > L ? L : rem)) : 0;
        // every load of the round is issued before the first exponential
#pragma unroll
        for (int i = 0; i <= L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                load_vec<VEC>(p.lc + (bb * g.T + t) * g.D + d, r.ea[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) r.ea[i][v] = -INFINITY;
            }
            if (i < L) {
                if (act && t < g.T) {
                    load_vec<VEC>(p.gh + (bb * g.T + t) * g.D + d, r.g[i]);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) r.g[i][v] = 0.f;
                }
            }
        }
#pragma unroll
        for (int i = 0; i <= L; ++i)
#pragma unroll
            for (int v = 0; v < VEC; ++v) r.ea[i][v] = ex2_sub(r.ea[i][v] * kLog2eF);
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            e.v[0][v] = i < r.nval ? r.ea[i + 1][v] : 1.f;  // past T: the identity
            e.v[1][v] = r.g[i][v];
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
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        float mu[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) mu[v] = st.v[1][v];
#pragma unroll
        for (int i = L - 1; i >= 0; --i) {
            if (i < r.nval) {
                const int64_t t = t0 + i;
                float hp[VEC], lvv[VEC], dlc[VEC], dlv[VEC];
                if (t > 0) {
                    load_vec<VEC>(p.h + (bb * g.T + t - 1) * g.D + d, hp);
                } else {
                    load_vec<VEC>(p.lv + (bb * (g.T + 1)) * g.D + d, hp);
#pragma unroll
                    for (int v = 0; v < VEC; ++v) hp[v] = ex2_sub(hp[v] * kLog2eF);
                }
                load_vec<VEC>(p.lv + (bb * (g.T + 1) + t + 1) * g.D + d, lvv);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    mu[v] = fmaf(r.ea[i + 1][v], mu[v], r.g[i][v]);
                    dlc[v] = mu[v] * r.ea[i][v] * hp[v];
                    dlv[v] = mu[v] * ex2_sub(lvv[v] * kLog2eF);
                }
                store_out<VEC>(p.dlc + (bb * g.T + t) * g.D + d, dlc);
                store_out<VEC>(p.dlv + (bb * (g.T + 1) + t + 1) * g.D + d, dlv);
                if (t == 0) store_out<VEC>(p.dlv + (bb * (g.T + 1)) * g.D + d, dlc);
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) st.v[1][v] = mu[v];
    }
};

// Tile choices (threads along channels TX, thread rows TY, steps per thread
// and round L, minimum resident CTAs per SM, rounds per thread R).  fp32: 4 channels (16 B) per thread;
// bf16: 8 channels (16 B).  A D that is not a multiple of the vector width
// takes the 1-channel variant.  Each can be overridden at build time.
#ifndef MG_LINF_TX
#define MG_LINF_TX 16
#endif
#ifndef MG_LINF_TY
#define MG_LINF_TY 16
#endif
#ifndef MG_LINF_L
#define MG_LINF_L 8
#endif
#ifndef MG_LINF_MB
#define MG_LINF_MB 1
#endif
#ifndef MG_LINF16_VEC
#define MG_LINF16_VEC 4
#endif
#ifndef MG_LINF16_TX
#define MG_LINF16_TX 32
#endif
#ifndef MG_LINF16_TY
#define MG_LINF16_TY 2
#endif
#ifndef MG_LINF16_L
#define MG_LINF16_L 12
#endif
#ifndef MG_LINF16_MB
#define MG_LINF16_MB 4
#endif
#ifndef MG_LINB_TX
#define MG_LINB_TX 16
#endif
#ifndef MG_LINB_TY
#define MG_LINB_TY 8
#endif
#ifndef MG_LINB_L
#define MG_LINB_L 8
#endif
#ifndef MG_LINB_MB
#define MG_LINB_MB 2
#endif
#ifndef MG_LINB16_TX
#define MG_LINB16_TX 32
#endif
#ifndef MG_LINB16_TY
#define MG_LINB16_TY 4
#endif
#ifndef MG_LINB16_L
#define MG_LINB16_L 4
#endif
#ifndef MG_LINB16_MB
#define MG_LINB16_MB 5
#endif
#ifndef MG_LOG_TX
#define MG_LOG_TX 32
#endif
#ifndef MG_LOG_TY
#define MG_LOG_TY 8
#endif
#ifndef MG_LOG_L
#define MG_LOG_L 4
#endif
#ifndef MG_LOG_MB
#define MG_LOG_MB 4
#endif
#ifndef MG_LINF_R
#define MG_LINF_R 2
#endif
#ifndef MG_LINF16_R
#define MG_LINF16_R 2
#endif
#ifndef MG_LINB_R
#define MG_LINB_R 2
#endif
#ifndef MG_LINB16_R
#define MG_LINB16_R 2
#endif
#ifndef MG_LOG_R
#define MG_LOG_R 2
#endif
#ifndef MG_LOGB_TX
#define MG_LOGB_TX 32
#endif
#ifndef MG_LOGB_TY
#define MG_LOGB_TY 8
#endif
#ifndef MG_LOGB_L
#define MG_LOGB_L 2
#endif
#ifndef MG_LOGB_MB
#define MG_LOGB_MB 4
#endif
#ifndef MG_LOGB_R
#define MG_LOGB_R 3
#endif
constexpr int kTX = 32, kTY = 8;
using LinFwdF32 = ChanPlan<LinFwd<float, 4, MG_LINF_L>, MG_LINF_TX, MG_LINF_TY, MG_LINF_MB, MG_LINF_R>;
using LinFwdF32s = ChanPlan<LinFwd<float, 1, 8>, kTX, kTY>;
using LinFwdB16 = ChanPlan<LinFwd<bf16_t, MG_LINF16_VEC, MG_LINF16_L>, MG_LINF16_TX, MG_LINF16_TY, MG_LINF16_MB, MG_LINF16_R>;
using LinFwdB16s = ChanPlan<LinFwd<bf16_t, 1, 8>, kTX, kTY>;
using LinBwdF32 = ChanPlan<LinBwd<float, 4, MG_LINB_L>, MG_LINB_TX, MG_LINB_TY, MG_LINB_MB, MG_LINB_R>;
using LinBwdF32s = ChanPlan<LinBwd<float, 1, 4>, kTX, kTY>;
using LinBwdB16 = ChanPlan<LinBwd<bf16_t, 4, MG_LINB16_L>, MG_LINB16_TX, MG_LINB16_TY, MG_LINB16_MB, MG_LINB16_R>;
using LinBwdB16s = ChanPlan<LinBwd<bf16_t, 1, 4>, kTX, kTY>;
using LinFwdF32h = ChanPlan<LinFwd<float, 4, MG_LINF_L, true>, MG_LINF_TX, MG_LINF_TY, MG_LINF_MB, MG_LINF_R>;
using LinFwdF32hs = ChanPlan<LinFwd<float, 1, 8, true>, kTX, kTY>;
using LinFwdB16h = ChanPlan<LinFwd<bf16_t, MG_LINF16_VEC, MG_LINF16_L, true>, MG_LINF16_TX, MG_LINF16_TY, MG_LINF16_MB, MG_LINF16_R>;
using LinFwdB16hs = ChanPlan<LinFwd<bf16_t, 1, 8, true>, kTX, kTY>;
using LinBwdF32h = ChanPlan<LinBwd<float, 4, MG_LINB_L, float, true>, MG_LINB_TX, MG_LINB_TY, MG_LINB_MB, MG_LINB_R>;
using LinBwdF32hs = ChanPlan<LinBwd<float, 1, 4, float, true>, kTX, kTY>;
using LinBwdB16h = ChanPlan<LinBwd<bf16_t, 4, MG_LINB16_L, float, true>, MG_LINB16_TX, MG_LINB16_TY, MG_LINB16_MB, MG_LINB16_R>;
using LinBwdB16hs = ChanPlan<LinBwd<bf16_t, 1, 4, float, true>, kTX, kTY>;
using LinBwdB16G = ChanPlan<LinBwd<bf16_t, 4, MG_LINB16_L, bf16_t>, MG_LINB16_TX, MG_LINB16_TY, MG_LINB16_MB, MG_LINB16_R>;
using LinBwdB16Gs = ChanPlan<LinBwd<bf16_t, 1, 4, bf16_t>, kTX, kTY>;
using LinBwdF32G = ChanPlan<LinBwd<float, 4, MG_LINB_L, bf16_t>, MG_LINB_TX, MG_LINB_TY, MG_LINB_MB, MG_LINB_R>;
using LinBwdF32Gs = ChanPlan<LinBwd<float, 1, 4, bf16_t>, kTX, kTY>;
using LogF32 = ChanPlan<LogFwd<4, MG_LOG_L>, MG_LOG_TX, MG_LOG_TY, MG_LOG_MB, MG_LOG_R>;
using LogBwdF32 = ChanPlan<LogBwd<4, MG_LOGB_L>, MG_LOGB_TX, MG_LOGB_TY, MG_LOGB_MB, MG_LOGB_R>;
using LogBwdF32s = ChanPlan<LogBwd<1, 4>, kTX, kTY>;
using LogF32s = ChanPlan<LogFwd<1, 8>, kTX, kTY>;

}  // namespace

size_t linear_fwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    if (dt == MG_F32) return D % 4 == 0 ? LinFwdF32::ws_bytes(B, T, D) : LinFwdF32s::ws_bytes(B, T, D);
    return D % MG_LINF16_VEC == 0 ? LinFwdB16::ws_bytes(B, T, D) : LinFwdB16s::ws_bytes(B, T, D);
}

size_t linear_bwd_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    if (dt == MG_F32) return D % 4 == 0 ? LinBwdF32::ws_bytes(B, T, D) : LinBwdF32s::ws_bytes(B, T, D);
    return D % 4 == 0 ? LinBwdB16::ws_bytes(B, T, D) : LinBwdB16s::ws_bytes(B, T, D);
}

size_t linear_h0_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    size_t f, b;
    if (dt == MG_F32) {
        f = D % 4 == 0 ? LinFwdF32h::ws_bytes(B, T, D) : LinFwdF32hs::ws_bytes(B, T, D);
        b = D % 4 == 0 ? LinBwdF32h::ws_bytes(B, T, D) : LinBwdF32hs::ws_bytes(B, T, D);
    } else {
        f = D % MG_LINF16_VEC == 0 ? LinFwdB16h::ws_bytes(B, T, D) : LinFwdB16hs::ws_bytes(B, T, D);
        b = D % 4 == 0 ? LinBwdB16h::ws_bytes(B, T, D) : LinBwdB16hs::ws_bytes(B, T, D);
    }
    return f > b ? f : b;
}

size_t linear_bwd16_ws_bytes(mg_dtype dt, int64_t B, int64_t T, int64_t D)
{
    if (dt == MG_F32) return D % 4 == 0 ? LinBwdF32G::ws_bytes(B, T, D) : LinBwdF32Gs::ws_bytes(B, T, D);
    return D % 4 == 0 ? LinBwdB16G::ws_bytes(B, T, D) : LinBwdB16Gs::ws_bytes(B, T, D);
}

size_t linear_ws_bytes(int64_t B, int64_t T, int64_t D)
{
    size_t m = 0;
    for (mg_dtype dt : {MG_F32, MG_BF16}) {
        const size_t f = linear_fwd_ws_bytes(dt, B, T, D), b = linear_bwd_ws_bytes(dt, B, T, D);
        const size_t b16 = linear_bwd16_ws_bytes(dt, B, T, D);
        const size_t h = linear_h0_ws_bytes(dt, B, T, D);
        m = f > m ? f : m;
        m = b > m ? b : m;
        m = b16 > m ? b16 : m;
        m = h > m ? h : m;
    }
    return m;
}

size_t log_ws_bytes(int64_t B, int64_t T, int64_t D)
{
    const size_t f = D % 4 == 0 ? LogF32::ws_bytes(B, T, D) : LogF32s::ws_bytes(B, T, D);
    const size_t b = D % 4 == 0 ? LogBwdF32::ws_bytes(B, T, D) : LogBwdF32s::ws_bytes(B, T, D);
    return f > b ? f : b;
}

mg_status launch_linear_fwd(const void *a, const void *b, mg_dtype dt, float *A, float *Bc,
                            int64_t B, int64_t T, int64_t D, void *ws, size_t wsb, cudaStream_t s,
                            const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_fwd";
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return LinFwdF32::launch({F(a), F(b), A, Bc}, B, T, D, ws, wsb, s, o, nm);
        return LinFwdF32s::launch({F(a), F(b), A, Bc}, B, T, D, ws, wsb, s, o, nm);
    }
    using H = const bf16_t *;
    if (D % MG_LINF16_VEC == 0) return LinFwdB16::launch({H(a), H(b), A, Bc}, B, T, D, ws, wsb, s, o, nm);
    return LinFwdB16s::launch({H(a), H(b), A, Bc}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_linear_bwd(const void *a, mg_dtype dt, const float *A, const float *Bc,
                            const float *gA, const float *gBc, float *da, float *db, int64_t B,
                            int64_t T, int64_t D, void *ws, size_t wsb, cudaStream_t s,
                            const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_bwd";
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return LinBwdF32::launch({F(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
        return LinBwdF32s::launch({F(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
    }
    using H = const bf16_t *;
    if (D % 4 == 0)
        return LinBwdB16::launch({H(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
    return LinBwdB16s::launch({H(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_linear_h0_fwd(const void *a, const void *b, mg_dtype dt, const float *h0,
                               float *A, float *H, int64_t B, int64_t T, int64_t D, void *ws,
                               size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_h0_fwd";
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0) return LinFwdF32h::launch({F(a), F(b), A, H, h0}, B, T, D, ws, wsb, s, o, nm);
        return LinFwdF32hs::launch({F(a), F(b), A, H, h0}, B, T, D, ws, wsb, s, o, nm);
    }
    using P = const bf16_t *;
    if (D % MG_LINF16_VEC == 0)
        return LinFwdB16h::launch({P(a), P(b), A, H, h0}, B, T, D, ws, wsb, s, o, nm);
    return LinFwdB16hs::launch({P(a), P(b), A, H, h0}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_linear_h0_bwd(const void *a, mg_dtype dt, const float *h0, const float *A,
                               const float *H, const float *gA, const float *gH, float *da,
                               float *db, float *dh0, int64_t B, int64_t T, int64_t D, void *ws,
                               size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_h0_bwd";
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return LinBwdF32h::launch({F(a), A, H, gA, gH, da, db, h0, dh0}, B, T, D, ws, wsb, s, o, nm);
        return LinBwdF32hs::launch({F(a), A, H, gA, gH, da, db, h0, dh0}, B, T, D, ws, wsb, s, o, nm);
    }
    using P = const bf16_t *;
    if (D % 4 == 0)
        return LinBwdB16h::launch({P(a), A, H, gA, gH, da, db, h0, dh0}, B, T, D, ws, wsb, s, o, nm);
    return LinBwdB16hs::launch({P(a), A, H, gA, gH, da, db, h0, dh0}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_linear_bwd_bf16_grads(const void *a, mg_dtype dt, const float *A, const float *Bc,
                                       const float *gA, const float *gBc, bf16_t *da, bf16_t *db,
                                       int64_t B, int64_t T, int64_t D, void *ws, size_t wsb,
                                       cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_bwd_bf16_grads";
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return LinBwdF32G::launch({F(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
        return LinBwdF32Gs::launch({F(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
    }
    using H = const bf16_t *;
    if (D % 4 == 0)
        return LinBwdB16G::launch({H(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
    return LinBwdB16Gs::launch({H(a), A, Bc, gA, gBc, da, db}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_log_bwd(const float *lc, const float *lv, const float *h, const float *gh,
                         float *dlc, float *dlv, int64_t B, int64_t T, int64_t D, void *ws,
                         size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_log_scan_bwd";
    if (D % 4 == 0) return LogBwdF32::launch({lc, lv, h, gh, dlc, dlv}, B, T, D, ws, wsb, s, o, nm);
    return LogBwdF32s::launch({lc, lv, h, gh, dlc, dlv}, B, T, D, ws, wsb, s, o, nm);
}

mg_status launch_log_fwd(const float *lc, const float *lv, float *h, int64_t B, int64_t T,
                         int64_t D, void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_log_scan_fwd";
    if (D % 4 == 0) return LogF32::launch({lc, lv, h}, B, T, D, ws, wsb, s, o, nm);
    return LogF32s::launch({lc, lv, h}, B, T, D, ws, wsb, s, o, nm);
}

}  // namespace mg

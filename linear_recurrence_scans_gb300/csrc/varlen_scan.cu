// The linear scan over a packed batch of variable-length sequences, each from
// its own start state (forward and gradients).
//
// Sequences s = 0 .. nseq-1 lie back to back in one (Ttot, D) tensor, rows
// cu[s] .. cu[s+1]-1 (cu_seqlens, int64, cu[0] = 0, cu[nseq] = Ttot; empty
// sequences allowed).  Within a sequence the recurrence is linear_scan_fwd's
// (page "minGRU - Triton kernels"), started from h0[s] (or 0) the way slot 0
// of parallel_scan_log_fwd's log_values starts that op:
//   A_r = a_r A_{r-1},  H_r = a_r H_{r-1} + b_r,   (A, H) before a sequence = (1, h0[s])
//
// The whole packed tensor is one scan on the chunk engine (scan_engine.cuh),
// so tiles and look-backs run across sequence boundaries.  A boundary is a
// step that forgets everything before it: the element of row r is the
// affine map (A, H) -> (m A + u, m H + w) with
//   m = a_r, u = 0, w = b_r                       inside a sequence
//   m = 0,   u = a_r, w = a_r h0[s] + b_r          at a sequence's first row
// and maps compose as (m1,u1,w1) then (m2,u2,w2) = (m2 m1, m2 u1 + u2,
// m2 w1 + w2).  Where m2 = 0 the result takes (u2, w2) outright (a select,
// not 0 * x), so a non-finite state of one sequence never reaches the next.
// The backward is the same in reverse: the adjoint of row r reaches row r-1
// only inside a sequence (coefficient a_{r+1}, 0 at a sequence's last row).
//
// Each thread finds the sequences of its rows by one binary search of cu per
// round and a walk forward; rows of a warp are the same for all its lanes, so
// every branch on a boundary is uniform.  The kernels trust cu for indexing
// only within [0, nseq): a cu that is not non-decreasing from 0 to Ttot gives
// unspecified outputs, no out-of-bounds access, and the error bit
// kErrBadSeqlens that mg_workspace_status reports.
#include <cmath>

#include "scan_engine.cuh"

#ifndef MG_VL_PEEK
#define MG_VL_PEEK 0
#endif

namespace mg {
namespace {

// The sequence that holds packed row r: the largest s in [0, nseq) with
// cu[s] <= r (empty sequences are skipped).
__device__ __forceinline__ int seq_of(const long long *cu, int nseq, long long r)
{
    int lo = 0, hi = nseq;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// Sequence-start flags and sequence indices of rows r0 .. r0+N-1 (rows past
// Ttot: not starts).  bit i of the mask: row r0+i begins its sequence.
template <int N>
__device__ __forceinline__ unsigned seq_walk(const long long *cu, int nseq, long long Ttot,
                                             long long r0, int (&sq)[N], bool &bad)
{
    unsigned mask = 0;
    if (r0 >= Ttot) {
#pragma unroll
        for (int i = 0; i < N; ++i) sq[i] = 0;
        return 0;
    }
    int s = seq_of(cu, nseq, r0);
    long long lo = __ldg(cu + s), hi = __ldg(cu + s + 1);
    bad = bad || lo > r0 || hi <= r0 || (s == 0 && lo != 0) || (s + 1 == nseq && hi != Ttot);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const long long r = r0 + i;
        if (r < Ttot) {
            while (r >= hi && s + 1 < nseq) {   // the next non-empty sequence
                ++s;
                lo = hi;
                hi = __ldg(cu + s + 1);
                bad = bad || hi < lo || (s + 1 == nseq && hi != Ttot);
            }
            if (r == lo) mask |= 1u << i;
        }
        sq[i] = s;
    }
    return mask;
}

// ------------------------------------------------------------- forward
template <typename Tin, int VEC_, int L_>
struct VarFwd {
    static constexpr int NS = 3, VEC = VEC_, L = L_;
    static constexpr unsigned kPrefixStates = 0b110u;   // a prefix's m feeds no output
    static constexpr bool kReverse = false;
    static constexpr bool kPeek = MG_VL_PEEK != 0;   // look-back peek (measured)
    using S = St<NS, VEC>;
    struct Args {
        const Tin *a;
        const Tin *b;
        const long long *cu;
        int nseq;
        const float *h0;   // (nseq, D) or NULL
        float *A;
        float *H;
        unsigned *err;     // Control::error of the workspace
    };
    struct Regs {
        Raw<Tin, VEC> a[L];
        Raw<Tin, VEC> b[L];
        int sq[L];
        unsigned start;
        const float *h0;   // the start states (NULL: zero)
        int64_t D;
        int d;
        bool act;          // the thread's channels exist
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        bool bad = false;
        r.start = seq_walk<L>(p.cu, p.nseq, g.T, t0, r.sq, bad);
        if (bad) atomicOr(p.err, kErrBadSeqlens);
        r.h0 = p.h0;
        r.D = g.D;
        r.d = d;
        r.act = act;
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
    // start state of row i's sequence (row i begins it)
    __device__ static void h0_of(const Regs &r, int i, float (&h)[VEC])
    {
        if (r.h0 != nullptr && r.act) {
            load_vec<VEC>(r.h0 + int64_t(r.sq[i]) * r.D + r.d, h);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) h[v] = 0.f;
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        S e;
        if (r.start & (1u << i)) {
            float h[VEC];
            h0_of(r, i, h);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                e.v[0][v] = 0.f;
                e.v[1][v] = r.a[i][v];
                e.v[2][v] = fmaf(r.a[i][v], h[v], r.b[i][v]);
            }
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                e.v[0][v] = r.a[i][v];
                e.v[1][v] = 0.f;
                e.v[2][v] = r.b[i][v];
            }
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
            const float m = y.v[0][v];
            o.v[0][v] = m * x.v[0][v];
            o.v[1][v] = m == 0.f ? y.v[1][v] : fmaf(m, x.v[1][v], y.v[1][v]);
            o.v[2][v] = m == 0.f ? y.v[2][v] : fmaf(m, x.v[2][v], y.v[2][v]);
        }
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        float Av[VEC], Hv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Av[v] = st.v[1][v];
            Hv[v] = st.v[2][v];
        }
#pragma unroll
        for (int i = 0; i < L; ++i) {
            if (r.start & (1u << i)) {
                float h[VEC];
                h0_of(r, i, h);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    Av[v] = r.a[i][v];
                    Hv[v] = fmaf(r.a[i][v], h[v], r.b[i][v]);
                }
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = r.a[i][v];
                    Av[v] = a == 0.f ? 0.f : a * Av[v];
                    Hv[v] = a == 0.f ? r.b[i][v] : fmaf(a, Hv[v], r.b[i][v]);
                }
            }
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                store_out<VEC>(p.A + off, Av);
                store_out<VEC>(p.H + off, Hv);
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            st.v[1][v] = Av[v];
            st.v[2][v] = Hv[v];
        }
    }
};

// ------------------------------------------------------------ backward
// Reverse time.  Element of row r: (c_r, gA_r, gH_r) with c_r = a_{r+1} when
// row r+1 continues r's sequence, else 0 (the sequence's last row); state
// (C, mu, lam).  Epilogue: da_r = mu_r A_{r-1} + lam_r H_{r-1} with
// (A_{r-1}, H_{r-1}) = (1, h0[s]) at a sequence's first row, db_r = lam_r, and
// there dh0[s] = a_r lam_r.
template <typename Tin, int VEC_, int L_>
struct VarBwd {
    static constexpr int NS = 3, VEC = VEC_, L = L_;
    static constexpr unsigned kPrefixStates = 0b110u;   // a prefix's m feeds no output
    static constexpr bool kReverse = true;
    static constexpr bool kPeek = MG_VL_PEEK != 0;   // look-back peek (measured)
    using S = St<NS, VEC>;
    struct Args {
        const Tin *a;
        const long long *cu;
        int nseq;
        const float *h0;   // (nseq, D) or NULL
        const float *A;
        const float *H;
        const float *gA;
        const float *gH;
        float *da;
        float *db;
        float *dh0;        // (nseq, D), written when h0 is given
        unsigned *err;
    };
    struct Regs {
        Raw<Tin, VEC> c[L];    // a_{r+1} of each row (0 past a sequence's last row)
        float gA[L][VEC];
        float gB[L][VEC];
        int sq[L + 1];
        unsigned start;        // bit i: row t0+i begins its sequence (i <= L)
    };

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        bool bad = false;
        r.start = seq_walk<L + 1>(p.cu, p.nseq, g.T, t0, r.sq, bad);
        if (bad) atomicOr(p.err, kErrBadSeqlens);
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                load_vec<VEC>(p.gA + off, r.gA[i]);
                load_vec<VEC>(p.gH + off, r.gB[i]);
                // the next row continues this sequence unless it begins one
                if (t + 1 < g.T && !(r.start & (1u << (i + 1)))) {
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
            const float m = y.v[0][v];
            o.v[0][v] = m * x.v[0][v];
            o.v[1][v] = m == 0.f ? y.v[1][v] : fmaf(m, x.v[1][v], y.v[1][v]);
            o.v[2][v] = m == 0.f ? y.v[2][v] : fmaf(m, x.v[2][v], y.v[2][v]);
        }
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0,
                                    int d, bool act, const Regs &r, S &st)
    {
        // A_{r-1}, H_{r-1} of each row: (1, h0 or 0) at a sequence's first row
        float Ap[L][VEC], Hp[L][VEC];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const int64_t t = t0 + i;
            const bool first = r.start & (1u << i);
            if (act && t < g.T && !first) {
                const int64_t off = (bb * g.T + t - 1) * g.D + d;
                load_vec<VEC>(p.A + off, Ap[i]);
                load_vec<VEC>(p.H + off, Hp[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    Ap[i][v] = 1.f;
                    Hp[i][v] = 0.f;
                }
                if (act && t < g.T && p.h0 != nullptr)
                    load_vec<VEC>(p.h0 + int64_t(r.sq[i]) * g.D + d, Hp[i]);
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
                const float c = r.c[i][v];
                mu[v] = c == 0.f ? r.gA[i][v] : fmaf(c, mu[v], r.gA[i][v]);
                lam[v] = c == 0.f ? r.gB[i][v] : fmaf(c, lam[v], r.gB[i][v]);
                da[v] = fmaf(mu[v], Ap[i][v], lam[v] * Hp[i][v]);
            }
            const int64_t t = t0 + i;
            if (act && t < g.T) {
                const int64_t off = (bb * g.T + t) * g.D + d;
                store_out<VEC>(p.da + off, da);
                store_out<VEC>(p.db + off, lam);
                if (p.h0 != nullptr && (r.start & (1u << i))) {   // dh0 = a_r lam_r
                    Raw<Tin, VEC> ar;
                    ar.load(p.a + off);
                    float dh[VEC];
#pragma unroll
                    for (int v = 0; v < VEC; ++v) dh[v] = ar[v] * lam[v];
                    store_out<VEC>(p.dh0 + int64_t(r.sq[i]) * g.D + d, dh);
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            st.v[1][v] = mu[v];
            st.v[2][v] = lam[v];
        }
    }
};

// Tiles: as the linear scans' (float32 forward / backward shapes).
#ifndef MG_VLF_TX
#define MG_VLF_TX 16
#endif
#ifndef MG_VLF_TY
#define MG_VLF_TY 8
#endif
#ifndef MG_VLF_L
#define MG_VLF_L 8
#endif
#ifndef MG_VLF_MB
#define MG_VLF_MB 2
#endif
#ifndef MG_VLF_R
#define MG_VLF_R 2
#endif
#ifndef MG_VLB_TX
#define MG_VLB_TX 32
#endif
#ifndef MG_VLB_TY
#define MG_VLB_TY 8
#endif
#ifndef MG_VLB_L
#define MG_VLB_L 4
#endif
#ifndef MG_VLB_MB
#define MG_VLB_MB 2
#endif
#ifndef MG_VLB_R
#define MG_VLB_R 4
#endif
constexpr int kVTX = 32, kVTY = 8;

template <typename Tin>
using VFwd = ChanPlan<VarFwd<Tin, 4, MG_VLF_L>, MG_VLF_TX, MG_VLF_TY, MG_VLF_MB, MG_VLF_R>;
template <typename Tin>
using VFwdS = ChanPlan<VarFwd<Tin, 1, 8>, kVTX, kVTY>;
template <typename Tin>
using VBwd = ChanPlan<VarBwd<Tin, 4, MG_VLB_L>, MG_VLB_TX, MG_VLB_TY, MG_VLB_MB, MG_VLB_R>;
template <typename Tin>
using VBwdS = ChanPlan<VarBwd<Tin, 1, 4>, kVTX, kVTY>;

}  // namespace

size_t varlen_ws_bytes(int64_t Ttot, int64_t D)
{
    const size_t f = D % 4 == 0 ? VFwd<float>::ws_bytes(1, Ttot, D) : VFwdS<float>::ws_bytes(1, Ttot, D);
    const size_t b = D % 4 == 0 ? VBwd<float>::ws_bytes(1, Ttot, D) : VBwdS<float>::ws_bytes(1, Ttot, D);
    return f > b ? f : b;
}

mg_status launch_varlen_fwd(const void *a, const void *b, mg_dtype dt, const int64_t *cu,
                            int64_t nseq, const float *h0, float *A, float *H, int64_t Ttot,
                            int64_t D, void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_varlen_fwd";
    unsigned *err = &static_cast<Control *>(ws)->error;
    const long long *c = reinterpret_cast<const long long *>(cu);
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return VFwd<float>::launch({F(a), F(b), c, int(nseq), h0, A, H, err}, 1, Ttot, D, ws,
                                       wsb, s, o, nm);
        return VFwdS<float>::launch({F(a), F(b), c, int(nseq), h0, A, H, err}, 1, Ttot, D, ws, wsb,
                                    s, o, nm);
    }
    using P = const bf16_t *;
    if (D % 4 == 0)
        return VFwd<bf16_t>::launch({P(a), P(b), c, int(nseq), h0, A, H, err}, 1, Ttot, D, ws,
                                    wsb, s, o, nm);
    return VFwdS<bf16_t>::launch({P(a), P(b), c, int(nseq), h0, A, H, err}, 1, Ttot, D, ws, wsb,
                                 s, o, nm);
}

mg_status launch_varlen_bwd(const void *a, mg_dtype dt, const int64_t *cu, int64_t nseq,
                            const float *h0, const float *A, const float *H, const float *gA,
                            const float *gH, float *da, float *db, float *dh0, int64_t Ttot,
                            int64_t D, void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_linear_scan_varlen_bwd";
    unsigned *err = &static_cast<Control *>(ws)->error;
    const long long *c = reinterpret_cast<const long long *>(cu);
    if (dt == MG_F32) {
        using F = const float *;
        if (D % 4 == 0)
            return VBwd<float>::launch({F(a), c, int(nseq), h0, A, H, gA, gH, da, db, dh0, err}, 1,
                                       Ttot, D, ws, wsb, s, o, nm);
        return VBwdS<float>::launch({F(a), c, int(nseq), h0, A, H, gA, gH, da, db, dh0, err}, 1,
                                    Ttot, D, ws, wsb, s, o, nm);
    }
    using P = const bf16_t *;
    if (D % 4 == 0)
        return VBwd<bf16_t>::launch({P(a), c, int(nseq), h0, A, H, gA, gH, da, db, dh0, err}, 1,
                                    Ttot, D, ws, wsb, s, o, nm);
    return VBwdS<bf16_t>::launch({P(a), c, int(nseq), h0, A, H, gA, gH, da, db, dh0, err}, 1,
                                 Ttot, D, ws, wsb, s, o, nm);
}

}  // namespace mg

// k x k affine scans: affine_scan_fwd and affine_scan_bwd of the page
// "minGRU - Triton kernels".
//
// Both are scans of the pair operator on (C, V) with C a k x k coefficient
// and V a k x w value, element 1 earlier:
//     (C1, V1) o (C2, V2) = (C2 C1, C2 V1 + V2)
// forward:  element (A_t, B_t), w = v, outputs Abar_t = C, Bbar_t = V;
// backward: reverse time, element (A_{t+1}^T, [gAbar_t | gBbar_t]), w = k + v,
//           V = [M_t | Lam_t]; outputs dB_t = Lam_t and
//           dA_t = M_t Abar_{t-1}^T + Lam_t Bbar_{t-1}^T.
//
// Kernel shapes:
//   * k <= 4 (k = 4 with v <= 8, k = 2 with v >= 2): one lane owns one
//     sequence's whole state (k x (k + w) floats in registers); each warp
//     streams its steps through a ring of asynchronous copies
//     (affine_lane_kernel below).  The other small shapes keep the state in
//     one thread on the generic chunk engine (scan_engine.cuh).
//   * k = 16 with v in {8, 16}: the state on the tensor cores
//     (affine_mma_kernel below): one warp owns one sequence's sub-chunk of L
//     steps and holds S = X^T in mma.sync accumulator fragments; a CTA of NW
//     warps covers NW*L consecutive steps of one sequence.
//   * the other k in {8, 16}: the same tiles with one lane per column of X
//     (affine_col_kernel below).
// Every shape takes part in the same decoupled look-back as the other scans
// (lookback.cuh).
#include <type_traits>

#include "scan_engine.cuh"

namespace mg {
namespace {

// -------------------------------------------------------------- helpers

template <int N>
__device__ __forceinline__ void ld_floats(const float *p, float *o)
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 x = *reinterpret_cast<const float4 *>(p + 4 * q);
            o[4 * q] = x.x;
            o[4 * q + 1] = x.y;
            o[4 * q + 2] = x.z;
            o[4 * q + 3] = x.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int q = 0; q < N / 2; ++q) {
            const float2 x = *reinterpret_cast<const float2 *>(p + 2 * q);
            o[2 * q] = x.x;
            o[2 * q + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) o[q] = p[q];
    }
}

// Output rows of the small-k kernels, stored with the streaming cache hint
// under MG_STREAM_OUT (as the channel ops' outputs: not read again, so they
// do not displace the inputs that pass 2 re-reads from L2).
template <int N>
__device__ __forceinline__ void st_floats(float *p, const float *x)
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 v = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            if constexpr (MG_STREAM_OUT != 0) __stcs(reinterpret_cast<float4 *>(p + 4 * q), v);
            else *reinterpret_cast<float4 *>(p + 4 * q) = v;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int q = 0; q < N / 2; ++q) {
            const float2 v = make_float2(x[2 * q], x[2 * q + 1]);
            if constexpr (MG_STREAM_OUT != 0) __stcs(reinterpret_cast<float2 *>(p + 2 * q), v);
            else *reinterpret_cast<float2 *>(p + 2 * q) = v;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) {
            if constexpr (MG_STREAM_OUT != 0) __stcs(p + q, x[q]);
            else p[q] = x[q];
        }
    }
}

// o (R x N) = X (R x M) @ Y (M x N) [+ Z], row-major register arrays.
template <int R, int M, int N>
__device__ __forceinline__ void mm(const float *X, const float *Y, float *o)
{
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < N; ++j) {
            float s = X[i * M] * Y[j];
#pragma unroll
            for (int l = 1; l < M; ++l) s = fmaf(X[i * M + l], Y[l * N + j], s);
            o[i * N + j] = s;
        }
}

template <int R, int M, int N>
__device__ __forceinline__ void mm_add(const float *X, const float *Y, const float *Z, float *o)
{
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < N; ++j) {
            float s = Z[i * N + j];
#pragma unroll
            for (int l = 0; l < M; ++l) s = fmaf(X[i * M + l], Y[l * N + j], s);
            o[i * N + j] = s;
        }
}

// ============================================================ k <= 4
// Thread-owned state on the generic engine (VEC = 1: one sequence per lane).
// State layout: C (K*K, row-major) then V (K*W, row-major).

template <int K, int V_, int L_>
struct AffFwdSmall {
    static constexpr int W = V_, KK = K * K, KW = K * W;
    static constexpr int NS = KK + KW, VEC = 1, L = L_;
    static constexpr bool kReverse = false;
    using S = St<NS, 1>;
    struct Args {
        const float *A;
        const float *Bm;
        float *Abar;
        float *Bbar;
        const float *H0;  // (B, n, k, v) start states, or NULL (Bbar_0 = 0)
    };
    struct Regs {
        const float *A;
        const float *Bm;
        int64_t s0;      // step index (b, t0, n) = (b*T + t0)*n + n_
        int64_t stride;  // steps between consecutive t: n
        int nvalid;      // steps t0 .. t0+nvalid-1 are < T
    };
    __device__ static float *f(S &x) { return &x.v[0][0]; }
    __device__ static const float *f(const S &x) { return &x.v[0][0]; }

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        r.A = p.A;
        r.Bm = p.Bm;
        r.s0 = (bb * g.T + t0) * g.D + d;
        r.stride = g.D;
        const int64_t rem = g.T - t0;
        r.nvalid = act ? int(rem < 0 ? 0 : (rem > L ? L : rem)) : 0;
    }
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int i = 0; i < NS; ++i) e.v[i][0] = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) e.v[i * K + i][0] = 1.f;
        return e;
    }
    __device__ static S element(const Regs &r, int i)
    {
        if (i >= r.nvalid) return identity();
        S e;
        const int64_t s = r.s0 + i * r.stride;
        ld_floats<KK>(r.A + s * KK, f(e));
        ld_floats<KW>(r.Bm + s * KW, f(e) + KK);
        return e;
    }
    // State before step 1: (I, H0 of the sequence), or the identity.
    __device__ static S initial(const Args &p, const ChanGeom &g, int64_t bb, int d, bool act)
    {
        S e = identity();
        if (p.H0 != nullptr && act) ld_floats<KW>(p.H0 + (bb * g.D + d) * KW, f(e) + KK);
        return e;
    }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
        mm<K, K, K>(f(y), f(x), f(o));
        mm_add<K, K, W>(f(y), f(x) + KK, f(y) + KK, f(o) + KK);
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &, int64_t, int64_t, int, bool,
                                    const Regs &r, S &st)
    {
        float C[KK], Vv[KW];
#pragma unroll
        for (int i = 0; i < KK; ++i) C[i] = st.v[i][0];
#pragma unroll
        for (int i = 0; i < KW; ++i) Vv[i] = st.v[KK + i][0];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            if (i < r.nvalid) {
                const int64_t s = r.s0 + i * r.stride;
                float At[KK], Bt[KW], nC[KK], nV[KW];
                ld_floats<KK>(r.A + s * KK, At);
                ld_floats<KW>(r.Bm + s * KW, Bt);
                mm<K, K, K>(At, C, nC);
                mm_add<K, K, W>(At, Vv, Bt, nV);
#pragma unroll
                for (int q = 0; q < KK; ++q) C[q] = nC[q];
#pragma unroll
                for (int q = 0; q < KW; ++q) Vv[q] = nV[q];
                st_floats<KK>(p.Abar + s * KK, C);
                st_floats<KW>(p.Bbar + s * KW, Vv);
            }
        }
#pragma unroll
        for (int i = 0; i < KK; ++i) st.v[i][0] = C[i];
#pragma unroll
        for (int i = 0; i < KW; ++i) st.v[KK + i][0] = Vv[i];
    }
};

template <int K, int V_, int L_>
struct AffBwdSmall {
    static constexpr int VV = V_, W = K + V_, KK = K * K, KW = K * W, KV = K * V_;
    static constexpr int NS = KK + KW, VEC = 1, L = L_;
    static constexpr bool kReverse = true;
    using S = St<NS, 1>;
    struct Args {
        const float *A;
        const float *Abar;
        const float *Bbar;
        const float *gAbar;
        const float *gBbar;
        float *dA;
        float *dB;
    };
    struct Regs {
        Args p;
        int64_t s0, stride, t0, T;
        bool act;
    };
    __device__ static float *f(S &x) { return &x.v[0][0]; }
    __device__ static const float *f(const S &x) { return &x.v[0][0]; }

    __device__ static void load(const Args &p, const ChanGeom &g, int64_t bb, int64_t t0, int d,
                                bool act, Regs &r)
    {
        r.p = p;
        r.s0 = (bb * g.T + t0) * g.D + d;
        r.stride = g.D;
        r.t0 = t0;
        r.T = g.T;
        r.act = act;
    }
    __device__ static S identity()
    {
        S e;
#pragma unroll
        for (int i = 0; i < NS; ++i) e.v[i][0] = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) e.v[i * K + i][0] = 1.f;
        return e;
    }
    // G = [gAbar_t | gBbar_t] (K x W) of step s.
    __device__ static void load_g(const Regs &r, int64_t s, float *G)
    {
        float ga[KK], gb[KV];
        ld_floats<KK>(r.p.gAbar + s * KK, ga);
        ld_floats<KV>(r.p.gBbar + s * KV, gb);
#pragma unroll
        for (int i = 0; i < K; ++i) {
#pragma unroll
            for (int j = 0; j < K; ++j) G[i * W + j] = ga[i * K + j];
#pragma unroll
            for (int j = 0; j < VV; ++j) G[i * W + K + j] = gb[i * VV + j];
        }
    }
    // E_C = A_{t+1}^T, or 0 at t = T-1.
    __device__ static void load_ct(const Regs &r, int64_t t, int64_t s, float *Ct)
    {
        if (t + 1 < r.T) {
            float a[KK];
            ld_floats<KK>(r.p.A + (s + r.stride) * KK, a);
#pragma unroll
            for (int i = 0; i < K; ++i)
#pragma unroll
                for (int j = 0; j < K; ++j) Ct[i * K + j] = a[j * K + i];
        } else {
#pragma unroll
            for (int q = 0; q < KK; ++q) Ct[q] = 0.f;
        }
    }
    __device__ static S element(const Regs &r, int i)
    {
        const int64_t t = r.t0 + i;
        if (!r.act || t >= r.T) return identity();
        S e;
        const int64_t s = r.s0 + i * r.stride;
        load_ct(r, t, s, f(e));
        load_g(r, s, f(e) + KK);
        return e;
    }
    __device__ static S initial(const Args &, const ChanGeom &, int64_t, int, bool)
    {
        return identity();
    }
    __device__ static S combine(const S &x, const S &y)
    {
        S o;
        mm<K, K, K>(f(y), f(x), f(o));
        mm_add<K, K, W>(f(y), f(x) + KK, f(y) + KK, f(o) + KK);
        return o;
    }
    __device__ static void epilogue(const Args &p, const ChanGeom &, int64_t, int64_t, int, bool,
                                    const Regs &r, S &st)
    {
        float Vv[KW];
#pragma unroll
        for (int i = 0; i < KW; ++i) Vv[i] = st.v[KK + i][0];
#pragma unroll
        for (int i = L - 1; i >= 0; --i) {
            const int64_t t = r.t0 + i;
            if (r.act && t < r.T) {
                const int64_t s = r.s0 + i * r.stride;
                float Ct[KK], G[KW], nV[KW];
                load_ct(r, t, s, Ct);
                load_g(r, s, G);
                mm_add<K, K, W>(Ct, Vv, G, nV);
#pragma unroll
                for (int q = 0; q < KW; ++q) Vv[q] = nV[q];
                // dB_t = Lam_t;  dA_t = M_t Abar_{t-1}^T + Lam_t Bbar_{t-1}^T
                float dB[KV], dA[KK];
#pragma unroll
                for (int a = 0; a < K; ++a)
#pragma unroll
                    for (int c = 0; c < VV; ++c) dB[a * VV + c] = Vv[a * W + K + c];
                if (t > 0) {
                    float Ap[KK], Bp[KV];
                    ld_floats<KK>(p.Abar + (s - r.stride) * KK, Ap);
                    ld_floats<KV>(p.Bbar + (s - r.stride) * KV, Bp);
#pragma unroll
                    for (int a = 0; a < K; ++a)
#pragma unroll
                        for (int b = 0; b < K; ++b) {
                            float acc = Vv[a * W] * Ap[b * K];
#pragma unroll
                            for (int l = 1; l < K; ++l) acc = fmaf(Vv[a * W + l], Ap[b * K + l], acc);
#pragma unroll
                            for (int l = 0; l < VV; ++l)
                                acc = fmaf(Vv[a * W + K + l], Bp[b * VV + l], acc);
                            dA[a * K + b] = acc;
                        }
                } else {
#pragma unroll
                    for (int a = 0; a < K; ++a)
#pragma unroll
                        for (int b = 0; b < K; ++b) dA[a * K + b] = Vv[a * W + b];
                }
                st_floats<KK>(p.dA + s * KK, dA);
                st_floats<KV>(p.dB + s * KV, dB);
            }
        }
        // (the running transition product is not needed past the outputs)
#pragma unroll
        for (int i = 0; i < KW; ++i) st.v[KK + i][0] = Vv[i];
    }
};

// ===================== k <= 4: one sequence per lane, asynchronously fed
// A tile is 32 consecutive sequences of one batch row x TC = NW*L steps; warp
// w owns steps [w*L, (w+1)*L) of the tile, lane l sequence n0 + l, and keeps
// that sequence's state in registers.  At one step the block's 32 matrices
// are 32 consecutive rows (S bytes each) of each array; the warp copies them
// with coalesced 16-byte asynchronous copies (cp.async, one commit group per
// step) into a slot of its ring (NSL slots), placing 16-byte chunk c of row r
// at chunk c ^ ((r*S >> 7) & (S/16 - 1)) of that row, so the 32 lanes then
// reading one chunk of their own rows hit distinct banks.
// Pass 1 folds the warp's steps into its aggregate; the warps' aggregates are
// folded in shared memory (leaving each warp its exclusive prefix); warp 0
// finds the tile's carry-in by decoupled look-back; pass 2 streams the same
// steps again (now from L2) from each warp's start state and writes the
// outputs.  Needs every per-sequence block to be 16..128 bytes: k = 4 with
// v <= 8, or k = 2 with 2 <= v.

// The E floats of lane `lane`'s row in a swizzled 32-row block (base aligned
// to 1024 bytes): 16-byte chunk q of row r sits at chunk q ^ ((r*S >> 7) &
// (S/16 - 1)) of that row.
template <int E>
__device__ __forceinline__ void lane_row(const float *box, int lane, float *o)
{
    constexpr int S = E * 4, NQ = S / 16;
    static_assert(S % 16 == 0 && S <= 128, "rows of 16..128 bytes");
    const char *row = reinterpret_cast<const char *>(box) + lane * S;
    const int sw = ((lane * S) >> 7) & (NQ - 1);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const float4 x = *reinterpret_cast<const float4 *>(row + 16 * (q ^ sw));
        o[4 * q] = x.x;
        o[4 * q + 1] = x.y;
        o[4 * q + 2] = x.z;
        o[4 * q + 3] = x.w;
    }
}

template <int K_, int V_, bool BWD_, int NW_, int L_, int NSL_>
struct LCfg {
    static constexpr int K = K_, VV = V_, L = L_, NSL = NSL_;
    static constexpr bool BWD = BWD_;
    static constexpr int KK = K * K, KV = K * VV;
    using Op = typename std::conditional<BWD, AffBwdSmall<K, VV, 1>, AffFwdSmall<K, VV, 1>>::type;
    static constexpr int NS = Op::NS, W = Op::W;
    // Slot arrays (32 rows each, every region 1024-byte aligned).  Forward:
    // A_t, B_t.  Backward: A_{t+1}, gAbar_t, gBbar_t, Abar_{t-1}, Bbar_{t-1}.
    static constexpr int NARR = BWD ? 5 : 2;
    static constexpr int elems(int a) { return BWD ? ((a == 2 || a == 4) ? KV : KK) : (a == 1 ? KV : KK); }
    static constexpr int region(int a) { return (32 * elems(a) + 255) / 256 * 256; }  // floats
    static constexpr int offset(int a) { return a == 0 ? 0 : offset(a - 1) + region(a - 1); }
    static constexpr int STEP = offset(NARR);  // floats per slot
    static constexpr size_t smem_for(int nw)
    {
        return 1024 + size_t(nw * NSL * STEP) * sizeof(float) +
               size_t((nw + 1) * NS * 32) * sizeof(float);
    }
    // warps per CTA: NW_, halved while the CTA would not fit in shared memory
    static constexpr size_t kMax = 225 * 1024;
    static constexpr int NW = smem_for(NW_) <= kMax ? NW_
                              : smem_for(NW_ / 2) <= kMax ? NW_ / 2
                              : smem_for(NW_ / 4) <= kMax ? NW_ / 4 : 1;
    static constexpr int TC = NW * L;
    static constexpr size_t SMEM = smem_for(NW);
    static_assert(SMEM <= kMax, "tile does not fit in shared memory");
};

template <int K, int V>
constexpr bool lane_kernel_ok()
{
    return K <= 4 && (K * K * 4) % 16 == 0 && (K * V * 4) % 16 == 0 && K * K * 4 <= 128 &&
           K * V * 4 <= 128;
}

template <class Cf>
__global__ void __launch_bounds__(Cf::NW * 32)
    affine_lane_kernel(const typename Cf::Op::Args args, const ChanGeom g, const Lookback lb)
{
    using Op = typename Cf::Op;
    using S = typename Op::S;
    constexpr int K = Cf::K, KK = Cf::KK, KV = Cf::KV, VV = Cf::VV, NS = Cf::NS, W = Cf::W;
    constexpr int NW = Cf::NW, L = Cf::L, NSL = Cf::NSL, STEP = Cf::STEP;
    extern __shared__ float4 lane_smem[];
    // ring first, 1024-byte aligned for the swizzle, then the rest
    float *const ring = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(lane_smem) + 1023) & ~uintptr_t(1023));  // [NW][NSL][STEP]
    float *const s_agg = ring + NW * NSL * STEP;                                // [NW][NS][32]
    float *const s_carry = s_agg + NW * NS * 32;                                // [NS][32]

    unsigned tile;
    unsigned long long epoch;
    take_ticket(lb, tile, epoch);
    if (tile >= g.n_tiles) {
        if (threadIdx.x == 0) raise_error(lb, epoch, kErrBadTicket);
        finish_cta(lb, epoch);
        return;
    }
    const int c = int(tile / unsigned(g.nJ));
    const int j = int(tile % unsigned(g.nJ));
    const int64_t bb = j / g.nJb;
    const int n0 = (j % g.nJb) * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = n0 + lane;                         // this lane's sequence in the row
    const bool act = d < g.D;
    const int nseq = int(g.D - n0 < 32 ? g.D - n0 : 32);  // sequences in the block
    const int ct = Cf::BWD ? (g.nC - 1 - c) : c;
    const int64_t t0 = int64_t(ct) * Cf::TC;
    const int nv = int(g.T - t0 < Cf::TC ? g.T - t0 : Cf::TC);
    const int wbase = warp * L;
    const int nvw = nv - wbase < 0 ? 0 : (nv - wbase < L ? nv - wbase : L);
    const int pw = Cf::BWD ? NW - 1 - warp : warp;  // position in processing order
    float *const wring = ring + warp * NSL * STEP;
    auto row = [&](int64_t t) { return (bb * g.T + t) * g.D + n0; };  // row of lane 0
    auto tile_step = [&](int q) {
        const int k = q < nvw ? q : q - nvw;
        return Cf::BWD ? wbase + nvw - 1 - k : wbase + k;
    };
    const int nq = 2 * nvw;

    // every lane copies 16-byte pieces of the step's rows (coalesced) into
    // their swizzled positions; every call closes one group, empty or not
    auto issue = [&](int q) {
        if (q < nq) {
            float *buf = wring + (q % NSL) * STEP;
            const int64_t t = t0 + tile_step(q), r = row(t);
            auto rows = [&](float *dst, const float *src, int E) {  // nseq rows of E floats
                const int S = E * 4, per = S / 16, n = nseq * per;
                for (int i = lane; i < n; i += 32) {
                    const int rr = i / per, c = i % per;
                    const int sw = ((rr * S) >> 7) & (per - 1);
                    cp_async16(reinterpret_cast<char *>(dst) + rr * S + 16 * (c ^ sw),
                               src + int64_t(i) * 4);
                }
            };
            if constexpr (!Cf::BWD) {
                rows(buf + Cf::offset(0), args.A + r * KK, KK);
                rows(buf + Cf::offset(1), args.Bm + r * KV, KV);
            } else {
                rows(buf + Cf::offset(1), args.gAbar + r * KK, KK);
                rows(buf + Cf::offset(2), args.gBbar + r * KV, KV);
                if (t + 1 < g.T) rows(buf + Cf::offset(0), args.A + (r + g.D) * KK, KK);
                if (q >= nvw && t >= 1) {
                    rows(buf + Cf::offset(3), args.Abar + (r - g.D) * KK, KK);
                    rows(buf + Cf::offset(4), args.Bbar + (r - g.D) * KV, KV);
                }
            }
        }
        cp_async_commit();
    };
    // entry q has landed for every lane (this lane's group q, then a warp
    // barrier for the others' copies)
    auto wait_slot = [&](int q) -> const float * {
        cp_async_wait<NSL - 1>();
        __syncwarp();
        return wring + (q % NSL) * STEP;
    };
    // the lane's element of a step: coefficient E (k x k) and value (k x W)
    auto element = [&](const float *slot, int64_t t, S &e) {
        float *f = &e.v[0][0];
        if constexpr (!Cf::BWD) {
            lane_row<KK>(slot + Cf::offset(0), lane, f);
            lane_row<KV>(slot + Cf::offset(1), lane, f + KK);
        } else {
            if (t + 1 < g.T) {  // E = A_{t+1}^T
                float a[KK];
                lane_row<KK>(slot + Cf::offset(0), lane, a);
#pragma unroll
                for (int r = 0; r < K; ++r)
#pragma unroll
                    for (int q = 0; q < K; ++q) f[r * K + q] = a[q * K + r];
            } else {
#pragma unroll
                for (int q = 0; q < KK; ++q) f[q] = 0.f;
            }
            float ga[KK], gb[KV];
            lane_row<KK>(slot + Cf::offset(1), lane, ga);
            lane_row<KV>(slot + Cf::offset(2), lane, gb);
#pragma unroll
            for (int r = 0; r < K; ++r) {
#pragma unroll
                for (int q = 0; q < K; ++q) f[KK + r * W + q] = ga[r * K + q];
#pragma unroll
                for (int q = 0; q < VV; ++q) f[KK + r * W + K + q] = gb[r * VV + q];
            }
        }
    };

    for (int q = 0; q < NSL; ++q) issue(q);
    auto refill = [&](int q) { issue(q); };  // after every lane has read entry q - NSL

    // ---- pass 1: the warp's aggregate, in processing order
    S agg = Op::identity();
#pragma unroll 1
    for (int q = 0; q < nvw; ++q) {
        const int64_t t = t0 + tile_step(q);
        const float *slot = wait_slot(q);
        S e;
        if (act) element(slot, t, e);
        __syncwarp();
        refill(q + NSL);
        if (act) agg = Op::combine(agg, e);
    }
#pragma unroll
    for (int s = 0; s < NS; ++s) s_agg[(pw * NS + s) * 32 + lane] = agg.v[s][0];
    __syncthreads();

    // ---- warp 0: fold the warps' aggregates (each row gets its exclusive
    //      prefix back), then the look-back for the tile's carry-in
    S excl = Op::identity(), cta = Op::identity();
    if (warp == 0) {
#pragma unroll 1
        for (int w = 0; w < NW; ++w) {
            S x;
#pragma unroll
            for (int s = 0; s < NS; ++s) x.v[s][0] = s_agg[(w * NS + s) * 32 + lane];
            if (w > 0) {
#pragma unroll
                for (int s = 0; s < NS; ++s) s_agg[(w * NS + s) * 32 + lane] = cta.v[s][0];
            }
            cta = (w == 0) ? x : Op::combine(cta, x);
        }
        const int p0 = publish_first<Op, 32>(args, g, lb, c, j, bb, d, true, act, tile, epoch, cta);
        excl = find_carry<Op, 32>(args, g, lb, c, j, bb, d, true, act, tile, epoch, p0);
#pragma unroll
        for (int s = 0; s < NS; ++s) s_carry[s * 32 + lane] = excl.v[s][0];
    }
    __syncthreads();
    if (warp == 0) publish_prefix<Op, 32>(g, lb, c, j, true, tile, epoch, excl, cta);

    // ---- start state of this warp: carry o (warps before it)
    S st;
#pragma unroll
    for (int s = 0; s < NS; ++s) st.v[s][0] = s_carry[s * 32 + lane];
    if (pw > 0) {
        S x;
#pragma unroll
        for (int s = 0; s < NS; ++s) x.v[s][0] = s_agg[(pw * NS + s) * 32 + lane];
        st = Op::combine(st, x);
    }

    // ---- pass 2: re-run the steps from the start state, write the outputs
#pragma unroll 1
    for (int q = nvw; q < nq; ++q) {
        const int64_t t = t0 + tile_step(q), sidx = row(t) + lane;
        const float *slot = wait_slot(q);
        if constexpr (!Cf::BWD) {
            S e;
            if (act) element(slot, t, e);
            __syncwarp();
            refill(q + NSL);
            if (act) {
                st = Op::combine(st, e);
                st_floats<KK>(args.Abar + sidx * KK, &st.v[0][0]);
                st_floats<KV>(args.Bbar + sidx * KV, &st.v[KK][0]);
            }
        } else {
            if (act) {
                S e;
                element(slot, t, e);
                float *V = &st.v[KK][0];
                float nV[K * W];
                mm_add<K, K, W>(&e.v[0][0], V, &e.v[KK][0], nV);
#pragma unroll
                for (int q2 = 0; q2 < K * W; ++q2) V[q2] = nV[q2];
                // dB_t = Lam_t;  dA_t = M_t Abar_{t-1}^T + Lam_t Bbar_{t-1}^T
                float dB[KV], dA[KK];
#pragma unroll
                for (int a = 0; a < K; ++a)
#pragma unroll
                    for (int b2 = 0; b2 < VV; ++b2) dB[a * VV + b2] = V[a * W + K + b2];
                if (t > 0) {
                    float Ap[KK], Bp[KV];
                    lane_row<KK>(slot + Cf::offset(3), lane, Ap);
                    lane_row<KV>(slot + Cf::offset(4), lane, Bp);
#pragma unroll
                    for (int a = 0; a < K; ++a)
#pragma unroll
                        for (int b2 = 0; b2 < K; ++b2) {
                            float acc = V[a * W] * Ap[b2 * K];
#pragma unroll
                            for (int l = 1; l < K; ++l) acc = fmaf(V[a * W + l], Ap[b2 * K + l], acc);
#pragma unroll
                            for (int l = 0; l < VV; ++l) acc = fmaf(V[a * W + K + l], Bp[b2 * VV + l], acc);
                            dA[a * K + b2] = acc;
                        }
                } else {
#pragma unroll
                    for (int a = 0; a < K; ++a)
#pragma unroll
                        for (int b2 = 0; b2 < K; ++b2) dA[a * K + b2] = V[a * W + b2];
                }
                st_floats<KK>(args.dA + sidx * KK, dA);
                st_floats<KV>(args.dB + sidx * KV, dB);
            }
            __syncwarp();  // every lane has read the slot
            refill(q + NSL);
        }
    }
    finish_cta(lb, epoch);
}

template <class Cf>
struct LanePlan {
    static ChanGeom geom(int64_t B, int64_t T, int64_t n)
    {
        ChanGeom g;
        g.B = B;
        g.T = T;
        g.D = n;
        g.nJb = int((n + 31) / 32);
        g.nJ = int(B * g.nJb);
        g.nC = int((T + Cf::TC - 1) / Cf::TC);
        g.n_tiles = unsigned(g.nJ) * unsigned(g.nC);
        return g;
    }
    static size_t n_tiles(int64_t B, int64_t T, int64_t n)
    {
        return size_t(B * ((n + 31) / 32)) * size_t((T + Cf::TC - 1) / Cf::TC);
    }
    static size_t ws_bytes(int64_t B, int64_t T, int64_t n)
    {
        return tiled_ws_bytes(n_tiles(B, T, n), size_t(2) * Cf::NS * 32 * sizeof(unsigned long long));
    }
    static mg_status launch(const typename Cf::Op::Args &args, int64_t B, int64_t T, int64_t n,
                            void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o,
                            const char *name)
    {
        const size_t nt = n_tiles(B, T, n);
        if (nt >= (size_t(1) << 31) || B * ((n + 31) / 32) >= (int64_t(1) << 31))
            return fail(MG_ERR_UNSUPPORTED, "%s: %zu tiles exceed the 2^31 ticket range", name, nt);
        const size_t need = ws_bytes(B, T, n);
        if (wsb < need)
            return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, wsb, need);
        const ChanGeom g = geom(B, T, n);
        const Lookback lb = make_lookback(ws, nt, o);
        static const cudaError_t attr = cudaFuncSetAttribute(
            affine_lane_kernel<Cf>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cf::SMEM));
        if (attr != cudaSuccess) return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        affine_lane_kernel<Cf><<<unsigned(nt), Cf::NW * 32, Cf::SMEM, s>>>(args, g, lb);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", name, cudaGetErrorString(e));
        return MG_OK;
    }
};

// ======================================================= shared by k >= 8

struct AffGeom {
    int64_t B, T, n;
    int nJ;   // sequences B*n
    int nC;   // chunks along time
    unsigned n_tiles;
};

struct AffPtrs {
    const float *A, *Bm;                            // forward inputs
    const float *H0;                                // forward start states (B, n, k, v) or NULL
    float *Abar_out, *Bbar_out;                     // forward outputs
    const float *Abar, *Bbar, *gAbar, *gBbar;       // backward inputs (A shared)
    float *dA, *dB;                                 // backward outputs
};

// 3xTF32 products on the tensor cores: each fp32 operand is split into a
// tf32 high part and a remainder, and hi*hi, hi*lo, lo*hi are accumulated in
// fp32 (the dropped lo*lo term is below 2^-22 of each product).  The
// remainder is passed as a float: the tensor core reads
// its tf32 bits (the low 13 mantissa bits of the remainder dropped, toward
// zero), an error below 2^-21 of x.  hi is x rounded to nearest, so the
// remainder is positive or negative with equal odds and the error of hi + lo
// falls to either side of x: it does not build up along a recurrence (the
// orthogonality invariant and the parity margins measured the same as with
// the rounded remainder).
__device__ __forceinline__ void split_tf32_fast(float x, unsigned &hi, unsigned &lo)
{
    unsigned h;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
    hi = h;
    lo = __float_as_uint(x - __uint_as_float(h));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const unsigned (&a)[4], unsigned b0,
                                         unsigned b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ============================================= k in {8, 16}: column lanes
// One warp owns one sequence's sub-chunk of L steps, and lane l owns columns
// l, l + 32, ... of the state X = [C | V] (k rows, NC columns).  A step
// X <- E_C X + [0 | E_V] is, for each of the lane's columns, k dot products
// of the rows of E_C with that column: the rows are read by all 32 lanes at
// once from shared memory (broadcast loads, one address per load), the
// column never leaves the lane's registers, and E_V's entries for the
// column are the lane's own.  No state is exchanged between lanes, so the
// only chain from step to step is the lane's k independent dot products.
// The steps reach shared memory through each warp's ring of bulk copies
// (one mbarrier per slot), as in the kernels above.  A CTA of NW warps covers
// NW*L consecutive steps of one sequence.
// Forward: X = [Abar | Bbar] (NC = k + v).  Backward: X = [C | M | Lam]
// (NC = 2k + v) in pass 1; pass 2 needs only the value part [M | Lam]
// (W = k + v columns), whose C columns feed nothing but the aggregates.
template <int K_, int V_, bool BWD_, int NW_, int L_, int NSL_>
struct CCfg {
    static constexpr int K = K_, VV = V_, NW = NW_, L = L_, NSL = NSL_;
    static constexpr bool BWD = BWD_;
    static constexpr int KK = K * K, KV = K * VV;
    static constexpr int W = BWD ? K + VV : VV;     // columns of the value part
    static constexpr int NC = K + W;                // columns of X
    static constexpr int NCP = (NC + 3) / 4 * 4;    // row stride of stored matrices
    static constexpr int CPL = (NC + 31) / 32;      // columns per lane, all of X
    static constexpr int CPL2 = (W + 31) / 32;      // columns per lane, value part
    static constexpr int MAT = K * NCP;             // floats per stored matrix
    static constexpr int REC = MAT;                 // floats per global record
    static constexpr int TC = NW * L;               // steps per tile
    // Ring slot contents.  Forward: A_t, B_t.  Backward: A_{t+1}, gAbar_t,
    // gBbar_t, Abar_{t-1}, Bbar_{t-1}.  Each block is a multiple of 16 bytes.
    static constexpr int STEP = BWD ? 3 * KK + 2 * KV : KK + KV;
    static constexpr int OFF_G = KK, OFF_GB = 2 * KK, OFF_AP = 2 * KK + KV, OFF_BP = 3 * KK + KV;
    // The backward stages [M | Lam] of each step in shared memory for dA_t:
    // row stride XS keeps the tensor-core fragment loads free of conflicts.
    static constexpr int XS = (W + 3) / 4 * 4 + 4;
    static constexpr int XMAT = BWD ? K * XS : 0;
    static constexpr int BAR_FLOATS = (NW * NSL * 2 + 3) / 4 * 4;
    static constexpr size_t SMEM =
        size_t(BAR_FLOATS + NW * NSL * STEP + (NW + 1) * MAT + NW * XMAT) * sizeof(float);
    static_assert(K == 8 || K == 16, "column kernel is for k in {8, 16}");
    static_assert(NSL >= 2, "the ring needs two slots at least");
    static_assert((KV * 4) % 16 == 0 && (KK * 4) % 16 == 0, "bulk copies need 16-byte blocks");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// The lane's columns COFF + lane + 32 j (j < CN) of a matrix stored with row
// stride Cf::NCP, in shared (GLOBAL false) or global memory; columns at or
// past NC read as zero.
template <class Cf, int COFF, int CN, bool GLOBAL>
__device__ __forceinline__ void col_get(const float *m, int lane, float (&x)[CN][Cf::K])
{
#pragma unroll
    for (int j = 0; j < CN; ++j) {
        const int col = COFF + lane + 32 * j;
#pragma unroll
        for (int i = 0; i < Cf::K; ++i) {
            const float *a = m + i * Cf::NCP + col;
            x[j][i] = col < Cf::NC ? (GLOBAL ? __ldcg(a) : *a) : 0.f;
        }
    }
}

template <class Cf, int COFF, int CN, bool GLOBAL>
__device__ __forceinline__ void col_put(float *m, int lane, const float (&x)[CN][Cf::K])
{
#pragma unroll
    for (int j = 0; j < CN; ++j) {
        const int col = COFF + lane + 32 * j;
        if (col < Cf::NC) {
#pragma unroll
            for (int i = 0; i < Cf::K; ++i) {
                if (GLOBAL) __stcg(m + i * Cf::NCP + col, x[j][i]);
                else m[i * Cf::NCP + col] = x[j][i];
            }
        }
    }
}

// Columns of the identity element [I | 0].
template <class Cf, int COFF, int CN>
__device__ __forceinline__ void col_identity(int lane, float (&x)[CN][Cf::K])
{
#pragma unroll
    for (int j = 0; j < CN; ++j) {
        const int col = COFF + lane + 32 * j;
#pragma unroll
        for (int i = 0; i < Cf::K; ++i) x[j][i] = (i == col) ? 1.f : 0.f;
    }
}

// x <- E_C x + E[:, col] (col >= K) for a stored element E = [E_C | E_V]
// (row stride NCP): the combine (x earlier) o (E later).
template <class Cf, int COFF, int CN, bool GLOBAL>
__device__ __forceinline__ void col_apply(const float *E, int lane, float (&x)[CN][Cf::K])
{
    constexpr int K = Cf::K;
    float y[CN][K];
#pragma unroll
    for (int j = 0; j < CN; ++j) {
        const int col = COFF + lane + 32 * j;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const float *a = E + i * Cf::NCP + col;
            y[j][i] = (col >= K && col < Cf::NC) ? (GLOBAL ? __ldcg(a) : *a) : 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float e[K];
        if (GLOBAL) {
#pragma unroll
            for (int l = 0; l < K; l += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(E + i * Cf::NCP + l));
                e[l] = v.x;
                e[l + 1] = v.y;
                e[l + 2] = v.z;
                e[l + 3] = v.w;
            }
        } else {
            ld_floats<K>(E + i * Cf::NCP, e);
        }
#pragma unroll
        for (int j = 0; j < CN; ++j)
#pragma unroll
            for (int l = 0; l < K; ++l) y[j][i] = fmaf(e[l], x[j][l], y[j][i]);
    }
#pragma unroll
    for (int j = 0; j < CN; ++j)
#pragma unroll
        for (int i = 0; i < K; ++i) x[j][i] = y[j][i];
}

// Forward step from a ring slot: x <- A_t x + [0 | B_t] on the lane's column.
template <class Cf>
__device__ __forceinline__ void col_step_fwd(const float *slot, int lane, float (&x)[1][Cf::K])
{
    constexpr int K = Cf::K, VV = Cf::VV;
    const int col = lane;
    float y[K];
#pragma unroll
    for (int i = 0; i < K; ++i)
        y[i] = (col >= K && col < Cf::NC) ? slot[Cf::KK + i * VV + col - K] : 0.f;
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float e[K];
        ld_floats<K>(slot + i * K, e);
#pragma unroll
        for (int l = 0; l < K; ++l) y[i] = fmaf(e[l], x[0][l], y[i]);
    }
#pragma unroll
    for (int i = 0; i < K; ++i) x[0][i] = y[i];
}

// Backward step from a ring slot on columns COFF + lane + 32 j of X = [C | M |
// Lam]: x <- A_{t+1}^T x + [0 | gAbar_t | gBbar_t] (the first term absent at
// t = T-1).  Row l of A_{t+1} is read once and scattered over the k sums.
template <class Cf, int COFF, int CN>
__device__ __forceinline__ void col_step_bwd(const float *slot, bool has_next, int lane,
                                             float (&x)[CN][Cf::K])
{
    constexpr int K = Cf::K, VV = Cf::VV;
    float y[CN][K];
#pragma unroll
    for (int j = 0; j < CN; ++j) {
        const int col = COFF + lane + 32 * j;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            float v = 0.f;
            if (col >= K && col < 2 * K) v = slot[Cf::OFF_G + i * K + col - K];
            else if (col >= 2 * K && col < Cf::NC) v = slot[Cf::OFF_GB + i * VV + col - 2 * K];
            y[j][i] = v;
        }
    }
    if (has_next) {
#pragma unroll
        for (int l = 0; l < K; ++l) {
            float e[K];
            ld_floats<K>(slot + l * K, e);
#pragma unroll
            for (int j = 0; j < CN; ++j)
#pragma unroll
                for (int i = 0; i < K; ++i) y[j][i] = fmaf(e[i], x[j][l], y[j][i]);
        }
    }
#pragma unroll
    for (int j = 0; j < CN; ++j)
#pragma unroll
        for (int i = 0; i < K; ++i) x[j][i] = y[j][i];
}

template <class Cf>
__global__ void __launch_bounds__(Cf::NW * 32)
    affine_col_kernel(const AffPtrs p, const AffGeom g, const Lookback lb)
{
    constexpr int K = Cf::K, NW = Cf::NW, L = Cf::L, NSL = Cf::NSL, STEP = Cf::STEP;
    constexpr int KK = Cf::KK, KV = Cf::KV, VV = Cf::VV, NC = Cf::NC, MAT = Cf::MAT;
    constexpr int CPL = Cf::CPL, CPL2 = Cf::CPL2, XS = Cf::XS;
    extern __shared__ float4 aff_smem[];
    unsigned long long *const bars = reinterpret_cast<unsigned long long *>(aff_smem);  // [NW][NSL]
    float *const ring = reinterpret_cast<float *>(aff_smem) + Cf::BAR_FLOATS;          // [NW][NSL][STEP]
    float *const G = ring + NW * NSL * STEP;   // [NW][MAT]: warp aggregates, then inclusive
    float *const carry = G + NW * MAT;         // [MAT]
    float *const xst = carry + MAT;            // [NW][XMAT] (backward)

    unsigned tile;
    unsigned long long epoch;
    take_ticket(lb, tile, epoch);
    if (tile >= g.n_tiles) {
        if (threadIdx.x == 0) raise_error(lb, epoch, kErrBadTicket);
        finish_cta(lb, epoch);
        return;
    }
    const int c = int(tile / unsigned(g.nJ));
    const int j = int(tile % unsigned(g.nJ));
    const int64_t bb = j / g.n, nn = j % g.n;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ct = Cf::BWD ? (g.nC - 1 - c) : c;
    const int64_t t0 = int64_t(ct) * Cf::TC;
    const int nv = int(g.T - t0 < Cf::TC ? g.T - t0 : Cf::TC);
    const int wbase = warp * L;
    const int nvw = nv - wbase < 0 ? 0 : (nv - wbase < L ? nv - wbase : L);
    const int pw = Cf::BWD ? NW - 1 - warp : warp;
    unsigned long long *const wbar = bars + warp * NSL;
    float *const wring = ring + warp * NSL * STEP;
    auto step_index = [&](int64_t t) { return (bb * g.T + t) * g.n + nn; };
    auto tile_step = [&](int q) {
        const int k = q < nvw ? q : q - nvw;
        return Cf::BWD ? wbase + nvw - 1 - k : wbase + k;
    };
    const int nq = 2 * nvw;

    auto issue = [&](int q) {
        if (q >= nq) return;
        unsigned long long *bar = wbar + q % NSL;
        float *buf = wring + (q % NSL) * STEP;
        const int64_t t = t0 + tile_step(q), s = step_index(t);
        if constexpr (!Cf::BWD) {
            mbar_arrive_expect_tx(bar, (KK + KV) * 4);
            tma_load_1d(buf, p.A + s * KK, KK * 4, bar);
            tma_load_1d(buf + KK, p.Bm + s * KV, KV * 4, bar);
        } else {
            const bool next = t + 1 < g.T, prev = q >= nvw && t >= 1;
            mbar_arrive_expect_tx(bar, (KK + KV + (next ? KK : 0) + (prev ? KK + KV : 0)) * 4);
            tma_load_1d(buf + Cf::OFF_G, p.gAbar + s * KK, KK * 4, bar);
            tma_load_1d(buf + Cf::OFF_GB, p.gBbar + s * KV, KV * 4, bar);
            if (next) tma_load_1d(buf, p.A + (s + g.n) * KK, KK * 4, bar);
            if (prev) {
                tma_load_1d(buf + Cf::OFF_AP, p.Abar + (s - g.n) * KK, KK * 4, bar);
                tma_load_1d(buf + Cf::OFF_BP, p.Bbar + (s - g.n) * KV, KV * 4, bar);
            }
        }
    };
    auto wait_slot = [&](int q) -> const float * {
        unsigned long long *bar = wbar + q % NSL;
        const unsigned parity = unsigned(q / NSL) & 1u;
        if (!mbar_wait_bounded(bar, parity, lb.wait_limit_ns)) {
            if (lane == 0) raise_error(lb, epoch, kErrLookbackTimeout);
            mbar_wait_bounded(bar, parity, lb.wait_limit_ns);
        }
        return wring + (q % NSL) * STEP;
    };
    // refill slot q % NSL once every lane has used entry q - NSL (each lane's
    // loads of it have been consumed by its arithmetic before the __syncwarp)
    auto refill = [&](int q) {
        __syncwarp();
        if (lane == 0) issue(q);
    };

    if (lane == 0) {
        for (int q = 0; q < NSL; ++q) mbar_init(wbar + q, 1);
        for (int q = 0; q < NSL; ++q) issue(q);
    }
    __syncwarp();

    // ---- pass 1: aggregate of the warp's steps (all NC columns)
    {
        float x[CPL][K];
        col_identity<Cf, 0, CPL>(lane, x);
#pragma unroll 1
        for (int q = 0; q < nvw; ++q) {
            const int64_t t = t0 + tile_step(q);
            const float *slot = wait_slot(q);
            if constexpr (!Cf::BWD) col_step_fwd<Cf>(slot, lane, x);
            else col_step_bwd<Cf, 0, CPL>(slot, t + 1 < g.T, lane, x);
            refill(q + NSL);
        }
        col_put<Cf, 0, CPL, false>(G + pw * MAT, lane, x);
    }
    __syncthreads();

    // ---- warp 0: inclusive prefixes over the warps (processing order), then
    //      the look-back for the tile's carry-in
    if (warp == 0) {
        float x[CPL][K];
        col_get<Cf, 0, CPL, false>(G, lane, x);
        for (int w = 1; w < NW; ++w) {  // G[w] <- G[w-1] o G[w]
            col_apply<Cf, 0, CPL, false>(G + w * MAT, lane, x);
            __syncwarp();
            col_put<Cf, 0, CPL, false>(G + w * MAT, lane, x);
        }
        __syncwarp();
        const float *cta = G + (NW - 1) * MAT;
        const size_t slot = size_t(c) * g.nJ + j;
        float *rec_agg = lb.data + slot * 2 * Cf::REC;
        float *rec_pre = rec_agg + Cf::REC;
        float xc[CPL][K];
        if (c == 0) {
            if (!Cf::BWD && p.H0 != nullptr) {
                // carry = the start state [I | H0]; prefix = carry o cta
                const float *h0 = p.H0 + (bb * g.n + nn) * KV;
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) {
                    const int col = lane + 32 * jj;
#pragma unroll
                    for (int i = 0; i < K; ++i)
                        xc[jj][i] = col < K ? (i == col ? 1.f : 0.f)
                                            : (col < NC ? h0[i * VV + col - K] : 0.f);
                }
                col_put<Cf, 0, CPL, false>(carry, lane, xc);
                col_apply<Cf, 0, CPL, false>(cta, lane, xc);
                col_put<Cf, 0, CPL, true>(rec_pre, lane, xc);
            } else {
                col_put<Cf, 0, CPL, true>(rec_pre, lane, x);
                col_identity<Cf, 0, CPL>(lane, xc);
                col_put<Cf, 0, CPL, false>(carry, lane, xc);
            }
            publish(lb, slot, kStatusPrefix, epoch, tile);
        } else {
            // one poll of the window; the aggregate is published (and the
            // wait entered) only when it does not resolve the carry yet
            int pp = poll_window(lb, size_t(j), size_t(g.nJ), c, epoch);
            if (pp < 0) {
                col_put<Cf, 0, CPL, true>(rec_agg, lane, x);
                publish(lb, slot, kStatusAggregate, epoch, tile);
                pp = wait_window(lb, size_t(j), size_t(g.nJ), c, epoch, tile);
            }
            if (pp >= 0) {
                col_get<Cf, 0, CPL, true>(lb.data + (size_t(pp) * g.nJ + j) * 2 * Cf::REC + Cf::REC,
                                          lane, xc);
                for (int q = pp + 1; q < c; ++q)  // carry <- carry o agg(q)
                    col_apply<Cf, 0, CPL, true>(lb.data + (size_t(q) * g.nJ + j) * 2 * Cf::REC,
                                                lane, xc);
            } else {
                col_identity<Cf, 0, CPL>(lane, xc);
            }
            col_put<Cf, 0, CPL, false>(carry, lane, xc);
            col_apply<Cf, 0, CPL, false>(cta, lane, xc);  // prefix of this tile
            col_put<Cf, 0, CPL, true>(rec_pre, lane, xc);
            publish(lb, slot, kStatusPrefix, epoch, tile);
        }
    }
    __syncthreads();

    if constexpr (!Cf::BWD) {
        // ---- pass 2: re-run the warp's steps from its start state carry o
        //      G[pw-1] and write Abar_t, Bbar_t
        float x[1][K];
        col_get<Cf, 0, 1, false>(carry, lane, x);
        if (pw > 0) col_apply<Cf, 0, 1, false>(G + (pw - 1) * MAT, lane, x);
        const int col = lane;
#pragma unroll 1
        for (int q = nvw; q < nq; ++q) {
            const int64_t t = t0 + tile_step(q), s = step_index(t);
            const float *slot = wait_slot(q);
            col_step_fwd<Cf>(slot, lane, x);
            refill(q + NSL);
            if (col < K) {
                float *o = p.Abar_out + s * KK + col;
#pragma unroll
                for (int i = 0; i < K; ++i) o[i * K] = x[0][i];
            } else if (col < NC) {
                float *o = p.Bbar_out + s * KV + col - K;
#pragma unroll
                for (int i = 0; i < K; ++i) o[i * VV] = x[0][i];
            }
        }
    } else {
        // ---- pass 2 of the adjoint on the value part [M | Lam]: dB_t = Lam_t,
        //      dA_t = [M_t | Lam_t] [Abar_{t-1} | Bbar_{t-1}]^T
        float x[CPL2][K];
        col_get<Cf, K, CPL2, false>(carry, lane, x);
        if (pw > 0) col_apply<Cf, K, CPL2, false>(G + (pw - 1) * MAT, lane, x);
        float *const xw = xst + warp * Cf::XMAT;   // [M | Lam] of the current step
#pragma unroll 1
        for (int q = nvw; q < nq; ++q) {
            const int64_t t = t0 + tile_step(q), s = step_index(t);
            const float *slot = wait_slot(q);
            col_step_bwd<Cf, K, CPL2>(slot, t + 1 < g.T, lane, x);
#pragma unroll
            for (int jj = 0; jj < CPL2; ++jj) {
                const int c2 = lane + 32 * jj;   // column of [M | Lam]
                if (c2 < Cf::W) {
#pragma unroll
                    for (int i = 0; i < K; ++i) xw[i * XS + c2] = x[jj][i];
                    if (c2 >= K) {
                        float *o = p.dB + s * KV + c2 - K;
#pragma unroll
                        for (int i = 0; i < K; ++i) o[i * VV] = x[jj][i];
                    }
                }
            }
            __syncwarp();
            const float *Ap = slot + Cf::OFF_AP;
            const float *Bp = slot + Cf::OFF_BP;
            {
                // dA_t[a][b] = sum_q X[a][q] Y[b][q], Y = [Abar_{t-1} | Bbar_{t-1}]
                // (Abar_0 = I, Bbar_0 = 0): entries lane, lane + 32, ...
#pragma unroll
                for (int e = 0; e < (KK + 31) / 32; ++e) {
                    const int idx = lane + 32 * e, a = idx / K, b2 = idx % K;
                    if (idx >= KK) break;
                    float acc;
                    if (t > 0) {
                        acc = 0.f;
#pragma unroll
                        for (int qq = 0; qq < K; ++qq) acc = fmaf(xw[a * XS + qq], Ap[b2 * K + qq], acc);
#pragma unroll
                        for (int qq = 0; qq < VV; ++qq) acc = fmaf(xw[a * XS + K + qq], Bp[b2 * VV + qq], acc);
                    } else {
                        acc = xw[a * XS + b2];
                    }
                    p.dA[s * KK + idx] = acc;
                }
            }
            refill(q + NSL);   // also orders this step's reads of xw before the next writes
        }
    }
    finish_cta(lb, epoch);
}

template <class Cf>
struct ColPlan {
    static size_t n_tiles(int64_t B, int64_t T, int64_t n)
    {
        return size_t(B * n) * size_t((T + Cf::TC - 1) / Cf::TC);
    }
    static size_t ws_bytes(int64_t B, int64_t T, int64_t n)
    {
        return tiled_ws_bytes(n_tiles(B, T, n), size_t(2) * Cf::REC * sizeof(float));
    }
    static mg_status launch(const AffPtrs &p, int64_t B, int64_t T, int64_t n, void *ws,
                            size_t wsb, cudaStream_t s, const LaunchOpts &o, const char *name)
    {
        const size_t nt = n_tiles(B, T, n);
        if (nt >= (size_t(1) << 31) || B * n >= (int64_t(1) << 31))
            return fail(MG_ERR_UNSUPPORTED, "%s: %zu tiles exceed the 2^31 ticket range", name, nt);
        const size_t need = ws_bytes(B, T, n);
        if (wsb < need)
            return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, wsb, need);
        AffGeom g;
        g.B = B;
        g.T = T;
        g.n = n;
        g.nJ = int(B * n);
        g.nC = int((T + Cf::TC - 1) / Cf::TC);
        g.n_tiles = unsigned(nt);
        const Lookback lb = make_lookback(ws, nt, o);
        if (Cf::SMEM > 48 * 1024) {
            static const cudaError_t attr = cudaFuncSetAttribute(
                affine_col_kernel<Cf>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cf::SMEM));
            if (attr != cudaSuccess)
                return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        }
        affine_col_kernel<Cf><<<unsigned(nt), Cf::NW * 32, Cf::SMEM, s>>>(p, g, lb);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", name, cudaGetErrorString(e));
        return MG_OK;
    }
};

// ================================ k = 16: the state on the tensor cores
// The same tiles, ring and look-back as the column kernel, with the state
// held as S = X^T ((k + w) x k) in the accumulator fragments of
// mma.sync.m16n8k8 (tf32 operands, fp32 accumulation).  A step X <- E_C X +
// [0 | E_V] is S <- S E_C^T + [0 | E_V]^T: S is the A operand, E_C^T the B
// operand, [0 | E_V]^T the accumulator's start value.  The accumulator
// fragment of one step is the A operand fragment of the next once the k
// index inside each 8-wide k tile is read in the order 0, 2, 4, 6, 1, 3, 5,
// 7 (fragment slot q holds k = 2q, slot q + 4 holds k = 2q + 1); the B
// operand is read in the same order, so the sum is unchanged and the state
// never moves between lanes.  The tensor cores then broadcast E_C to the
// whole product, which from shared memory costs each lane only its own
// eight values per step.
// Every product is done in three parts on the split x = hi + lo (hi = x
// rounded to tf32, lo = the remainder rounded to tf32): hi*hi + hi*lo +
// lo*hi, dropping the lo*lo term (below 2^-22 of each product).
// The outputs are written with streaming stores, so that L2 keeps the
// inputs that pass 2 reads again rather than the outputs.
// Stored elements (warp aggregates, carries, look-back records) use the
// ring slot's layout: C (k x k) first, then the value blocks (forward: B
// (k x v); backward: M-part (k x k), then Lam-part (k x v)).
template <int V_, bool BWD_, int NW_, int L_, int NSL_, int MINB_ = 1>
struct MCfg {
    static constexpr int K = 16, VV = V_, NW = NW_, L = L_, NSL = NSL_;
    static constexpr int MINB = MINB_;   // CTAs per SM the registers must allow
    static constexpr bool BWD = BWD_;
    static constexpr int KK = K * K, KV = K * VV;
    static constexpr int W = BWD ? K + VV : VV;     // value columns of X
    static constexpr int NR = K + W;                // rows of S = X^T
    static constexpr int MT = (NR + 15) / 16;       // 16-row tiles of S
    static constexpr int EL = (BWD ? 2 * KK : KK) + KV;  // floats per stored element
    static constexpr int REC = EL;
    static constexpr int TC = NW * L;
    static constexpr int STEP = BWD ? 3 * KK + 2 * KV : KK + KV;
    static constexpr int OFF_AP = 2 * KK + KV, OFF_BP = 3 * KK + KV;
    static constexpr int XS = 40;                   // staged [M | Lam] row stride (backward)
    static constexpr int XMAT = BWD ? K * XS : 0;
    static constexpr int BAR_FLOATS = (NW * NSL * 2 + 3) / 4 * 4;
    static constexpr size_t SMEM =
        size_t(BAR_FLOATS + NW * NSL * STEP + (NW + 1) * EL + NW * XMAT) * sizeof(float);
    static_assert(VV == 8 || VV == 16, "tensor-core state for v in {8, 16}");
    static_assert(NSL >= 2, "the ring needs two slots at least");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// Address of value entry (row i, value column rp) of a stored element.
template <class Cf>
__device__ __forceinline__ int el_val_off(int i, int rp)
{
    if constexpr (!Cf::BWD) return Cf::KK + i * Cf::VV + rp;
    else return rp < Cf::K ? Cf::KK + i * Cf::K + rp : 2 * Cf::KK + i * Cf::VV + rp - Cf::K;
}

template <bool GLOBAL>
__device__ __forceinline__ float ldf(const float *a)
{
    return GLOBAL ? __ldcg(a) : *a;
}

// Fragment entry e of tile (mt, nt): S[16 mt + g + 8 (e >> 1)][8 nt + 2 q + (e & 1)].
template <class Cf>
using SFrag = float[Cf::MT][2][4];

template <class Cf, int MBEG>
__device__ __forceinline__ void mf_identity(int g, int q, SFrag<Cf> &s)
{
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s[mt][nt][e] = (16 * mt + g + 8 * (e >> 1) == 8 * nt + 2 * q + (e & 1)) ? 1.f : 0.f;
}

// S <- the stored element at E (S[r][i] = X[i][r]).
template <class Cf, int MBEG, bool GLOBAL>
__device__ __forceinline__ void mf_get(const float *E, int g, int q, SFrag<Cf> &s)
{
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * mt + g + 8 * (e >> 1), i = 8 * nt + 2 * q + (e & 1);
                float v = 0.f;
                if (r < Cf::K) v = ldf<GLOBAL>(E + i * Cf::K + r);
                else if (r - Cf::K < Cf::W) v = ldf<GLOBAL>(E + el_val_off<Cf>(i, r - Cf::K));
                s[mt][nt][e] = v;
            }
}

template <class Cf, int MBEG, bool GLOBAL>
__device__ __forceinline__ void mf_put(float *E, int g, int q, const SFrag<Cf> &s)
{
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * mt + g + 8 * (e >> 1), i = 8 * nt + 2 * q + (e & 1);
                float *a = nullptr;
                if (r < Cf::K) a = E + i * Cf::K + r;
                else if (r - Cf::K < Cf::W) a = E + el_val_off<Cf>(i, r - Cf::K);
                if (a) {
                    if (GLOBAL) __stcg(a, s[mt][nt][e]);
                    else *a = s[mt][nt][e];
                }
            }
}

// An element's operands for one step: the B fragments of E_C^T and the
// accumulator start [0 | E_V]^T (m tiles from MBEG on).
template <class Cf, int MBEG>
struct EFrag {
    float b[2][2][2];            // [kt][nt][slot]
    float v[Cf::MT][2][4];
};

// Load the element at E (ring slot or stored element).  TRANS: E holds A
// with E_C = A^T (the adjoint's ring).  has_c false: E_C = 0.
template <class Cf, int MBEG, bool GLOBAL, bool TRANS>
__device__ __forceinline__ void mf_load(const float *E, bool has_c, int g, int q,
                                        EFrag<Cf, MBEG> &f)
{
    constexpr int K = Cf::K;
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * mt + g + 8 * (e >> 1), i = 8 * nt + 2 * q + (e & 1);
                f.v[mt][nt][e] = (r >= K && r - K < Cf::W) ? ldf<GLOBAL>(E + el_val_off<Cf>(i, r - K)) : 0.f;
            }
#pragma unroll
    for (int kt = 0; kt < 2; ++kt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float v0 = 0.f, v1 = 0.f;
            if (has_c) {
                if constexpr (!TRANS) {   // B[j][i] = E_C[i][j]
                    const float *a = E + (8 * nt + g) * K + 8 * kt + 2 * q;
                    float2 p2;
                    if constexpr (GLOBAL) p2 = __ldcg(reinterpret_cast<const float2 *>(a));
                    else p2 = *reinterpret_cast<const float2 *>(a);
                    v0 = p2.x;
                    v1 = p2.y;
                } else {                  // B[j][i] = A[j][i]
                    v0 = ldf<GLOBAL>(E + (8 * kt + 2 * q) * K + 8 * nt + g);
                    v1 = ldf<GLOBAL>(E + (8 * kt + 2 * q + 1) * K + 8 * nt + g);
                }
            }
            f.b[kt][nt][0] = v0;
            f.b[kt][nt][1] = v1;
        }
}

// S <- S E_C^T + [0 | E_V]^T on the m tiles from MBEG on (each row of S
// evolves on its own).
template <class Cf, int MBEG>
__device__ __forceinline__ void mf_apply(const EFrag<Cf, MBEG> &f, bool has_c, SFrag<Cf> &s)
{
    float d[Cf::MT][2][4];
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[mt][nt][e] = f.v[mt][nt][e];
    if (has_c) {
        // Both operands are split with one conversion each (split_tf32_fast):
        // the remainder's dropped bits err to either side of x with equal
        // odds, so the error does not build up along the recurrence.
        unsigned bh[2][2][2], bl[2][2][2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                split_tf32_fast(f.b[kt][nt][0], bh[kt][nt][0], bl[kt][nt][0]);
                split_tf32_fast(f.b[kt][nt][1], bh[kt][nt][1], bl[kt][nt][1]);
            }
#pragma unroll
        for (int mt = MBEG; mt < Cf::MT; ++mt) {
            unsigned ah[2][4], al[2][4];
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                split_tf32_fast(s[mt][kt][0], ah[kt][0], al[kt][0]);
                split_tf32_fast(s[mt][kt][2], ah[kt][1], al[kt][1]);
                split_tf32_fast(s[mt][kt][1], ah[kt][2], al[kt][2]);
                split_tf32_fast(s[mt][kt][3], ah[kt][3], al[kt][3]);
            }
            // Each tensor-core accumulation rounds at its result's magnitude,
            // so the small hi*lo and lo*hi terms are summed before any hi*hi
            // term: on rows of the C part (start value 0) in the accumulator
            // itself, first; on value rows (start value E_V) in an
            // accumulator of their own, added after.
            const bool c_rows = 16 * mt + 15 < Cf::K;
            if (c_rows) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        mma_tf32(d[mt][nt], al[kt], bh[kt][nt][0], bh[kt][nt][1]);
                        mma_tf32(d[mt][nt], ah[kt], bl[kt][nt][0], bl[kt][nt][1]);
                    }
#pragma unroll
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        mma_tf32(d[mt][nt], ah[kt], bh[kt][nt][0], bh[kt][nt][1]);
            } else {
                float cr[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) cr[nt][e] = 0.f;
#pragma unroll
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        mma_tf32(cr[nt], al[kt], bh[kt][nt][0], bh[kt][nt][1]);
                        mma_tf32(cr[nt], ah[kt], bl[kt][nt][0], bl[kt][nt][1]);
                        mma_tf32(d[mt][nt], ah[kt], bh[kt][nt][0], bh[kt][nt][1]);
                    }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[mt][nt][e] += cr[nt][e];
            }
        }
    }
#pragma unroll
    for (int mt = MBEG; mt < Cf::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[mt][nt][e] = d[mt][nt][e];
}

template <class Cf, int MBEG, bool GLOBAL, bool TRANS>
__device__ __forceinline__ void mf_step(const float *E, bool has_c, int g, int q, SFrag<Cf> &s)
{
    EFrag<Cf, MBEG> f;
    mf_load<Cf, MBEG, GLOBAL, TRANS>(E, has_c, g, q, f);
    mf_apply<Cf, MBEG>(f, has_c, s);
}

// The C rows (m tile 0) of S <- those of the stored element at E, exactly
// (the product of an identity C part with E's, which the split products
// would round).
template <class Cf>
__device__ __forceinline__ void mf_copy_c_rows(const float *E, int g, int q, SFrag<Cf> &s)
{
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = g + 8 * (e >> 1), i = 8 * nt + 2 * q + (e & 1);
            s[0][nt][e] = E[i * Cf::K + r];
        }
}

template <class Cf>
__global__ void __launch_bounds__(Cf::NW * 32, Cf::MINB)
    affine_mma_kernel(const AffPtrs p, const AffGeom g, const Lookback lb)
{
    constexpr int K = Cf::K, NW = Cf::NW, L = Cf::L, NSL = Cf::NSL, STEP = Cf::STEP;
    constexpr int KK = Cf::KK, KV = Cf::KV, VV = Cf::VV, EL = Cf::EL, XS = Cf::XS;
    extern __shared__ float4 aff_smem[];
    unsigned long long *const bars = reinterpret_cast<unsigned long long *>(aff_smem);  // [NW][NSL]
    float *const ring = reinterpret_cast<float *>(aff_smem) + Cf::BAR_FLOATS;          // [NW][NSL][STEP]
    float *const G = ring + NW * NSL * STEP;   // [NW][EL]: warp aggregates, then inclusive
    float *const carry = G + NW * EL;          // [EL]
    float *const xst = carry + EL;             // [NW][XMAT] (backward)

    unsigned tile;
    unsigned long long epoch;
    take_ticket(lb, tile, epoch);
    if (tile >= g.n_tiles) {
        if (threadIdx.x == 0) raise_error(lb, epoch, kErrBadTicket);
        finish_cta(lb, epoch);
        return;
    }
    const int c = int(tile / unsigned(g.nJ));
    const int j = int(tile % unsigned(g.nJ));
    const int64_t bb = j / g.n, nn = j % g.n;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int fg = lane >> 2, fq = lane & 3;   // fragment row group, column pair
    const int ct = Cf::BWD ? (g.nC - 1 - c) : c;
    const int64_t t0 = int64_t(ct) * Cf::TC;
    const int nv = int(g.T - t0 < Cf::TC ? g.T - t0 : Cf::TC);
    const int wbase = warp * L;
    const int nvw = nv - wbase < 0 ? 0 : (nv - wbase < L ? nv - wbase : L);
    const int pw = Cf::BWD ? NW - 1 - warp : warp;
    unsigned long long *const wbar = bars + warp * NSL;
    float *const wring = ring + warp * NSL * STEP;
    auto step_index = [&](int64_t t) { return (bb * g.T + t) * g.n + nn; };
    auto tile_step = [&](int qq) {
        const int k = qq < nvw ? qq : qq - nvw;
        return Cf::BWD ? wbase + nvw - 1 - k : wbase + k;
    };
    const int nq = 2 * nvw;

    auto issue = [&](int qq) {
        if (qq >= nq) return;
        unsigned long long *bar = wbar + qq % NSL;
        float *buf = wring + (qq % NSL) * STEP;
        const int64_t t = t0 + tile_step(qq), s = step_index(t);
        if constexpr (!Cf::BWD) {
            mbar_arrive_expect_tx(bar, (KK + KV) * 4);
            tma_load_1d(buf, p.A + s * KK, KK * 4, bar);
            tma_load_1d(buf + KK, p.Bm + s * KV, KV * 4, bar);
        } else {
            const bool next = t + 1 < g.T, prev = qq >= nvw && t >= 1;
            mbar_arrive_expect_tx(bar, (KK + KV + (next ? KK : 0) + (prev ? KK + KV : 0)) * 4);
            tma_load_1d(buf + KK, p.gAbar + s * KK, KK * 4, bar);
            tma_load_1d(buf + 2 * KK, p.gBbar + s * KV, KV * 4, bar);
            if (next) tma_load_1d(buf, p.A + (s + g.n) * KK, KK * 4, bar);
            if (prev) {
                tma_load_1d(buf + Cf::OFF_AP, p.Abar + (s - g.n) * KK, KK * 4, bar);
                tma_load_1d(buf + Cf::OFF_BP, p.Bbar + (s - g.n) * KV, KV * 4, bar);
            }
        }
    };
    auto wait_slot = [&](int qq) -> const float * {
        unsigned long long *bar = wbar + qq % NSL;
        const unsigned parity = unsigned(qq / NSL) & 1u;
        if (!mbar_wait_bounded(bar, parity, lb.wait_limit_ns)) {
            if (lane == 0) raise_error(lb, epoch, kErrLookbackTimeout);
            mbar_wait_bounded(bar, parity, lb.wait_limit_ns);
        }
        return wring + (qq % NSL) * STEP;
    };
    // refill slot qq % NSL once every lane has used entry qq - NSL (each
    // lane's loads of it were consumed by its arithmetic before the
    // __syncwarp)
    auto refill = [&](int qq) {
        __syncwarp();
        if (lane == 0) issue(qq);
    };

    if (lane == 0) {
        for (int qq = 0; qq < NSL; ++qq) mbar_init(wbar + qq, 1);
        for (int qq = 0; qq < NSL; ++qq) issue(qq);
    }
    __syncwarp();

    SFrag<Cf> s;
    // ---- pass 1: aggregate of the warp's steps (every row of S)
    mf_identity<Cf, 0>(fg, fq, s);
#pragma unroll 1
    for (int qq = 0; qq < nvw; ++qq) {
        const int64_t t = t0 + tile_step(qq);
        const float *slot = wait_slot(qq);
        mf_step<Cf, 0, false, Cf::BWD>(slot, !Cf::BWD || t + 1 < g.T, fg, fq, s);
        refill(qq + NSL);
    }
    mf_put<Cf, 0, false>(G + pw * EL, fg, fq, s);
    __syncthreads();

    // ---- warp 0: inclusive prefixes over the warps (processing order), then
    //      the look-back for the tile's carry-in
    if (warp == 0) {
        mf_get<Cf, 0, false>(G, fg, fq, s);
        for (int w = 1; w < NW; ++w) {  // G[w] <- G[w-1] o G[w]
            mf_step<Cf, 0, false, false>(G + w * EL, true, fg, fq, s);
            __syncwarp();
            mf_put<Cf, 0, false>(G + w * EL, fg, fq, s);
        }
        __syncwarp();
        const float *cta = G + (NW - 1) * EL;
        const size_t slot = size_t(c) * g.nJ + j;
        float *rec_agg = lb.data + slot * 2 * Cf::REC;
        float *rec_pre = rec_agg + Cf::REC;
        SFrag<Cf> sc;
        if (c == 0) {
            if (!Cf::BWD && p.H0 != nullptr) {
                // carry = the start state [I | H0]; prefix = carry o cta
                const float *h0 = p.H0 + (bb * g.n + nn) * KV;
#pragma unroll
                for (int mt = 0; mt < Cf::MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = 16 * mt + fg + 8 * (e >> 1), i = 8 * nt + 2 * fq + (e & 1);
                            sc[mt][nt][e] = r < K ? (r == i ? 1.f : 0.f)
                                                  : (r - K < VV ? h0[i * VV + r - K] : 0.f);
                        }
                mf_put<Cf, 0, false>(carry, fg, fq, sc);
                mf_step<Cf, 1, false, false>(cta, true, fg, fq, sc);   // value rows
                mf_copy_c_rows<Cf>(cta, fg, fq, sc);                  // C rows: I o cta = cta
                mf_put<Cf, 0, true>(rec_pre, fg, fq, sc);
            } else {
                mf_put<Cf, 0, true>(rec_pre, fg, fq, s);
                mf_identity<Cf, 0>(fg, fq, sc);
                mf_put<Cf, 0, false>(carry, fg, fq, sc);
            }
            publish(lb, slot, kStatusPrefix, epoch, tile);
        } else {
            // one poll of the window; the aggregate is published (and the
            // wait entered) only when it does not resolve the carry yet
            int pp = poll_window(lb, size_t(j), size_t(g.nJ), c, epoch);
            if (pp < 0) {
                mf_put<Cf, 0, true>(rec_agg, fg, fq, s);
                publish(lb, slot, kStatusAggregate, epoch, tile);
                pp = wait_window(lb, size_t(j), size_t(g.nJ), c, epoch, tile);
            }
            if (pp >= 0) {
                mf_get<Cf, 0, true>(lb.data + (size_t(pp) * g.nJ + j) * 2 * Cf::REC + Cf::REC,
                                    fg, fq, sc);
                // carry <- carry o agg(qc), the records fetched four at a time
                auto rec = [&](int qc) { return lb.data + (size_t(qc) * g.nJ + j) * 2 * Cf::REC; };
                int qc = pp + 1;
                for (; qc + 4 <= c; qc += 4) {
                    EFrag<Cf, 0> f[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) mf_load<Cf, 0, true, false>(rec(qc + u), true, fg, fq, f[u]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) mf_apply<Cf, 0>(f[u], true, sc);
                }
                for (; qc < c; ++qc) mf_step<Cf, 0, true, false>(rec(qc), true, fg, fq, sc);
            } else {
                mf_identity<Cf, 0>(fg, fq, sc);
            }
            mf_put<Cf, 0, false>(carry, fg, fq, sc);
            mf_step<Cf, 0, false, false>(cta, true, fg, fq, sc);  // prefix of this tile
            mf_put<Cf, 0, true>(rec_pre, fg, fq, sc);
            publish(lb, slot, kStatusPrefix, epoch, tile);
        }
    }
    __syncthreads();

    constexpr int M0 = Cf::BWD ? 1 : 0;   // pass 2 of the adjoint: [M | Lam] rows only
    mf_get<Cf, M0, false>(carry, fg, fq, s);
    if (pw > 0) {
        if (!Cf::BWD && c == 0) {
            // the carry of chunk 0 is [I | H0] (H0 = 0 without a start
            // state): the C rows of carry o G[pw-1] are G[pw-1]'s own
            mf_step<Cf, 1, false, false>(G + (pw - 1) * EL, true, fg, fq, s);
            mf_copy_c_rows<Cf>(G + (pw - 1) * EL, fg, fq, s);
        } else {
            mf_step<Cf, M0, false, false>(G + (pw - 1) * EL, true, fg, fq, s);
        }
    }
    if constexpr (!Cf::BWD) {
        // ---- pass 2: re-run the warp's steps from its start state, write
        //      Abar_t (rows r < k of S, transposed) and Bbar_t (rows k..)
#pragma unroll 1
        for (int qq = nvw; qq < nq; ++qq) {
            const int64_t t = t0 + tile_step(qq), si = step_index(t);
            const float *slot = wait_slot(qq);
            mf_step<Cf, 0, false, false>(slot, true, fg, fq, s);
            refill(qq + NSL);
            float *ab = p.Abar_out + si * KK, *bo = p.Bbar_out + si * KV;
#pragma unroll
            for (int mt = 0; mt < Cf::MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = 16 * mt + fg + 8 * (e >> 1), i = 8 * nt + 2 * fq + (e & 1);
                        if (r < K) __stcs(ab + i * K + r, s[mt][nt][e]);
                        else if (r - K < VV) __stcs(bo + i * VV + r - K, s[mt][nt][e]);
                    }
        }
    } else {
        // ---- pass 2 of the adjoint: dB_t = Lam_t; dA_t = [M_t | Lam_t]
        //      [Abar_{t-1} | Bbar_{t-1}]^T, as dA_t^T = Y S_v with Y =
        //      [Abar_{t-1} | Bbar_{t-1}] (A operand, from the ring slot) and
        //      S_v = [M_t | Lam_t]^T (B operand, staged in shared memory as
        //      [M_t | Lam_t], row stride XS)
        constexpr int W = Cf::W, KTD = W / 8;
        float *const xw = xst + warp * Cf::XMAT;
#pragma unroll 1
        for (int qq = nvw; qq < nq; ++qq) {
            const int64_t t = t0 + tile_step(qq), si = step_index(t);
            const float *slot = wait_slot(qq);
            mf_step<Cf, 1, false, true>(slot, t + 1 < g.T, fg, fq, s);
#pragma unroll
            for (int mt = 1; mt < Cf::MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = 16 * mt + fg + 8 * (e >> 1), i = 8 * nt + 2 * fq + (e & 1);
                        if (r - K < W) {
                            xw[i * XS + r - K] = s[mt][nt][e];
                            if (r >= 2 * K) __stcs(p.dB + si * KV + i * VV + r - 2 * K, s[mt][nt][e]);
                        }
                    }
            __syncwarp();
            float *da = p.dA + si * KK;
            if (t > 0) {
                const float *Ap = slot + Cf::OFF_AP;
                const float *Bp = slot + Cf::OFF_BP;
                float acc[2][4] = {};
#pragma unroll
                for (int kt = 0; kt < KTD; ++kt) {
                    // A operand: Y rows fg, fg + 8, columns 8 kt + 2 fq (+1)
                    float y0[2], y1[2];
                    if (kt < 2) {
                        const float2 u0 = *reinterpret_cast<const float2 *>(Ap + fg * K + 8 * kt + 2 * fq);
                        const float2 u1 = *reinterpret_cast<const float2 *>(Ap + (fg + 8) * K + 8 * kt + 2 * fq);
                        y0[0] = u0.x; y0[1] = u0.y; y1[0] = u1.x; y1[1] = u1.y;
                    } else {
                        const float2 u0 = *reinterpret_cast<const float2 *>(Bp + fg * VV + 8 * kt - K + 2 * fq);
                        const float2 u1 = *reinterpret_cast<const float2 *>(Bp + (fg + 8) * VV + 8 * kt - K + 2 * fq);
                        y0[0] = u0.x; y0[1] = u0.y; y1[0] = u1.x; y1[1] = u1.y;
                    }
                    unsigned ah[4], al[4];
                    split_tf32_fast(y0[0], ah[0], al[0]);
                    split_tf32_fast(y1[0], ah[1], al[1]);
                    split_tf32_fast(y0[1], ah[2], al[2]);
                    split_tf32_fast(y1[1], ah[3], al[3]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float2 xv = *reinterpret_cast<const float2 *>(xw + (8 * nt + fg) * XS + 8 * kt + 2 * fq);
                        unsigned bh0, bl0, bh1, bl1;
                        split_tf32_fast(xv.x, bh0, bl0);
                        split_tf32_fast(xv.y, bh1, bl1);
                        mma_tf32(acc[nt], al, bh0, bh1);
                        mma_tf32(acc[nt], ah, bl0, bl1);
                        mma_tf32(acc[nt], ah, bh0, bh1);
                    }
                }
                // acc[nt][e] = dA^T[fg + 8 (e >> 1)][8 nt + 2 fq + (e & 1)]
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        __stcs(da + (8 * nt + 2 * fq + (e & 1)) * K + fg + 8 * (e >> 1), acc[nt][e]);
            } else {   // Abar_0 = I, Bbar_0 = 0: dA_0 = M_0
#pragma unroll
                for (int e = 0; e < KK / 32; ++e) {
                    const int idx = lane + 32 * e;
                    __stcs(da + idx, xw[(idx / K) * XS + idx % K]);
                }
            }
            refill(qq + NSL);   // also orders this step's reads of xw before the next writes
        }
    }
    finish_cta(lb, epoch);
}

template <class Cf>
struct MmaPlan {
    static size_t n_tiles(int64_t B, int64_t T, int64_t n)
    {
        return size_t(B * n) * size_t((T + Cf::TC - 1) / Cf::TC);
    }
    static size_t ws_bytes(int64_t B, int64_t T, int64_t n)
    {
        return tiled_ws_bytes(n_tiles(B, T, n), size_t(2) * Cf::REC * sizeof(float));
    }
    static mg_status launch(const AffPtrs &p, int64_t B, int64_t T, int64_t n, void *ws,
                            size_t wsb, cudaStream_t s, const LaunchOpts &o, const char *name)
    {
        const size_t nt = n_tiles(B, T, n);
        if (nt >= (size_t(1) << 31) || B * n >= (int64_t(1) << 31))
            return fail(MG_ERR_UNSUPPORTED, "%s: %zu tiles exceed the 2^31 ticket range", name, nt);
        const size_t need = ws_bytes(B, T, n);
        if (wsb < need)
            return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, wsb, need);
        AffGeom g;
        g.B = B;
        g.T = T;
        g.n = n;
        g.nJ = int(B * n);
        g.nC = int((T + Cf::TC - 1) / Cf::TC);
        g.n_tiles = unsigned(nt);
        const Lookback lb = make_lookback(ws, nt, o);
        if (Cf::SMEM > 48 * 1024) {
            static const cudaError_t attr = cudaFuncSetAttribute(
                affine_mma_kernel<Cf>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cf::SMEM));
            if (attr != cudaSuccess)
                return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        }
        affine_mma_kernel<Cf><<<unsigned(nt), Cf::NW * 32, Cf::SMEM, s>>>(p, g, lb);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", name, cudaGetErrorString(e));
        return MG_OK;
    }
};

// ------------------------------------------------------------ dispatch

// Tiles, each overridable at build time.  k <= 4 (thread-owned state on the
// chunk engine): TY thread rows x L steps of 32 sequences, MB minimum CTAs per
// SM.  k = 8, 16 (warp kernel): NW warps x L steps of one sequence, DB =
// double-buffered state exchange, NSL ring slots per warp.
#ifndef MG_AFS_TY
#define MG_AFS_TY 8
#endif
#ifndef MG_AFS_L
#define MG_AFS_L 4
#endif
#ifndef MG_AFS_MB
#define MG_AFS_MB 1
#endif
#ifndef MG_AFSB_TY
#define MG_AFSB_TY 8
#endif
#ifndef MG_AFSB_L
#define MG_AFSB_L 4
#endif
#ifndef MG_AFSB_MB
#define MG_AFSB_MB 1
#endif
#ifndef MG_AFL_NW
#define MG_AFL_NW 4
#endif
#ifndef MG_AFL_L
#define MG_AFL_L 32
#endif
#ifndef MG_AFL_NSL
#define MG_AFL_NSL 6
#endif
#ifndef MG_AFLB_NW
#define MG_AFLB_NW 4
#endif
#ifndef MG_AFLB_L
#define MG_AFLB_L 32
#endif
#ifndef MG_AFLB_NSL
#define MG_AFLB_NSL 4
#endif

template <int K, int V>
using LaneFwd = LanePlan<LCfg<K, V, false, MG_AFL_NW, MG_AFL_L, MG_AFL_NSL>>;
template <int K, int V>
using LaneBwd = LanePlan<LCfg<K, V, true, MG_AFLB_NW, MG_AFLB_L, MG_AFLB_NSL>>;
template <int K, int V>
using SmallFwd = ChanPlan<AffFwdSmall<K, V, MG_AFS_L>, 32, MG_AFS_TY, MG_AFS_MB>;
template <int K, int V>
using SmallBwd = ChanPlan<AffBwdSmall<K, V, MG_AFSB_L>, 32, MG_AFSB_TY, MG_AFSB_MB>;
#ifndef MG_AFC_NW
#define MG_AFC_NW 4
#endif
#ifndef MG_AFC_L
#define MG_AFC_L 16
#endif
#ifndef MG_AFC_NSL
#define MG_AFC_NSL 4
#endif
#ifndef MG_AFCB_NW
#define MG_AFCB_NW 4
#endif
#ifndef MG_AFCB_L
#define MG_AFCB_L 16
#endif
#ifndef MG_AFCB_NSL
#define MG_AFCB_NSL 3
#endif

#ifndef MG_AFM_NW
#define MG_AFM_NW 4
#endif
#ifndef MG_AFM_L
#define MG_AFM_L 32
#endif
#ifndef MG_AFM_NSL
#define MG_AFM_NSL 4
#endif
#ifndef MG_AFMB_NW
#define MG_AFMB_NW 4
#endif
#ifndef MG_AFMB_L
#define MG_AFMB_L 16
#endif
#ifndef MG_AFMB_NSL
#define MG_AFMB_NSL 2
#endif

// k = 16 with v in {8, 16}: the tensor-core state; other k in {8, 16}: the
// column kernel.
template <int K, int V>
constexpr bool mma_state_ok() { return K == 16 && (V == 8 || V == 16); }
template <int K, int V, bool BWD>
struct BigSel {
    using type = ColPlan<CCfg<K, V, BWD, BWD ? MG_AFCB_NW : MG_AFC_NW, BWD ? MG_AFCB_L : MG_AFC_L,
                              BWD ? MG_AFCB_NSL : MG_AFC_NSL>>;
};
template <int V, bool BWD>
struct BigSel<16, V, BWD> {
    using type = std::conditional_t<
        mma_state_ok<16, V>(),
        MmaPlan<MCfg<(V == 8 || V == 16) ? V : 16, BWD, BWD ? MG_AFMB_NW : MG_AFM_NW,
                     BWD ? MG_AFMB_L : MG_AFM_L, BWD ? MG_AFMB_NSL : MG_AFM_NSL>>,
        ColPlan<CCfg<16, V, BWD, BWD ? MG_AFCB_NW : MG_AFC_NW, BWD ? MG_AFCB_L : MG_AFC_L,
                     BWD ? MG_AFCB_NSL : MG_AFC_NSL>>>;
};

template <int K, int V>
using BigFwd = typename BigSel<K, V, false>::type;
template <int K, int V>
using BigBwd = typename BigSel<K, V, true>::type;

// k <= 4: the lane kernel where its blocks are 16 to 128 bytes, the chunk
// engine otherwise; k in {8, 16}: the warp kernel.
template <int K, int V>
size_t ws_kv(int64_t B, int64_t T, int64_t n)
{
    size_t a, b;
    if constexpr (K <= 4) {
        if constexpr (lane_kernel_ok<K, V>()) {
            a = LaneFwd<K, V>::ws_bytes(B, T, n);
            b = LaneBwd<K, V>::ws_bytes(B, T, n);
        } else {
            a = SmallFwd<K, V>::ws_bytes(B, T, n);
            b = SmallBwd<K, V>::ws_bytes(B, T, n);
        }
    } else {
        a = BigFwd<K, V>::ws_bytes(B, T, n);
        b = BigBwd<K, V>::ws_bytes(B, T, n);
    }
    return a > b ? a : b;
}

template <int K, int V>
mg_status fwd_kv(const float *A, const float *Bm, const float *H0, float *Abar, float *Bbar,
                 int64_t B, int64_t T, int64_t n, void *ws, size_t wsb, cudaStream_t s,
                 const LaunchOpts &o)
{
    const char *nm = H0 ? "mg_affine_scan_h0_fwd" : "mg_affine_scan_fwd";
    if constexpr (K <= 4) {
        if constexpr (lane_kernel_ok<K, V>())
            return LaneFwd<K, V>::launch({A, Bm, Abar, Bbar, H0}, B, T, n, ws, wsb, s, o, nm);
        else
            return SmallFwd<K, V>::launch({A, Bm, Abar, Bbar, H0}, B, T, n, ws, wsb, s, o, nm);
    } else {
        AffPtrs p{};
        p.A = A;
        p.Bm = Bm;
        p.H0 = H0;
        p.Abar_out = Abar;
        p.Bbar_out = Bbar;
        return BigFwd<K, V>::launch(p, B, T, n, ws, wsb, s, o, nm);
    }
}

template <int K, int V>
mg_status bwd_kv(const float *A, const float *Abar, const float *Bbar, const float *gAbar,
                 const float *gBbar, float *dA, float *dB, int64_t B, int64_t T, int64_t n,
                 void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
    const char *nm = "mg_affine_scan_bwd";
    if constexpr (K <= 4) {
        if constexpr (lane_kernel_ok<K, V>())
            return LaneBwd<K, V>::launch({A, Abar, Bbar, gAbar, gBbar, dA, dB}, B, T, n, ws, wsb,
                                         s, o, nm);
        else
            return SmallBwd<K, V>::launch({A, Abar, Bbar, gAbar, gBbar, dA, dB}, B, T, n, ws, wsb,
                                          s, o, nm);
    } else {
        AffPtrs p{};
        p.A = A;
        p.Abar = Abar;
        p.Bbar = Bbar;
        p.gAbar = gAbar;
        p.gBbar = gBbar;
        p.dA = dA;
        p.dB = dB;
        return BigBwd<K, V>::launch(p, B, T, n, ws, wsb, s, o, nm);
    }
}

// The backward from a start state H0 differs from the H0 = 0 one only at the
// first step (the forward's Bbar, passed in, already carries H0 at every
// later step): dA_1 gains Lam_1 H0^T (Bbar_0 = H0), and dH0 = A_1^T Lam_1,
// with Lam_1 = dB_1.  One thread per output element (k*k of dA_1 and k*v of
// dH0 per sequence), each a dot product of length v or k, after the main
// backward on the same stream.
template <int K, int V>
__global__ void affine_h0_grad_kernel(const float *A, const float *H0, const float *dB, float *dA,
                                      float *dH0, int64_t B, int64_t T, int64_t n)
{
    constexpr int KK = K * K, KV = K * V, PER = KK + KV;
    const int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (q >= B * n * PER) return;
    const int64_t sq = q / PER;          // sequence (b, n)
    const int e = int(q % PER);
    const int64_t bb = sq / n, nn = sq % n;
    const int64_t s1 = (bb * T) * n + nn;   // its first step
    const float *lam = dB + s1 * KV;
    if (e < KK) {   // dA_1[i][j] += sum_l Lam_1[i][l] H0[j][l]
        const int i = e / K, j = e % K;
        const float *h = H0 + sq * KV;
        float acc = dA[s1 * KK + e];
#pragma unroll
        for (int l = 0; l < V; ++l) acc = fmaf(lam[i * V + l], h[j * V + l], acc);
        dA[s1 * KK + e] = acc;
    } else {        // dH0[i][l] = sum_j A_1[j][i] Lam_1[j][l]
        const int i = (e - KK) / V, l = (e - KK) % V;
        const float *a1 = A + s1 * KK;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) acc = fmaf(a1[j * K + i], lam[j * V + l], acc);
        dH0[sq * KV + i * V + l] = acc;
    }
}

template <int K, int V>
mg_status h0_grad_kv(const float *A, const float *H0, const float *dB, float *dA, float *dH0,
                     int64_t B, int64_t T, int64_t n, cudaStream_t s)
{
    const int64_t nq = B * n * (K * K + K * V);
    const unsigned blocks = unsigned((nq + 255) / 256);
    affine_h0_grad_kernel<K, V><<<blocks, 256, 0, s>>>(A, H0, dB, dA, dH0, B, T, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MG_ERR_LAUNCH, "mg_affine_scan_h0_bwd: launch failed: %s", cudaGetErrorString(e));
    return MG_OK;
}

// Expand CALL(K, V) for the runtime (k, v) in {1,2,4,8,16}^2.
#define MG_KV_DISPATCH(k, v, CALL)                                                        \
    switch ((k) * 32 + (v)) {                                                             \
    case 1 * 32 + 1: CALL(1, 1); case 1 * 32 + 2: CALL(1, 2); case 1 * 32 + 4: CALL(1, 4);    \
    case 1 * 32 + 8: CALL(1, 8); case 1 * 32 + 16: CALL(1, 16);                             \
    case 2 * 32 + 1: CALL(2, 1); case 2 * 32 + 2: CALL(2, 2); case 2 * 32 + 4: CALL(2, 4);    \
    case 2 * 32 + 8: CALL(2, 8); case 2 * 32 + 16: CALL(2, 16);                             \
    case 4 * 32 + 1: CALL(4, 1); case 4 * 32 + 2: CALL(4, 2); case 4 * 32 + 4: CALL(4, 4);    \
    case 4 * 32 + 8: CALL(4, 8); case 4 * 32 + 16: CALL(4, 16);                             \
    case 8 * 32 + 1: CALL(8, 1); case 8 * 32 + 2: CALL(8, 2); case 8 * 32 + 4: CALL(8, 4);    \
    case 8 * 32 + 8: CALL(8, 8); case 8 * 32 + 16: CALL(8, 16);                             \
    case 16 * 32 + 1: CALL(16, 1); case 16 * 32 + 2: CALL(16, 2);                          \
    case 16 * 32 + 4: CALL(16, 4); case 16 * 32 + 8: CALL(16, 8);                          \
    case 16 * 32 + 16: CALL(16, 16);                                                      \
    default: break;                                                                       \
    }

}  // namespace

size_t affine_ws_bytes(int64_t B, int64_t T, int64_t n, int k, int v)
{
#define MG_CALL(K, V) return ws_kv<K, V>(B, T, n)
    MG_KV_DISPATCH(k, v, MG_CALL)
#undef MG_CALL
    return 0;
}

mg_status launch_affine_fwd(const float *A, const float *Bm, const float *H0, float *Abar,
                            float *Bbar, int64_t B, int64_t T, int64_t n, int k, int v, void *ws,
                            size_t wsb, cudaStream_t s, const LaunchOpts &o)
{
#define MG_CALL(K, V) return fwd_kv<K, V>(A, Bm, H0, Abar, Bbar, B, T, n, ws, wsb, s, o)
    MG_KV_DISPATCH(k, v, MG_CALL)
#undef MG_CALL
    return fail(MG_ERR_UNSUPPORTED, "mg_affine_scan_fwd: k=%d v=%d outside {1,2,4,8,16}", k, v);
}

mg_status launch_affine_h0_grad(const float *A, const float *H0, const float *dB, float *dA,
                                float *dH0, int64_t B, int64_t T, int64_t n, int k, int v,
                                cudaStream_t s)
{
#define MG_CALL(K, V) return h0_grad_kv<K, V>(A, H0, dB, dA, dH0, B, T, n, s)
    MG_KV_DISPATCH(k, v, MG_CALL)
#undef MG_CALL
    return fail(MG_ERR_UNSUPPORTED, "mg_affine_scan_h0_bwd: k=%d v=%d outside {1,2,4,8,16}", k, v);
}

mg_status launch_affine_bwd(const float *A, const float *Abar, const float *Bbar,
                            const float *gAbar, const float *gBbar, float *dA, float *dB,
                            int64_t B, int64_t T, int64_t n, int k, int v, void *ws, size_t wsb,
                            cudaStream_t s, const LaunchOpts &o)
{
#define MG_CALL(K, V) return bwd_kv<K, V>(A, Abar, Bbar, gAbar, gBbar, dA, dB, B, T, n, ws, wsb, s, o)
    MG_KV_DISPATCH(k, v, MG_CALL)
#undef MG_CALL
    return fail(MG_ERR_UNSUPPORTED, "mg_affine_scan_bwd: k=%d v=%d outside {1,2,4,8,16}", k, v);
}

}  // namespace mg

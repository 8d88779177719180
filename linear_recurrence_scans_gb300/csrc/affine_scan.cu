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
//   * k in {8, 16}: one warp owns one sequence's sub-chunk of L steps; the
//     state X = [C | V] (k x (k + w), padded to a multiple of 8 columns) is
//     split into 4 row blocks x 8 column blocks, one per lane.  Each step
//     X <- E_C X + [0 | E_V] reads the column strip of X that the lane needs
//     from a shared copy and the lane's rows of E_C from the warp's ring of
//     bulk copies (affine_warp_kernel below).  A CTA of NW warps covers NW*L
//     consecutive steps of one sequence.
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

template <int N>
__device__ __forceinline__ void st_floats(float *p, const float *x)
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q)
            *reinterpret_cast<float4 *>(p + 4 * q) =
                make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int q = 0; q < N / 2; ++q)
            *reinterpret_cast<float2 *>(p + 2 * q) = make_float2(x[2 * q], x[2 * q + 1]);
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) p[q] = x[q];
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
        publish_first<Op, 32>(args, g, lb, c, j, bb, d, true, act, tile, epoch, cta);
        excl = find_carry<Op, 32>(args, g, lb, c, j, bb, d, true, act, tile, epoch);
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
        return tiled_ws_bytes(n_tiles(B, T, n), size_t(2) * Cf::NS * 32 * sizeof(float));
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

// ============================================================ k in {8, 16}

template <int K_, int W_, bool BWD_, int NW_, int L_, bool DB_, int NSL_>
struct WCfg {
    static constexpr int K = K_, W = W_, NW = NW_, L = L_, NSL = NSL_;
    static constexpr bool BWD = BWD_, DB = DB_;  // DB: double-buffered state exchange
    static constexpr int VV = BWD ? W - K : W;  // v
    static constexpr int KK = K * K, KV = K * VV;
    static constexpr int NC = K + W;            // columns of X = [C | V]
    static constexpr int NCP = (NC + 7) / 8 * 8;
    static constexpr int R = K / 4;             // rows per lane (4 row blocks)
    static constexpr int CC = NCP / 8;          // columns per lane (8 column blocks)
    static constexpr int XS = NCP;              // shared row stride (floats)
    static constexpr int MAT = K * XS;          // floats per shared state matrix
    static constexpr int REC = K * NC;          // floats per global record
    static constexpr int TC = NW * L;           // steps per tile (L per warp)
    static constexpr int JD = K / 8;            // dA columns per lane (8 column blocks)
    // One ring slot holds the inputs of one step.  Forward: A_t, B_t.
    // Backward: A_{t+1}, gAbar_t, gBbar_t, Abar_{t-1}, Bbar_{t-1}.  Each block
    // is a multiple of 16 bytes.
    static constexpr int STEP = BWD ? 3 * KK + 2 * KV : KK + KV;
    static constexpr int OFF_G = KK, OFF_GB = 2 * KK, OFF_AP = 2 * KK + KV, OFF_BP = 3 * KK + KV;
    static constexpr int NXB = DB ? 2 : 1;
    static constexpr int BAR_FLOATS = (NW * NSL * 2 + 3) / 4 * 4;  // mbarriers, 16-byte padded
    static constexpr size_t SMEM = size_t(BAR_FLOATS + NW * NSL * STEP) * sizeof(float) +
                                   size_t((NXB + 1) * NW + 1) * MAT * sizeof(float);
    static_assert(K == 8 || K == 16, "warp kernel is for k in {8, 16}");
    static_assert(NSL >= 2, "the ring needs two slots at least");
    static_assert((KV * 4) % 16 == 0 && (KK * 4) % 16 == 0, "bulk copies need 16-byte blocks");
};

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

// Lane block of the combine (x earlier, full matrix in shared memory) o
// (y later, rows `yc` = y.C[rows][0..K) and `yv` = y.V on the lane's columns).
template <class Cf>
__device__ __forceinline__ void block_gemm(const float *xs, const float (&yc)[Cf::R][Cf::K],
                                           const float (&yv)[Cf::R][Cf::CC], int cb,
                                           float (&o)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r)
#pragma unroll
        for (int c = 0; c < Cf::CC; ++c) o[r][c] = yv[r][c];
#pragma unroll
    for (int l = 0; l < Cf::K; ++l) {
        float xv[Cf::CC];
        ld_floats<Cf::CC>(xs + l * Cf::XS + cb * Cf::CC, xv);
#pragma unroll
        for (int r = 0; r < Cf::R; ++r)
#pragma unroll
            for (int c = 0; c < Cf::CC; ++c) o[r][c] = fmaf(yc[r][l], xv[c], o[r][c]);
    }
}

// y operand from a matrix stored with row stride `ld` (shared or global):
// C part = columns 0..K-1, V part on the lane's columns (zero outside [K, NC)).
template <class Cf, bool GLOBAL>
__device__ __forceinline__ void load_y(const float *m, int ld, int rb, int cb,
                                       float (&yc)[Cf::R][Cf::K], float (&yv)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r) {
        const float *row = m + (rb * Cf::R + r) * ld;
#pragma unroll
        for (int l = 0; l < Cf::K; ++l) yc[r][l] = GLOBAL ? __ldcg(row + l) : row[l];
#pragma unroll
        for (int c = 0; c < Cf::CC; ++c) {
            const int col = cb * Cf::CC + c;
            yv[r][c] = (col >= Cf::K && col < Cf::NC) ? (GLOBAL ? __ldcg(row + col) : row[col]) : 0.f;
        }
    }
}

// The element held in a ring slot as a y operand.  `has_next`: step t+1
// exists (the adjoint's coefficient A_{t+1}^T is zero at t = T-1).
template <class Cf>
__device__ __forceinline__ void load_elem(const float *slot, bool has_next, int rb, int cb,
                                          float (&yc)[Cf::R][Cf::K], float (&yv)[Cf::R][Cf::CC])
{
    constexpr int K = Cf::K, KK = Cf::KK, VV = Cf::VV, R = Cf::R;
    if constexpr (!Cf::BWD) {
        const float *At = slot;
        const float *Bt = slot + KK;
#pragma unroll
        for (int r = 0; r < R; ++r) ld_floats<K>(At + (rb * R + r) * K, yc[r]);
        if constexpr (K % Cf::CC == 0 && VV % Cf::CC == 0) {
            // a lane's columns lie wholly in the C part (zero) or in B_t
            const int col = cb * Cf::CC;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (col >= K) {
                    ld_floats<Cf::CC>(Bt + (rb * R + r) * VV + col - K, yv[r]);
                } else {
#pragma unroll
                    for (int c = 0; c < Cf::CC; ++c) yv[r][c] = 0.f;
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < Cf::CC; ++c) {
                    const int col = cb * Cf::CC + c;
                    yv[r][c] = (col >= K && col < Cf::NC) ? Bt[(rb * R + r) * VV + col - K] : 0.f;
                }
        }
    } else {
        const float *An = slot;
        const float *ga = slot + Cf::OFF_G;
        const float *gb = slot + Cf::OFF_GB;
        if (has_next) {  // E_C[row][l] = A_{t+1}[l][row]
#pragma unroll
            for (int l = 0; l < K; ++l) {
                float a[R];
                ld_floats<R>(An + l * K + rb * R, a);
#pragma unroll
                for (int r = 0; r < R; ++r) yc[r][l] = a[r];
            }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int l = 0; l < K; ++l) yc[r][l] = 0.f;
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < Cf::CC; ++c) {
                const int col = cb * Cf::CC + c, row = rb * R + r;
                float x = 0.f;
                if (col >= K && col < 2 * K) x = ga[row * K + col - K];
                else if (col >= 2 * K && col < Cf::NC) x = gb[row * VV + col - 2 * K];
                yv[r][c] = x;
            }
    }
}

template <class Cf>
__device__ __forceinline__ void identity_block(int rb, int cb, float (&o)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r)
#pragma unroll
        for (int c = 0; c < Cf::CC; ++c) o[r][c] = (rb * Cf::R + r == cb * Cf::CC + c) ? 1.f : 0.f;
}

template <class Cf>
__device__ __forceinline__ void put_block_smem(float *xs, int rb, int cb,
                                               const float (&o)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r) st_floats<Cf::CC>(xs + (rb * Cf::R + r) * Cf::XS + cb * Cf::CC, o[r]);
}

template <class Cf>
__device__ __forceinline__ void put_block_record(float *rec, int rb, int cb,
                                                 const float (&o)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r)
#pragma unroll
        for (int c = 0; c < Cf::CC; ++c) {
            const int col = cb * Cf::CC + c;
            if (col < Cf::NC) __stcg(rec + (rb * Cf::R + r) * Cf::NC + col, o[r][c]);
        }
}

template <class Cf>
__device__ __forceinline__ void get_block_record(const float *rec, int rb, int cb,
                                                 float (&o)[Cf::R][Cf::CC])
{
#pragma unroll
    for (int r = 0; r < Cf::R; ++r)
#pragma unroll
        for (int c = 0; c < Cf::CC; ++c) {
            const int col = cb * Cf::CC + c;
            o[r][c] = col < Cf::NC ? __ldcg(rec + (rb * Cf::R + r) * Cf::NC + col) : 0.f;
        }
}

// One step of a warp's scan: o <- E o X + [0 | E_V] with X read from the warp's
// shared state buffer(s), then the new X written back.  `cur` selects the
// buffer holding X (double-buffered) and is advanced.
template <class Cf>
__device__ __forceinline__ void warp_step(float *xw, int &cur, const float (&yc)[Cf::R][Cf::K],
                                          const float (&yv)[Cf::R][Cf::CC], int rb, int cb,
                                          float (&o)[Cf::R][Cf::CC])
{
    if constexpr (Cf::DB) {
        block_gemm<Cf>(xw + cur * Cf::MAT, yc, yv, cb, o);
        cur ^= 1;
        put_block_smem<Cf>(xw + cur * Cf::MAT, rb, cb, o);
        __syncwarp();
    } else {
        block_gemm<Cf>(xw, yc, yv, cb, o);
        __syncwarp();
        put_block_smem<Cf>(xw, rb, cb, o);
        __syncwarp();
    }
}

// ------------------------------------------------ dA_t on the tensor cores
// dA_t = Xv Y^T with Xv = [M_t | Lam_t] (16 x W) and Y = [Abar_{t-1} |
// Bbar_{t-1}] (16 x W), W = 16 + v: an independent product per step (no
// recurrence runs through it), done as mma.sync.m16n8k8 tf32 tiles (M = 16,
// N = 16, K = W).  Each fp32 operand is split into a tf32 high part and a
// tf32 remainder and the products hi*hi, hi*lo, lo*hi are accumulated in
// fp32: the dropped lo*lo term is below 2^-22 of each product.

#ifndef MG_AFW_MMA_DA
#define MG_AFW_MMA_DA 1
#endif

__device__ __forceinline__ void split_tf32(float x, unsigned &hi, unsigned &lo)
{
    unsigned h, l;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
    const float rem = x - __uint_as_float(h);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(rem));
    hi = h;
    lo = l;
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

// xs: X rows with stride XS (Xv = columns 16 .. 16+W-1); ap, bp: Abar_{t-1}
// (16 x 16) and Bbar_{t-1} (16 x V) row-major; writes dA (16 x 16) at `out`.
template <int XS, int V>
__device__ __forceinline__ void mma_dA16(const float *xs, const float *ap, const float *bp,
                                         int lane, float *out)
{
    constexpr int W = 16 + V, NKT = W / 8;
    const int g = lane >> 2, q = lane & 3;
    float d[2][4] = {};
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt) {
        unsigned ah[4], al[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            split_tf32(xs[(g + 8 * (e & 1)) * XS + 16 + 8 * kt + q + 4 * (e >> 1)], ah[e], al[e]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            unsigned bh[2], bl[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {  // B[k][n] = Y[n][k]
                const int n = 8 * nt + g, k = 8 * kt + q + 4 * e;
                split_tf32(k < 16 ? ap[n * 16 + k] : bp[n * V + k - 16], bh[e], bl[e]);
            }
            mma_tf32(d[nt], al, bh[0], bh[1]);
            mma_tf32(d[nt], ah, bl[0], bl[1]);
            mma_tf32(d[nt], ah, bh[0], bh[1]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<float2 *>(out + (g + 8 * h) * 16 + 8 * nt + 2 * q) =
                make_float2(d[nt][2 * h], d[nt][2 * h + 1]);
}

// One tile = one sequence x TC steps, warp w owning L consecutive steps.
// Each warp streams its steps through its own ring of NSL slots (1D bulk
// copies completing on one mbarrier per slot): pass 1 folds them into the
// warp's aggregate, pass 2 streams them again (now from L2) and writes the
// outputs.  Both passes form one issue sequence, so the first loads of pass 2
// are in flight while warp 0 does the look-back.
template <class Cf>
__global__ void __launch_bounds__(Cf::NW * 32)
    affine_warp_kernel(const AffPtrs p, const AffGeom g, const Lookback lb)
{
    constexpr int K = Cf::K, R = Cf::R, CC = Cf::CC, NW = Cf::NW, L = Cf::L, MAT = Cf::MAT;
    constexpr int XS = Cf::XS, NC = Cf::NC, VV = Cf::VV, KK = Cf::KK, KV = Cf::KV;
    constexpr int NSL = Cf::NSL, STEP = Cf::STEP;
    extern __shared__ float4 aff_smem[];
    unsigned long long *const bars = reinterpret_cast<unsigned long long *>(aff_smem);  // [NW][NSL]
    float *const ring = reinterpret_cast<float *>(aff_smem) + Cf::BAR_FLOATS;          // [NW][NSL][STEP]
    float *const xb = ring + NW * NSL * STEP;                                          // [NW][NXB][MAT]
    float *const G = xb + NW * Cf::NXB * MAT;                                          // [NW][MAT]
    float *const carry = G + NW * MAT;                                                 // [MAT]

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
    const int rb = lane >> 3, cb = lane & 7;
    const int ct = Cf::BWD ? (g.nC - 1 - c) : c;
    const int64_t t0 = int64_t(ct) * Cf::TC;        // first step of the tile
    const int nv = int(g.T - t0 < Cf::TC ? g.T - t0 : Cf::TC);  // valid steps in the tile
    const int wbase = warp * L;                     // first tile step of this warp
    const int nvw = nv - wbase < 0 ? 0 : (nv - wbase < L ? nv - wbase : L);  // its valid steps
    const int pw = Cf::BWD ? NW - 1 - warp : warp;  // position in processing order
    float *const xw = xb + warp * Cf::NXB * MAT;
    unsigned long long *const wbar = bars + warp * NSL;
    float *const wring = ring + warp * NSL * STEP;
    auto step_index = [&](int64_t t) { return (bb * g.T + t) * g.n + nn; };
    // issue-sequence entry q: pass 1 for q < nvw, pass 2 after; the tile step
    // in processing order (reverse time for the adjoint)
    auto tile_step = [&](int q) {
        const int k = q < nvw ? q : q - nvw;
        return Cf::BWD ? wbase + nvw - 1 - k : wbase + k;
    };
    const int nq = 2 * nvw;

    // lane 0 of each warp: arm slot q % NSL and start its copies
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
    // every lane: wait for entry q (bounded; a second bounded wait after a
    // timeout lets the copies land before the slot is reused or the CTA ends)
    auto wait_slot = [&](int q) -> const float * {
        unsigned long long *bar = wbar + q % NSL;
        const unsigned parity = unsigned(q / NSL) & 1u;
        if (!mbar_wait_bounded(bar, parity, lb.wait_limit_ns)) {
            if (lane == 0) raise_error(lb, epoch, kErrLookbackTimeout);
            mbar_wait_bounded(bar, parity, lb.wait_limit_ns);
        }
        return wring + (q % NSL) * STEP;
    };

    if (lane == 0) {
        for (int q = 0; q < NSL; ++q) mbar_init(wbar + q, 1);
        for (int q = 0; q < NSL; ++q) issue(q);
    }
    __syncwarp();
    auto refill = [&](int q) {  // after every lane has read entry q - NSL
        if (lane == 0) issue(q);
    };

    float yc[R][K], yv[R][CC], o[R][CC];

    // ---- pass 1: aggregate of the warp's steps, in processing order
    int cur = 0;
    {
        identity_block<Cf>(rb, cb, o);
        put_block_smem<Cf>(xw, rb, cb, o);
        __syncwarp();
#pragma unroll 1
        for (int q = 0; q < nvw; ++q) {
            const int64_t t = t0 + tile_step(q);
            const float *slot = wait_slot(q);
            load_elem<Cf>(slot, t + 1 < g.T, rb, cb, yc, yv);
            __syncwarp();  // every lane has read the slot
            refill(q + NSL);
            warp_step<Cf>(xw, cur, yc, yv, rb, cb, o);
        }
        put_block_smem<Cf>(G + pw * MAT, rb, cb, o);
    }
    __syncthreads();

    // ---- warp 0: inclusive prefixes over the warps (processing order), then
    //      the look-back for the tile's carry-in
    if (warp == 0) {
        for (int w = 1; w < NW; ++w) {  // G[w] <- G[w-1] o G[w]
            load_y<Cf, false>(G + w * MAT, XS, rb, cb, yc, yv);
            block_gemm<Cf>(G + (w - 1) * MAT, yc, yv, cb, o);
            __syncwarp();
            put_block_smem<Cf>(G + w * MAT, rb, cb, o);
            __syncwarp();
        }
        const float *cta = G + (NW - 1) * MAT;
        const size_t slot = size_t(c) * g.nJ + j;
        float *rec_agg = lb.data + slot * 2 * Cf::REC;
        float *rec_pre = rec_agg + Cf::REC;
        float cblk[R][CC];
#pragma unroll
        for (int r = 0; r < R; ++r) ld_floats<CC>(cta + (rb * R + r) * XS + cb * CC, cblk[r]);
        if (c == 0) {
            if (!Cf::BWD && p.H0 != nullptr) {
                // carry = the start state [I | H0]; prefix = carry o cta
                const float *h0 = p.H0 + (bb * g.n + nn) * KV;
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int cc = 0; cc < CC; ++cc) {
                        const int row = rb * R + r, col = cb * CC + cc;
                        o[r][cc] = col < K ? (row == col ? 1.f : 0.f)
                                           : (col < NC ? h0[row * VV + col - K] : 0.f);
                    }
                put_block_smem<Cf>(carry, rb, cb, o);
                __syncwarp();
                load_y<Cf, false>(cta, XS, rb, cb, yc, yv);
                block_gemm<Cf>(carry, yc, yv, cb, o);
                put_block_record<Cf>(rec_pre, rb, cb, o);
                publish(lb, slot, kStatusPrefix, epoch, tile);
            } else {
                put_block_record<Cf>(rec_pre, rb, cb, cblk);
                publish(lb, slot, kStatusPrefix, epoch, tile);
                identity_block<Cf>(rb, cb, o);
                put_block_smem<Cf>(carry, rb, cb, o);
            }
        } else {
            if (peek_status(lb, slot - g.nJ, epoch) != kStatusPrefix) {
                put_block_record<Cf>(rec_agg, rb, cb, cblk);
                publish(lb, slot, kStatusAggregate, epoch, tile);
            }
            const int pp = wait_window(lb, size_t(j), size_t(g.nJ), c, epoch, tile);
            if (pp >= 0) {
                get_block_record<Cf>(lb.data + (size_t(pp) * g.nJ + j) * 2 * Cf::REC + Cf::REC, rb,
                                     cb, o);
            } else {
                identity_block<Cf>(rb, cb, o);
            }
            put_block_smem<Cf>(carry, rb, cb, o);
            __syncwarp();
            if (pp >= 0) {
                for (int q = pp + 1; q < c; ++q) {  // carry <- carry o agg(q)
                    load_y<Cf, true>(lb.data + (size_t(q) * g.nJ + j) * 2 * Cf::REC, NC, rb, cb,
                                     yc, yv);
                    block_gemm<Cf>(carry, yc, yv, cb, o);
                    __syncwarp();
                    put_block_smem<Cf>(carry, rb, cb, o);
                    __syncwarp();
                }
            }
            // prefix of this tile = carry o cta
            load_y<Cf, false>(cta, XS, rb, cb, yc, yv);
            block_gemm<Cf>(carry, yc, yv, cb, o);
            put_block_record<Cf>(rec_pre, rb, cb, o);
            publish(lb, slot, kStatusPrefix, epoch, tile);
        }
    }
    __syncthreads();

    // ---- start state of this warp: carry o G[pw-1]
    if (pw == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) ld_floats<CC>(carry + (rb * R + r) * XS + cb * CC, o[r]);
    } else {
        load_y<Cf, false>(G + (pw - 1) * MAT, XS, rb, cb, yc, yv);
        block_gemm<Cf>(carry, yc, yv, cb, o);
    }
    cur = 0;
    put_block_smem<Cf>(xw, rb, cb, o);
    __syncwarp();

    // ---- pass 2 of the k = 16 adjoint on [M | Lam] only: the running
    //      product C (the first 16 columns of X) feeds the aggregates of pass
    //      1 and no output, so pass 2 updates the W = 16 + v columns after it
    //      with C2 = W / 8 columns per lane.
    if constexpr (Cf::BWD && K == 16 && (K + VV) % 8 == 0 && MG_AFW_MMA_DA != 0) {
        constexpr int C2 = (K + VV) / 8, WV = K + VV;
#pragma unroll 1
        for (int q = nvw; q < nq; ++q) {
            const int64_t t = t0 + tile_step(q), s = step_index(t);
            const float *slot = wait_slot(q);
            // E rows (A_{t+1}^T) as in the full step; values [gA | gB] on the lane's columns
            if (t + 1 < g.T) {
#pragma unroll
                for (int l = 0; l < K; ++l) {
                    float a[R];
                    ld_floats<R>(slot + l * K + rb * R, a);
#pragma unroll
                    for (int r = 0; r < R; ++r) yc[r][l] = a[r];
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int l = 0; l < K; ++l) yc[r][l] = 0.f;
            }
            float y2[R][C2], o2[R][C2];
            const int col0 = cb * C2;  // in [M | Lam]
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rb * R + r;
                if constexpr (C2 == 4) {
                    if (col0 < K) ld_floats<4>(slot + Cf::OFF_G + row * K + col0, y2[r]);
                    else ld_floats<4>(slot + Cf::OFF_GB + row * VV + col0 - K, y2[r]);
                } else {
#pragma unroll
                    for (int c = 0; c < C2; ++c) {
                        const int j = col0 + c;
                        y2[r][c] = j < K ? slot[Cf::OFF_G + row * K + j] : slot[Cf::OFF_GB + row * VV + j - K];
                    }
                }
            }
            // o2 = E [M | Lam] + [gA | gB] on the lane's block
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < C2; ++c) o2[r][c] = y2[r][c];
#pragma unroll
            for (int l = 0; l < K; ++l) {
                float xv[C2];
                ld_floats<C2>(xw + l * XS + K + col0, xv);
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int c = 0; c < C2; ++c) o2[r][c] = fmaf(yc[r][l], xv[c], o2[r][c]);
            }
            __syncwarp();  // every lane has read X
#pragma unroll
            for (int r = 0; r < R; ++r) st_floats<C2>(xw + (rb * R + r) * XS + K + col0, o2[r]);
            __syncwarp();
            // dB_t = Lam_t
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rb * R + r;
                if constexpr (C2 == 4) {
                    if (col0 >= K) st_floats<4>(p.dB + s * KV + row * VV + col0 - K, o2[r]);
                } else {
#pragma unroll
                    for (int c = 0; c < C2; ++c)
                        if (col0 + c >= K) p.dB[s * KV + row * VV + col0 + c - K] = o2[r][c];
                }
            }
            // dA_t = M_t Abar_{t-1}^T + Lam_t Bbar_{t-1}^T  (Abar_0 = I, Bbar_0 = 0)
            if (t > 0) {
                mma_dA16<XS, VV>(xw, slot + Cf::OFF_AP, slot + Cf::OFF_BP, lane, p.dA + s * KK);
            } else {
#pragma unroll
                for (int e = 0; e < KK / 32; ++e) {
                    const int idx = lane + 32 * e, a = idx / K, b2 = idx % K;
                    p.dA[s * KK + idx] = xw[a * XS + K + b2];
                }
            }
            (void)WV;
            __syncwarp();  // the slot and xw are read by every lane before reuse
            refill(q + NSL);
        }
        finish_cta(lb, epoch);
        return;
    }

    // ---- pass 2: re-run the warp's steps from its start state, write outputs
#pragma unroll 1
    for (int q = nvw; q < nq; ++q) {
        const int64_t t = t0 + tile_step(q), s = step_index(t);
        const float *slot = wait_slot(q);
        load_elem<Cf>(slot, t + 1 < g.T, rb, cb, yc, yv);
        if constexpr (!Cf::BWD) {
            __syncwarp();  // every lane has read the slot
            refill(q + NSL);
        }
        warp_step<Cf>(xw, cur, yc, yv, rb, cb, o);
        if constexpr (!Cf::BWD) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rb * R + r;
                if constexpr (CC % 4 == 0 && K % 4 == 0 && VV % 4 == 0) {
#pragma unroll
                    for (int qq = 0; qq < CC; qq += 4) {
                        const int col = cb * CC + qq;
                        float v4[4] = {o[r][qq], o[r][qq + 1], o[r][qq + 2], o[r][qq + 3]};
                        if (col < K) st_floats<4>(p.Abar_out + s * KK + row * K + col, v4);
                        else if (col < NC) st_floats<4>(p.Bbar_out + s * KV + row * VV + col - K, v4);
                    }
                } else {
#pragma unroll
                    for (int cc = 0; cc < CC; ++cc) {
                        const int col = cb * CC + cc;
                        if (col < K) p.Abar_out[s * KK + row * K + col] = o[r][cc];
                        else if (col < NC) p.Bbar_out[s * KV + row * VV + col - K] = o[r][cc];
                    }
                }
            }
        } else {
            // dB_t = Lam_t (columns 2K .. NC of X)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int cc = 0; cc < CC; ++cc) {
                    const int col = cb * CC + cc, row = rb * R + r;
                    if (col >= 2 * K && col < NC) p.dB[s * KV + row * VV + col - 2 * K] = o[r][cc];
                }
            // dA_t[row][jc] = sum_q X[row][K + q] * Y[jc][q],  Y = [Abar_{t-1} | Bbar_{t-1}]
            constexpr int JD = Cf::JD, WW = Cf::W;
            const float *xs = xw + (Cf::DB ? cur * MAT : 0);
            const float *Ap = slot + Cf::OFF_AP;
            const float *Bp = slot + Cf::OFF_BP;
            if constexpr (MG_AFW_MMA_DA != 0 && K == 16 && VV % 8 == 0) {
                if (t > 0) {
                    mma_dA16<XS, VV>(xs, Ap, Bp, lane, p.dA + s * KK);
                    __syncwarp();  // the slot and xw are read by every lane before reuse
                    refill(q + NSL);
                    continue;
                }
            }
            // the JD rows of Y first, then each row of X once
            float y[JD][WW];
#pragma unroll
            for (int jj = 0; jj < JD; ++jj) {
                const int jc = cb * JD + jj;
                if (t > 0) {
                    ld_floats<K>(Ap + jc * K, y[jj]);
                    ld_floats<VV>(Bp + jc * VV, y[jj] + K);
                } else {  // Abar_0 = I, Bbar_0 = 0
#pragma unroll
                    for (int qq = 0; qq < WW; ++qq) y[jj][qq] = (qq == jc) ? 1.f : 0.f;
                }
            }
            float da[R][JD];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float xr[WW];
                ld_floats<WW>(xs + (rb * R + r) * XS + K, xr);
#pragma unroll
                for (int jj = 0; jj < JD; ++jj) {
                    float acc = 0.f;
#pragma unroll
                    for (int qq = 0; qq < WW; ++qq) acc = fmaf(xr[qq], y[jj][qq], acc);
                    da[r][jj] = acc;
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
                st_floats<JD>(p.dA + s * KK + (rb * R + r) * K + cb * JD, da[r]);
            __syncwarp();  // the slot and xw are read by every lane before reuse
            refill(q + NSL);
        }
    }
    finish_cta(lb, epoch);
}

template <class Cf>
struct WarpPlan {
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
                affine_warp_kernel<Cf>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cf::SMEM));
            if (attr != cudaSuccess)
                return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        }
        affine_warp_kernel<Cf><<<unsigned(nt), Cf::NW * 32, Cf::SMEM, s>>>(p, g, lb);
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
#ifndef MG_AFW_NW
#define MG_AFW_NW 4
#endif
#ifndef MG_AFW_L
#define MG_AFW_L 16
#endif
#ifndef MG_AFW_DB
#define MG_AFW_DB 1
#endif
#ifndef MG_AFW_NSL
#define MG_AFW_NSL 5
#endif
#ifndef MG_AFWB_NW
#define MG_AFWB_NW 4
#endif
#ifndef MG_AFWB_L
#define MG_AFWB_L 16
#endif
#ifndef MG_AFWB_DB
#define MG_AFWB_DB 0
#endif
#ifndef MG_AFWB_NSL
#define MG_AFWB_NSL 2
#endif

template <int K, int V>
using LaneFwd = LanePlan<LCfg<K, V, false, MG_AFL_NW, MG_AFL_L, MG_AFL_NSL>>;
template <int K, int V>
using LaneBwd = LanePlan<LCfg<K, V, true, MG_AFLB_NW, MG_AFLB_L, MG_AFLB_NSL>>;
template <int K, int V>
using SmallFwd = ChanPlan<AffFwdSmall<K, V, MG_AFS_L>, 32, MG_AFS_TY, MG_AFS_MB>;
template <int K, int V>
using SmallBwd = ChanPlan<AffBwdSmall<K, V, MG_AFSB_L>, 32, MG_AFSB_TY, MG_AFSB_MB>;
template <int K, int V>
using BigFwd = WarpPlan<WCfg<K, V, false, MG_AFW_NW, MG_AFW_L, bool(MG_AFW_DB), MG_AFW_NSL>>;
template <int K, int V>
using BigBwd = WarpPlan<WCfg<K, K + V, true, MG_AFWB_NW, MG_AFWB_L, bool(MG_AFWB_DB), MG_AFWB_NSL>>;

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

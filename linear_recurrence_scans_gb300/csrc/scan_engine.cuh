// Generic chunked scan over time for independent "channels" (one state per
// channel), shared by the channel-wise ops and the small-matrix affine ops.
//
// An op supplies: NS floats of state per channel group of VEC channels, the
// identity, the combine (x earlier, y later), the initial state of chunk 0,
// how a thread loads L steps and forms their elements, and the epilogue
// that re-runs those steps from a start state, writes the outputs and leaves
// the state after the last step.  The engine does the rest: ticketed tiles of
// DC = TX*VEC channels by TC = TY*L*R steps (R rounds of L steps per thread),
// a shared-memory fold of the TY thread aggregates (which also leaves each
// row its exclusive prefix within the tile), the decoupled look-back of warp
// 0, and the hand-off of each thread's start state.  kReverse ops walk time
// backwards (adjoint scans).
#pragma once

#include "common.cuh"

namespace mg {
namespace {

struct ChanGeom {
    int64_t B, T, D;
    int nJb;  // channel tiles per batch row
    int nJ;   // channel tiles in total (B * nJb)
    int nC;   // chunks along time
    unsigned n_tiles;  // nJ * nC
};

template <int NS, int VEC>
struct St {
    float v[NS][VEC];
};

// An op may ask the engine to keep the elements that pass 1 forms in shared
// memory (static constexpr bool kStash = true): pass 2 then neither re-reads
// the op's inputs nor forms the elements again (for ops whose elements cost
// more to form than to keep).  Its pass 2 is epilogue_stash, which reads the
// round's elements through a StashView.  Layout: [round][step][state][thread]
// of VEC floats, so a warp's accesses to one (round, step, state) are one
// contiguous run of 32 * VEC floats (no bank conflicts).
template <class Op, class = void>
struct op_stashes {
    static constexpr bool value = false;
};
template <class Op>
struct op_stashes<Op, decltype(void(Op::kStash))> {
    static constexpr bool value = Op::kStash;
};

// Before publishing its aggregate, a tile may first look at its
// predecessor's flag and skip the aggregate when a prefix is already there
// (Op::kPeek, default on): one L2 round trip more on the tile's look-back
// path, one record store less.  Which wins depends on the op (measured).
#ifndef MG_LB_PEEK
#define MG_LB_PEEK 1
#endif
template <class Op, class = void>
struct op_peeks {
    static constexpr bool value = MG_LB_PEEK != 0;
};
template <class Op>
struct op_peeks<Op, decltype(void(Op::kPeek))> {
    static constexpr bool value = Op::kPeek;
};

template <class Op>
struct StashView {
    float *base;   // this thread's slot of step 0, state 0 of the round
    int nt;        // threads per CTA
    __device__ __forceinline__ float *at(int i, int q) const
    {
        return base + size_t(i * Op::NS + q) * nt * Op::VEC;
    }
    __device__ __forceinline__ void put(int i, const typename Op::S &e) const
    {
#pragma unroll
        for (int q = 0; q < Op::NS; ++q) store_vec<Op::VEC>(at(i, q), e.v[q]);
    }
    __device__ __forceinline__ typename Op::S get(int i) const
    {
        typename Op::S e;
#pragma unroll
        for (int q = 0; q < Op::NS; ++q) load_vec<Op::VEC>(at(i, q), e.v[q]);
        return e;
    }
};

// ------------------------------------------------------------ the engine

// Records: [slot][kind: aggregate, prefix][state][DC] tagged 64-bit words
// (record_tag), one per float; a lane owns VEC consecutive words per state.
template <class Op, int TX>
__device__ __forceinline__ unsigned long long *chan_record(const Lookback &lb, size_t slot,
                                                           int kind, int s, int lane)
{
    constexpr int DC = TX * Op::VEC;
    return reinterpret_cast<unsigned long long *>(lb.data) +
           ((slot * 2 + kind) * Op::NS + s) * DC + lane * Op::VEC;
}

// A lane's part of a record as loaded (tags included).
template <class Op>
struct RawRecord {
    unsigned long long w[Op::NS][Op::VEC];
};

// The states a prefix record keeps (bit s: state s; Op::kPrefixStates,
// default all).  A state may be left out when no epilogue reads it and the
// combine uses the earlier operand's copy of it only for the same state of
// the result (the running coefficient product of the adjoints, the summed
// log-coefficient of the log forward): a prefix's copy then feeds nothing
// but the next prefix's copy.  Readers fill a left-out state with the
// identity's value.  Aggregate records keep every state.
// A mask names states 0..31 only; states from 32 on (the small-matrix affine
// ops hold up to 80) are always kept.
#ifndef MG_PREFIX_TRIM
#define MG_PREFIX_TRIM 1
#endif
template <class Op, class = void>
struct op_prefix_states {
    static constexpr unsigned value = ~0u;
};
template <class Op>
struct op_prefix_states<Op, decltype(void(Op::kPrefixStates))> {
    static constexpr unsigned value = MG_PREFIX_TRIM != 0 ? Op::kPrefixStates : ~0u;
};
template <class Op>
constexpr unsigned all_states()
{
    return ~0u;
}
// Whether mask MASK keeps state s.
template <unsigned MASK>
__device__ __forceinline__ constexpr bool keeps(int s)
{
    return s >= 32 || ((MASK >> (s & 31)) & 1u) != 0u;
}

template <class Op, int TX, unsigned MASK = all_states<Op>()>
__device__ __forceinline__ void put_record(const Lookback &lb, size_t slot, int kind, int lane,
                                           const typename Op::S &x, unsigned tag)
{
#pragma unroll
    for (int s = 0; s < Op::NS; ++s) {
        if (!keeps<MASK>(s)) continue;
        unsigned long long *p = chan_record<Op, TX>(lb, slot, kind, s, lane);
        if constexpr (Op::VEC % 2 == 0) {
#pragma unroll
            for (int v = 0; v < Op::VEC; v += 2)
                st_relaxed_v2u64(p + v, tag_word(tag, x.v[s][v]), tag_word(tag, x.v[s][v + 1]));
        } else {
#pragma unroll
            for (int v = 0; v < Op::VEC; ++v) st_relaxed_u64(p + v, tag_word(tag, x.v[s][v]));
        }
    }
}

// Issue the loads of a lane's part of a record; the values are waited for
// only where they are used.
template <class Op, int TX, unsigned MASK = all_states<Op>()>
__device__ __forceinline__ void read_record(const Lookback &lb, size_t slot, int kind, int lane,
                                            RawRecord<Op> &r)
{
#pragma unroll
    for (int s = 0; s < Op::NS; ++s) {
        if (!keeps<MASK>(s)) continue;
        const unsigned long long *p = chan_record<Op, TX>(lb, slot, kind, s, lane);
        if constexpr (Op::VEC % 2 == 0) {
#pragma unroll
            for (int v = 0; v < Op::VEC; v += 2) ld_relaxed_v2u64(p + v, r.w[s][v], r.w[s][v + 1]);
        } else {
#pragma unroll
            for (int v = 0; v < Op::VEC; ++v) r.w[s][v] = ld_relaxed_u64(p + v);
        }
    }
}

template <class Op, unsigned MASK = all_states<Op>()>
__device__ __forceinline__ typename Op::S record_values(const RawRecord<Op> &r)
{
    typename Op::S x = Op::identity();
#pragma unroll
    for (int s = 0; s < Op::NS; ++s)
        if (keeps<MASK>(s)) {
#pragma unroll
            for (int v = 0; v < Op::VEC; ++v) x.v[s][v] = __uint_as_float(unsigned(r.w[s][v]));
        }
    return x;
}

// Whether every kept word of the lane's part carries `tag`.
template <class Op, unsigned MASK = all_states<Op>()>
__device__ __forceinline__ bool record_tagged(const RawRecord<Op> &r, unsigned tag)
{
    bool ok = true;
#pragma unroll
    for (int s = 0; s < Op::NS; ++s)
        if (keeps<MASK>(s)) {
#pragma unroll
            for (int v = 0; v < Op::VEC; ++v) ok &= unsigned(r.w[s][v] >> 32) == tag;
        }
    return ok;
}

// A record published under a flag this warp has acquired.
template <class Op, int TX, unsigned MASK = all_states<Op>()>
__device__ __forceinline__ typename Op::S get_record(const Lookback &lb, size_t slot, int kind,
                                                     int lane)
{
    RawRecord<Op> r;
    read_record<Op, TX, MASK>(lb, slot, kind, lane, r);
    return record_values<Op, MASK>(r);
}

// Before its fold, a chunk may load its predecessor's prefix record and take
// it as its carry-in if every word already carries this launch's tag
// (Op::kTagged, default on for records of at most 16 floats per lane): one
// round trip on the tile's critical path instead of a flag poll followed by
// the record's loads.  If any word is not there yet, the flag look-back runs
// as usual.
#ifndef MG_LB_TAGGED
#define MG_LB_TAGGED 1
#endif
template <class Op, class = void>
struct op_tagged {
    static constexpr bool value = MG_LB_TAGGED != 0 && Op::NS * Op::VEC <= 16;
};
template <class Op>
struct op_tagged<Op, decltype(void(Op::kTagged))> {
    static constexpr bool value = MG_LB_TAGGED != 0 && Op::kTagged;
};

// First half of the look-back (one warp): publish this chunk's record as
// early as possible.  Chunk 0 publishes its inclusive prefix (initial o cta)
// at once; any other chunk publishes its aggregate, unless `peek` is set and
// one poll of its predecessors' flags already resolves its carry (then its
// prefix follows shortly).  Returns the predecessor that poll resolved to,
// or -2 (find_carry then waits for one).
#ifndef MG_LB_FIRSTPOLL
#define MG_LB_FIRSTPOLL 1
#endif
template <class Op, int TX, bool PEEK = true>
__device__ int publish_first(const typename Op::Args &args, const ChanGeom &g,
                             const Lookback &lb, int c, int j, int64_t bb, int ld, bool lact,
                             bool lchan, unsigned tile, unsigned long long epoch,
                             const typename Op::S &cta)
{
    const int lane = threadIdx.x & 31;
    const size_t slot = size_t(c) * g.nJ + j;
    const unsigned tag = record_tag(lb, epoch, tile);
    if (c == 0) {
        if (lact)
            put_record<Op, TX, op_prefix_states<Op>::value>(
                lb, slot, 1, lane, Op::combine(Op::initial(args, g, bb, ld, lchan), cta), tag);
        publish(lb, slot, kStatusPrefix, epoch, tile);
        return -2;
    }
    int p0 = -2;
    bool agg = true;
    if (PEEK) {
        if (MG_LB_FIRSTPOLL) {
            p0 = poll_window(lb, size_t(j), size_t(g.nJ), c, epoch);
            agg = p0 < 0;
        } else {
            agg = peek_status(lb, slot - g.nJ, epoch) != kStatusPrefix;
        }
    }
    if (agg) {
        if (lact) put_record<Op, TX>(lb, slot, 0, lane, cta, tag);
        publish(lb, slot, kStatusAggregate, epoch, tile);
    }
    return p0;
}

// Second half (one warp): the exclusive carry-in of chunk c of channel tile j
// from its predecessors' records (after publish_first).
template <class Op, int TX>
__device__ typename Op::S find_carry(const typename Op::Args &args, const ChanGeom &g,
                                     const Lookback &lb, int c, int j, int64_t bb, int ld,
                                     bool lact, bool lchan, unsigned tile,
                                     unsigned long long epoch, int p0)
{
    using S = typename Op::S;
    const int lane = threadIdx.x & 31;
    if (c == 0) return Op::initial(args, g, bb, ld, lchan);
    S excl = Op::identity();
    // p0: the predecessor publish_first's poll already resolved, if any
    const int p = p0 >= 0 ? p0 : wait_window(lb, size_t(j), size_t(g.nJ), c, epoch, tile);
    if (p >= 0 && lact) {
        // excl = pref(p) o agg(p+1) o ... o agg(c-1), folded left to right;
        // the record loads of a batch are independent and issued together.
        excl = get_record<Op, TX, op_prefix_states<Op>::value>(lb, size_t(p) * g.nJ + j, 1, lane);
        int q = p + 1;
        for (; q + 4 <= c; q += 4) {
            const S r0 = get_record<Op, TX>(lb, size_t(q) * g.nJ + j, 0, lane);
            const S r1 = get_record<Op, TX>(lb, size_t(q + 1) * g.nJ + j, 0, lane);
            const S r2 = get_record<Op, TX>(lb, size_t(q + 2) * g.nJ + j, 0, lane);
            const S r3 = get_record<Op, TX>(lb, size_t(q + 3) * g.nJ + j, 0, lane);
            excl = Op::combine(Op::combine(Op::combine(Op::combine(excl, r0), r1), r2), r3);
        }
        for (; q < c; ++q) excl = Op::combine(excl, get_record<Op, TX>(lb, size_t(q) * g.nJ + j, 0, lane));
    }
    return excl;
}

// The whole look-back of chunk c (one warp, after its fold into `cta`): the
// predecessor's prefix words `pre` (read_record, issued before the fold) if
// TAGGED and every word already carries this launch's tag, else
// publish_first and find_carry.
template <class Op, int TX, bool PEEK, bool TAGGED>
__device__ __forceinline__ typename Op::S look_back(const typename Op::Args &args,
                                                    const ChanGeom &g, const Lookback &lb, int c,
                                                    int j, int64_t bb, int ld, bool lact,
                                                    bool lchan, unsigned tile,
                                                    unsigned long long epoch,
                                                    const typename Op::S &cta,
                                                    const RawRecord<Op> &pre)
{
    constexpr unsigned PS = op_prefix_states<Op>::value;
    if (TAGGED && c > 0 &&
        __all_sync(0xffffffffu, !lact || record_tagged<Op, PS>(pre, launch_tag(epoch))))
        return lact ? record_values<Op, PS>(pre) : Op::identity();
    const int p0 = publish_first<Op, TX, PEEK>(args, g, lb, c, j, bb, ld, lact, lchan, tile, epoch,
                                               cta);
    return find_carry<Op, TX>(args, g, lb, c, j, bb, ld, lact, lchan, tile, epoch, p0);
}

// Publish chunk c's inclusive prefix excl o cta (chunk 0 did at once).  Kept
// apart from find_carry so that the carry can be handed to the consumers
// before this release store's fence.
template <class Op, int TX>
__device__ void publish_prefix(const ChanGeom &g, const Lookback &lb, int c, int j, bool lact,
                               unsigned tile, unsigned long long epoch,
                               const typename Op::S &excl, const typename Op::S &cta)
{
    if (c == 0) return;
    const size_t slot = size_t(c) * g.nJ + j;
    if (lact)
        put_record<Op, TX, op_prefix_states<Op>::value>(lb, slot, 1, threadIdx.x & 31,
                                                        Op::combine(excl, cta),
                                                        record_tag(lb, epoch, tile));
    publish(lb, slot, kStatusPrefix, epoch, tile);
}

template <class Op, int TX, int TY, int MINB, int R>
__global__ void __launch_bounds__(TX *TY, MINB)
    channel_scan_kernel(const typename Op::Args args, const ChanGeom g, const Lookback lb)
{
    using S = typename Op::S;
    constexpr int NS = Op::NS, VEC = Op::VEC, L = Op::L;
    constexpr int DC = TX * VEC;
    constexpr bool STASH = op_stashes<Op>::value;
    extern __shared__ float4 engine_smem[];
    // s_agg[TY][NS][DC], s_carry[NS][DC], then (stashing ops) the elements
    float *const s_agg = reinterpret_cast<float *>(engine_smem);
    float *const s_carry = s_agg + TY * NS * DC;
    float *const s_stash = s_carry + NS * DC;
    auto stash = [&](int k) {
        return StashView<Op>{s_stash + (size_t(k) * L * NS * (TX * TY) + threadIdx.x) * VEC,
                             TX * TY};
    };

    unsigned tile;
    unsigned long long epoch;
    take_ticket(lb, tile, epoch);
    if (tile >= g.n_tiles) {  // a workspace that was not zero-filled before first use
        if (threadIdx.x == 0) raise_error(lb, epoch, kErrBadTicket);
        finish_cta(lb, epoch);
        return;
    }
    const int c = int(tile / unsigned(g.nJ));
    const int j = int(tile % unsigned(g.nJ));
    const int64_t bb = j / g.nJb;
    const int dbase = (j % g.nJb) * DC;
    const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
    const int d = dbase + tx * VEC;
    const bool act = d < g.D;
    const int ct = Op::kReverse ? (g.nC - 1 - c) : c;
    // The thread owns R*L consecutive steps, handled as R rounds of L steps
    // (the register footprint of one round); rounds run in processing order.
    const int64_t tspan = int64_t(ct) * (TY * L * R) + int64_t(ty) * (L * R);
    auto round_t0 = [&](int k) { return tspan + int64_t(Op::kReverse ? R - 1 - k : k) * L; };

    // Pass 1: read the thread's steps and fold them into its aggregate.  The
    // inputs are not kept across the look-back: pass 2 reads them again (the
    // tile is still in L1/L2), so registers stay free for occupancy.
    S agg;
#pragma unroll 1
    for (int k = 0; k < R; ++k) {
        typename Op::Regs r;
        Op::load(args, g, bb, round_t0(k), d, act, r);
        const int i0 = Op::kReverse ? L - 1 : 0;
        S ragg = Op::element(r, i0);
        if constexpr (STASH) stash(k).put(i0, ragg);
#pragma unroll
        for (int i = 1; i < L; ++i) {
            const int ii = Op::kReverse ? L - 1 - i : i;
            const S e = Op::element(r, ii);
            if constexpr (STASH) stash(k).put(ii, e);
            ragg = Op::combine(ragg, e);
        }
        agg = (k == 0) ? ragg : Op::combine(agg, ragg);
    }
#pragma unroll
    for (int s = 0; s < NS; ++s) store_vec<VEC>(&s_agg[((ty) * NS + s) * DC + tx * VEC], agg.v[s]);
    __syncthreads();

    S excl = Op::identity(), cta_keep = Op::identity();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const bool lact = lane < TX;
        const int ld = dbase + lane * VEC;
        const bool lchan = lact && ld < g.D;
        constexpr bool TAGGED = op_tagged<Op>::value;
        RawRecord<Op> pre;
        if (TAGGED && c > 0 && lact)
            read_record<Op, TX, op_prefix_states<Op>::value>(lb, size_t(c - 1) * g.nJ + j, 1,
                                                              lane, pre);
        S cta = Op::identity();
        if (lact) {
            // Fold the rows in processing order; each row but the first gets
            // back the fold of the rows before it (its exclusive prefix
            // within the tile), so every thread needs one combine below.
#pragma unroll
            for (int k = 0; k < TY; ++k) {
                const int y = Op::kReverse ? TY - 1 - k : k;
                float *const row = &s_agg[(y * NS) * DC + lane * VEC];
                S x;
#pragma unroll
                for (int s = 0; s < NS; ++s) load_vec<VEC>(row + s * DC, x.v[s]);
                if (k > 0) {
#pragma unroll
                    for (int s = 0; s < NS; ++s) store_vec<VEC>(row + s * DC, cta.v[s]);
                }
                cta = (k == 0) ? x : Op::combine(cta, x);
            }
        }
        excl = look_back<Op, TX, op_peeks<Op>::value, TAGGED>(args, g, lb, c, j, bb, ld, lact,
                                                              lchan, tile, epoch, cta, pre);
        if (lact) {
#pragma unroll
            for (int s = 0; s < NS; ++s) store_vec<VEC>(&s_carry[s * DC + lane * VEC], excl.v[s]);
        }
        cta_keep = cta;
    }
    __syncthreads();
    // warp 0 publishes the chunk's prefix while the others start pass 2
    if (threadIdx.x < 32)
        publish_prefix<Op, TX>(g, lb, c, j, (threadIdx.x & 31) < TX, tile, epoch, excl, cta_keep);

    // start state: carry o (rows before this one within the tile)
    S st;
#pragma unroll
    for (int s = 0; s < NS; ++s) load_vec<VEC>(&s_carry[s * DC + tx * VEC], st.v[s]);
    if (ty != (Op::kReverse ? TY - 1 : 0)) {
        S x;
#pragma unroll
        for (int s = 0; s < NS; ++s) load_vec<VEC>(&s_agg[(ty * NS + s) * DC + tx * VEC], x.v[s]);
        st = Op::combine(st, x);
    }
    // Pass 2: re-read the steps and re-run them from the start state; the
    // epilogue leaves in `st` the state after its round.
#pragma unroll 1
    for (int k = 0; k < R; ++k) {
        if constexpr (STASH) {
            Op::epilogue_stash(args, g, bb, round_t0(k), d, act, stash(k), st);
        } else {
            typename Op::Regs r2;
            Op::load(args, g, bb, round_t0(k), d, act, r2);
            Op::epilogue(args, g, bb, round_t0(k), d, act, r2, st);
        }
    }
    finish_cta(lb, epoch);
}

// ------------------------------------------------------------ launchers

template <class Op, int TX, int TY, int MINB = 1, int R = 1>
struct ChanPlan {
    static constexpr int DC = TX * Op::VEC;
    static constexpr int TC = TY * Op::L * R;
    static ChanGeom geom(int64_t B, int64_t T, int64_t D)
    {
        ChanGeom g;
        g.B = B;
        g.T = T;
        g.D = D;
        g.nJb = int((D + DC - 1) / DC);
        g.nJ = int(B * g.nJb);
        g.nC = int((T + TC - 1) / TC);
        g.n_tiles = unsigned(g.nJ) * unsigned(g.nC);
        return g;
    }
    static size_t n_tiles(int64_t B, int64_t T, int64_t D)
    {
        const int64_t nJ = B * ((D + DC - 1) / DC);
        const int64_t nC = (T + TC - 1) / TC;
        return size_t(nJ) * size_t(nC);
    }
    static size_t ws_bytes(int64_t B, int64_t T, int64_t D)
    {
        return tiled_ws_bytes(n_tiles(B, T, D), size_t(2) * Op::NS * DC * sizeof(unsigned long long));
    }
    static mg_status launch(const typename Op::Args &args, int64_t B, int64_t T, int64_t D,
                            void *ws, size_t ws_bytes_given, cudaStream_t s, const LaunchOpts &o,
                            const char *name)
    {
        const size_t nt = n_tiles(B, T, D);
        if (nt >= (size_t(1) << 31) || B * ((D + DC - 1) / DC) >= (int64_t(1) << 31))
            return fail(MG_ERR_UNSUPPORTED, "%s: %zu tiles exceed the 2^31 ticket range", name, nt);
        const size_t need = ws_bytes(B, T, D);
        if (ws_bytes_given < need)
            return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name,
                        ws_bytes_given, need);
        const ChanGeom g = geom(B, T, D);
        const Lookback lb = make_lookback(ws, nt, o);
        constexpr size_t smem =
            (size_t(TY + 1) * Op::NS * DC +
             (op_stashes<Op>::value ? size_t(R) * Op::L * Op::NS * TX * TY * Op::VEC : 0)) *
            sizeof(float);
        static_assert(smem <= 227 * 1024, "more shared memory than a CTA may have");
        if (smem > 48 * 1024) {
            static const cudaError_t attr = cudaFuncSetAttribute(
                channel_scan_kernel<Op, TX, TY, MINB, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                int(smem));
            if (attr != cudaSuccess)
                return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        }
        channel_scan_kernel<Op, TX, TY, MINB, R><<<unsigned(nt), TX * TY, smem, s>>>(args, g, lb);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", name, cudaGetErrorString(e));
        return MG_OK;
    }
};

}  // namespace
}  // namespace mg

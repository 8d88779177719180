// Persistent, warp-specialised chunked scan over time for channel-wise ops.
//
// One CTA per SM loops over (channel tile, time chunk) tiles taken by ticket
// (chunk-major, so every predecessor a tile waits on has started).  Its warps
// have fixed roles:
//
//   warp 0        producer: takes tickets and streams each tile's input rows
//                 into a ring of STAGES shared-memory buffers with 1D TMA bulk
//                 copies (one mbarrier per stage counts the bytes);
//   publishers    (NPUB warps, tiles round-robin) fold the compute warps' row
//                 aggregates into the tile aggregate and publish it at once
//                 (the first half of the decoupled look-back, lookback.cuh),
//                 so successors in other CTAs never wait on this CTA's
//                 look-back warps;
//   look-back     (NLB warps, tiles round-robin) resolve each tile's carry-in
//                 from its predecessors' records and hand it back through
//                 shared memory;
//   the rest      compute: each owns L consecutive steps of a tile for 32*VEC
//                 channels (one 16-byte vector per lane per row).  Pass 1 folds
//                 the steps into a row aggregate; pass 2 re-runs them from the
//                 row's start state (carry o earlier rows) and writes outputs.
//
// The compute warps run pass 2 of tile i only after pass 1 of tile i+NLB, so
// NLB look-backs (each a few L2 round trips) are in flight per SM at once,
// overlapped with the compute warps' work and the producer's loads.  Inputs
// are read from HBM once (staged), outputs written once (vector stores).
//
// Synchronisation per stage s (phase parity = use count & 1):
//   full[s]   producer  -> compute             (tx bytes of the copies)
//   aggr[s]   compute   -> publisher           (row aggregates written)
//   pub[s]    publisher -> look-back           (tile aggregate published)
//   carry[s]  look-back -> compute             (carry-in written)
//   empty[s]  compute   -> producer            (stage free again)
// Every wait is bounded (time and the launch's error word); a role that gives
// up leaves its loop, the producer drains its copies, and the launch ends
// with the error recorded for mg_workspace_status.
#pragma once

#include "scan_engine.cuh"

namespace mg {
namespace {

constexpr unsigned kSentinelTile = 0xffffffffu;
constexpr int kTicketBatch = 4;  // tiles per ticket grab

// A staged input: rows of `elt`-byte elements; tile row i of a tile starting
// at step t0 copies source row t0 + i + shift of a tensor with `rows` rows per
// batch (T or T+1) and the tile's channel range.
struct Staged {
    const char *base;
    long long rows;
};

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 : : "r"(smem_addr(bar)) : "memory");
}

// Bounded wait that also gives up as soon as the launch has an error.
__device__ __forceinline__ bool mbar_wait_or_error(unsigned long long *bar, unsigned parity,
                                                   const Lookback &lb, unsigned long long epoch)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0u) {
            if (launch_failed(lb, epoch)) return false;
            if (global_timer_ns() - t0 > lb.wait_limit_ns || it >= lb.max_polls) {
                raise_error(lb, epoch, kErrLookbackTimeout);
                return false;
            }
        }
    }
}

template <class Op>
struct StreamLayout {
    static constexpr int NS = Op::NS, VEC = Op::VEC, NCW = Op::NCW, L = Op::L;
    static constexpr int SG = Op::STAGES, NARR = Op::NARR;
    static constexpr int DC = 32 * VEC, TC = NCW * L;
    static constexpr int arr_bytes(int a) { return TC * DC * Op::elt(a); }
    static constexpr int arr_off(int a) { return a == 0 ? 0 : arr_off(a - 1) + arr_bytes(a - 1); }
    static constexpr int STAGE = arr_off(NARR);
    // Aggregate buffers live per stage: a stage is refilled (and its
    // aggregates rewritten) only after every compute warp released it.
    static constexpr int NAG = SG;
    static constexpr int BAR_BYTES = 5 * SG * 8;
    static constexpr int HDR = (BAR_BYTES + SG * 4 + 127) / 128 * 128;
    static constexpr size_t AGG = size_t(NCW) * NS * DC;  // floats per aggregate slot
    // per aggregate slot: row aggregates, the tile aggregate, the carry-in
    static constexpr size_t SMEM = HDR + size_t(SG) * STAGE + size_t(NAG) * (AGG + 2 * NS * DC) * 4;
    static_assert(STAGE % 16 == 0, "stage buffers must stay 16-byte aligned");
    static_assert(SMEM + 64 <= 232448, "more shared memory than one SM offers");
};

// Row i of staged array a, at this lane's channel group (VEC channels of
// elt(a) bytes each; a "channel" may be a whole matrix).
template <class Op, typename E>
__device__ __forceinline__ const E *srow(const char *st, int a, int i, int lane)
{
    using Ly = StreamLayout<Op>;
    return reinterpret_cast<const E *>(
        st + Ly::arr_off(a) + (size_t(i) * Ly::DC + size_t(lane) * Op::VEC) * Op::elt(a));
}

// Wait for phase `parity` of `bar`, or until iteration `it` is past the end
// of the CTA's work (`*end` set by the producer).  1 = phase done, 0 = past
// the end, -1 = gave up (error recorded).
__device__ __forceinline__ int mbar_wait_or_end(unsigned long long *bar, unsigned parity,
                                                const Lookback &lb, unsigned long long epoch,
                                                const volatile int *end, int it)
{
    if (mbar_try_wait(bar, parity)) return 1;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned k = 1;; ++k) {
        if (mbar_try_wait(bar, parity)) return 1;
        if (it >= *end) return 0;
        if ((k & 31u) == 0u) {
            if (launch_failed(lb, epoch)) return -1;
            if (global_timer_ns() - t0 > lb.wait_limit_ns || k >= lb.max_polls) {
                raise_error(lb, epoch, kErrLookbackTimeout);
                return -1;
            }
        }
    }
}

constexpr int kNPub = 2;  // publisher warps per CTA

template <class Op>
__global__ void __launch_bounds__((Op::NCW + Op::NLB + 1 + kNPub) * 32, 1)
    stream_scan_kernel(const typename Op::Args args, const ChanGeom g, const Lookback lb)
{
    using S = typename Op::S;
    using Ly = StreamLayout<Op>;
    constexpr int NS = Op::NS, VEC = Op::VEC, L = Op::L, NCW = Op::NCW, SG = Ly::SG;
    constexpr int NLB = Op::NLB, LAG = NLB;
    constexpr int DC = Ly::DC, TC = Ly::TC;
    static_assert(SG >= LAG + 2, "the ring needs the lagged tiles plus one in flight");
    extern __shared__ float4 stream_smem[];
    char *const smem = reinterpret_cast<char *>(stream_smem);
    unsigned long long *const full = reinterpret_cast<unsigned long long *>(smem);
    unsigned long long *const empty = full + SG;
    unsigned long long *const aggr = empty + SG;
    unsigned long long *const carry = aggr + SG;
    unsigned long long *const pub = carry + SG;
    unsigned *const s_tile = reinterpret_cast<unsigned *>(smem + Ly::BAR_BYTES);
    char *const stages = smem + Ly::HDR;
    float *const s_agg = reinterpret_cast<float *>(stages + size_t(SG) * Ly::STAGE);  // [SG][NCW][NS][DC]
    float *const s_carry = s_agg + Ly::NAG * Ly::AGG;   // [NAG][NS][DC]
    float *const s_cta = s_carry + Ly::NAG * NS * DC;    // [NAG][NS][DC]
    __shared__ unsigned long long s_epoch;
    __shared__ int s_end;  // first iteration index without a tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < SG; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NCW);
            mbar_init(aggr + s, NCW);
            mbar_init(carry + s, 1);
            mbar_init(pub + s, 1);
        }
        s_epoch = ld_relaxed_u64(&lb.ctl->epoch);
        s_end = 0x7fffffff;
    }
    __syncthreads();
    const unsigned long long epoch = s_epoch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *const end = &s_end;

    auto geom_of = [&](unsigned tile, int &c, int &j, int64_t &bb, int &d0, int64_t &t0) {
        c = int(tile / unsigned(g.nJ));
        j = int(tile % unsigned(g.nJ));
        bb = j / g.nJb;
        d0 = (j % g.nJb) * DC;
        const int ct = Op::kReverse ? (g.nC - 1 - c) : c;
        t0 = int64_t(ct) * TC;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Tickets come in batches of kTicketBatch consecutive tiles; the next
        // batch's atomic is issued as soon as a batch starts, so its latency
        // stays off the load path.  Consecutive tickets are different channel
        // tiles of one chunk (or later chunks), so a CTA never waits on its
        // own later tiles.
        int it = 0;
        unsigned next_batch = 0, batch = 0;
        int left = 0;
        if (lane == 0) next_batch = atomicAdd(&lb.ctl->ticket, unsigned(kTicketBatch));
        for (;; ++it) {
            const int s = it % SG;
            const unsigned u = unsigned(it / SG);
            if (u > 0 && !mbar_wait_or_error(empty + s, (u - 1) & 1u, lb, epoch)) break;
            if (left == 0) {
                batch = __shfl_sync(0xffffffffu, next_batch, 0);
                left = kTicketBatch;
                if (lane == 0 && batch < g.n_tiles)
                    next_batch = atomicAdd(&lb.ctl->ticket, unsigned(kTicketBatch));
            }
            const unsigned tile = batch + unsigned(kTicketBatch - left);
            --left;
            if (tile >= g.n_tiles) {
                if (lane == 0) {
                    if (batch >= g.n_tiles + 2u * kTicketBatch * gridDim.x)
                        raise_error(lb, epoch, kErrBadTicket);
                    s_tile[s] = kSentinelTile;
                    *end = it;
                    mbar_arrive(full + s);
                }
                ++it;
                break;
            }
            int c, j, d0;
            int64_t bb, t0;
            geom_of(tile, c, j, bb, d0, t0);
            const int ch = int(g.D - d0 < DC ? g.D - d0 : DC);
            unsigned bytes = 0;
            for (int i = lane; i < TC; i += 32) {
                if (t0 + i >= g.T) continue;
#pragma unroll
                for (int a = 0; a < Op::NARR; ++a) {
                    const long long r = t0 + i + Op::shift(a);
                    if (r >= 0 && r < args.src[a].rows) bytes += unsigned(ch * Op::elt(a));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, off);
            if (lane == 0) {
                s_tile[s] = tile;
                mbar_arrive_expect_tx(full + s, bytes);
            }
            __syncwarp();
            char *const st = stages + size_t(s) * Ly::STAGE;
            for (int i = lane; i < TC; i += 32) {
                if (t0 + i >= g.T) continue;
#pragma unroll
                for (int a = 0; a < Op::NARR; ++a) {
                    const long long r = t0 + i + Op::shift(a);
                    if (r >= 0 && r < args.src[a].rows) {
                        const char *src = args.src[a].base +
                                          ((bb * args.src[a].rows + r) * g.D + d0) * Op::elt(a);
                        tma_load_1d(st + Ly::arr_off(a) + size_t(i) * DC * Op::elt(a), src,
                                    unsigned(ch * Op::elt(a)), full + s);
                    }
                }
            }
        }
        if (lane == 0 && *end > it) *end = it;  // stopped early on an error
        // Drain: the copies of the last uses of every stage must land before
        // the CTA's shared memory is released (normally already done).
        for (int k = (it > SG ? it - SG : 0); k < it; ++k)
            mbar_wait_bounded(full + (k % SG), unsigned(k / SG) & 1u, lb.wait_limit_ns);
    } else if (warp <= kNPub) {
        // ----------------------------------------------------------- publisher
        for (int it = warp - 1;; it += kNPub) {
            const int s = it % SG;
            if (mbar_wait_or_end(aggr + s, unsigned(it / SG) & 1u, lb, epoch, end, it) != 1) break;
            const unsigned tile = s_tile[s];
            if (tile >= g.n_tiles) break;
            int c, j, d0;
            int64_t bb, t0;
            geom_of(tile, c, j, bb, d0, t0);
            const int ld = d0 + lane * VEC;
            const int a_slot = s;
            const float *agg = s_agg + a_slot * Ly::AGG;
            S cta;
#pragma unroll
            for (int k = 0; k < NCW; ++k) {
                const int y = Op::kReverse ? NCW - 1 - k : k;
                S x;
#pragma unroll
                for (int q = 0; q < NS; ++q) load_vec<VEC>(&agg[(y * NS + q) * DC + lane * VEC], x.v[q]);
                cta = (k == 0) ? x : Op::combine(cta, x);
            }
#pragma unroll
            for (int q = 0; q < NS; ++q)
                store_vec<VEC>(&s_cta[(a_slot * NS + q) * DC + lane * VEC], cta.v[q]);
            publish_first<Op, 32, false>(args, g, lb, c, j, bb, ld, true, ld < g.D, tile, epoch, cta);
            __syncwarp();
            if (lane == 0) mbar_arrive(pub + s);
        }
    } else if (warp <= kNPub + NLB) {
        // ----------------------------------------------------------- look-back
        for (int it = warp - 1 - kNPub;; it += NLB) {
            const int s = it % SG;
            if (mbar_wait_or_end(pub + s, unsigned(it / SG) & 1u, lb, epoch, end, it) != 1) break;
            const unsigned tile = s_tile[s];
            if (tile >= g.n_tiles) break;
            int c, j, d0;
            int64_t bb, t0;
            geom_of(tile, c, j, bb, d0, t0);
            const int ld = d0 + lane * VEC;
            const bool lchan = ld < g.D;
            const int a_slot = s;
            S cta;
#pragma unroll
            for (int q = 0; q < NS; ++q)
                load_vec<VEC>(&s_cta[(a_slot * NS + q) * DC + lane * VEC], cta.v[q]);
            const S excl = find_carry<Op, 32>(args, g, lb, c, j, bb, ld, true, lchan, tile, epoch);
            float *cr = s_carry + a_slot * NS * DC;
#pragma unroll
            for (int q = 0; q < NS; ++q) store_vec<VEC>(&cr[q * DC + lane * VEC], excl.v[q]);
            __syncwarp();
            if (lane == 0) mbar_arrive(carry + s);
            publish_prefix<Op, 32>(g, lb, c, j, true, tile, epoch, excl, cta);
        }
    } else {
        // ------------------------------------------------------------- compute
        const int ty = warp - 1 - kNPub - NLB;
        auto pass1 = [&](int s, int a_slot, unsigned tile) {
            int c, j, d0;
            int64_t bb, t0;
            geom_of(tile, c, j, bb, d0, t0);
            const char *st = stages + size_t(s) * Ly::STAGE;
            S agg = Op::identity();
#pragma unroll
            for (int k = 0; k < L; ++k) {
                const int i = ty * L + (Op::kReverse ? L - 1 - k : k);
                const S e = Op::elem(st, i, lane, t0 + i, g);
                agg = (k == 0) ? e : Op::combine(agg, e);
            }
            float *dst = s_agg + a_slot * Ly::AGG;
#pragma unroll
            for (int q = 0; q < NS; ++q) store_vec<VEC>(&dst[(ty * NS + q) * DC + lane * VEC], agg.v[q]);
        };
        auto pass2 = [&](int s, int a_slot, unsigned tile) {
            int c, j, d0;
            int64_t bb, t0;
            geom_of(tile, c, j, bb, d0, t0);
            const char *st = stages + size_t(s) * Ly::STAGE;
            const float *agg = s_agg + a_slot * Ly::AGG;
            const float *cr = s_carry + a_slot * NS * DC;
            S state;
#pragma unroll
            for (int q = 0; q < NS; ++q) load_vec<VEC>(&cr[q * DC + lane * VEC], state.v[q]);
            for (int k = 0; k < NCW; ++k) {  // earlier rows of the tile, processing order
                const int y = Op::kReverse ? NCW - 1 - k : k;
                if (y == ty) break;
                S x;
#pragma unroll
                for (int q = 0; q < NS; ++q) load_vec<VEC>(&agg[(y * NS + q) * DC + lane * VEC], x.v[q]);
                state = Op::combine(state, x);
            }
            const int d = d0 + lane * VEC;
            const bool act = d < g.D;
#pragma unroll
            for (int k = 0; k < L; ++k) {
                const int i = ty * L + (Op::kReverse ? L - 1 - k : k);
                Op::step2(args, st, i, lane, t0 + i, g, bb, d, act, state);
            }
        };
        // pass 2 of iteration k: wait for its carry, re-run, free the stage
        auto finish = [&](int k) -> bool {
            const int s = k % SG;
            if (!mbar_wait_or_error(carry + s, unsigned(k / SG) & 1u, lb, epoch)) return false;
            pass2(s, s, s_tile[s]);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
            return true;
        };
        int it = 0;
        bool ok = true;
        for (;; ++it) {
            const int s = it % SG;
            if (!mbar_wait_or_error(full + s, unsigned(it / SG) & 1u, lb, epoch)) {
                ok = false;
                break;
            }
            const unsigned tile = s_tile[s];
            if (tile >= g.n_tiles) break;
            pass1(s, s, tile);
            __syncwarp();
            if (lane == 0) mbar_arrive(aggr + s);
            if (it >= LAG && !finish(it - LAG)) {
                ok = false;
                break;
            }
        }
        if (ok)
            for (int k = (it > LAG ? it - LAG : 0); k < it; ++k)
                if (!finish(k)) break;
    }
    finish_cta(lb, epoch);
}

template <class Op>
struct StreamPlan {
    using Ly = StreamLayout<Op>;
    static constexpr int DC = Ly::DC, TC = Ly::TC;
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
        return size_t(B * ((D + DC - 1) / DC)) * size_t((T + TC - 1) / TC);
    }
    static size_t ws_bytes(int64_t B, int64_t T, int64_t D)
    {
        return tiled_ws_bytes(n_tiles(B, T, D), size_t(2) * Op::NS * DC * sizeof(float));
    }
    static mg_status launch(const typename Op::Args &args, int64_t B, int64_t T, int64_t D,
                            void *ws, size_t wsb, cudaStream_t s, const LaunchOpts &o,
                            const char *name)
    {
        const size_t nt = n_tiles(B, T, D);
        if (nt >= (size_t(1) << 30) || B * ((D + DC - 1) / DC) >= (int64_t(1) << 31))
            return fail(MG_ERR_UNSUPPORTED, "%s: %zu tiles exceed the 2^31 ticket range", name, nt);
        const size_t need = ws_bytes(B, T, D);
        if (wsb < need)
            return fail(MG_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, wsb, need);
        static int n_sm = 0;
        static cudaError_t attr = cudaSuccess;
        static bool once = false;
        if (!once) {
            int dev = 0;
            attr = cudaGetDevice(&dev);
            if (attr == cudaSuccess)
                attr = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
            if (attr == cudaSuccess)
                attr = cudaFuncSetAttribute(stream_scan_kernel<Op>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            int(Ly::SMEM));
            once = true;
        }
        if (attr != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: %s", name, cudaGetErrorString(attr));
        const ChanGeom g = geom(B, T, D);
        const Lookback lb = make_lookback(ws, nt, o);
        const unsigned grid = unsigned(nt < size_t(n_sm) ? nt : size_t(n_sm));
        stream_scan_kernel<Op><<<grid, (Op::NCW + Op::NLB + 1 + kNPub) * 32, Ly::SMEM, s>>>(args, g, lb);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(MG_ERR_LAUNCH, "%s: launch failed: %s", name, cudaGetErrorString(e));
        return MG_OK;
    }
};

}  // namespace
}  // namespace mg

// Chunk look-back machinery shared by every scan kernel of the library.
//
// A scan along time is cut into chunks.  Each CTA takes one (channel tile,
// chunk) pair by ticket, reduces its chunk to an aggregate, and needs the
// composition of every earlier chunk of the same channel tile (its exclusive
// prefix).  It finds that prefix with a decoupled look-back: it publishes its
// aggregate, walks back over its predecessors' published records until it
// meets one that holds an inclusive prefix, and publishes its own inclusive
// prefix.  Tickets are handed out in launch order, chunk-major, so every
// predecessor a CTA waits on has already started: the waits always end.
//
// Determinism.  After the walk back finds an inclusive prefix at chunk p, the
// waiting CTA folds the aggregates p+1 .. c-1 FORWARD onto it.  Every prefix
// is therefore the left fold agg(0) o agg(1) o ... o agg(c) in the same
// order whatever the walk met, so results are bitwise reproducible run to run.
//
// Workspace layout (caller-owned, zero-filled once before first use):
//   [0, 256)            Control
//   [256, 256 + 8*N)    one 64-bit record flag per tile:
//                       kFlagTag | epoch << 2 | status
//   then                per-tile data, op-specific (aggregate and prefix),
//                       as tagged 64-bit words where the op's records go
//                       through the chunk engine (see record_tag)
// A flag counts only if its epoch equals the launch's epoch, so stale flags
// of earlier launches need no clearing.  The last CTA of every launch resets
// the ticket and done counters and advances the epoch.  Where the flags of a
// launch with more tiles overlay the data records of an earlier launch with
// fewer, the old words are float pairs; the tag sets the top 13 bits, which
// as the upper float of a pair is a negative quiet NaN with a non-zero
// payload bit pattern that no arithmetic result has (the GPU's NaN is
// 0x7fffffff), so no stale record reads as a flag of the running launch.
//
// Bounded waits.  A wait gives up after `max_polls` polls or `wait_limit_ns`
// nanoseconds of %globaltimer, or as soon as another CTA of the SAME launch
// has given up.  Giving up sets the sticky Control::error word (read and
// cleared by mg_workspace_status), tags it with the launch's epoch
// (Control::error_epoch), and the CTA carries on with an identity carry, so
// the launch always finishes and the GPU stays usable.  A later launch on the
// same workspace does not give up early because of an earlier launch's
// error: it compares the tag with its own epoch.
#pragma once

#include <cstdint>

namespace mg {

enum : unsigned { kStatusNone = 0, kStatusAggregate = 1, kStatusPrefix = 2 };
enum : unsigned { kErrLookbackTimeout = 1u, kErrBadTicket = 2u, kErrBadSeqlens = 4u };

struct Control {
    unsigned int ticket;       // next tile ticket of the running launch
    unsigned int done;         // CTAs of the running launch that have finished
    unsigned long long epoch;  // launch counter; tags the record flags
    unsigned int error;        // sticky error bits (kErr*)
    unsigned int error_tile;   // 1 + a tile that gave up a wait (0 = none)
    unsigned long long error_epoch;  // 1 + epoch of the last launch that set an error
    unsigned int pad[56];
};
static_assert(sizeof(Control) == 256, "control block is 256 bytes");

constexpr size_t kControlBytes = 256;

struct Lookback {
    Control *ctl;
    unsigned long long *flags;   // [n_tiles]
    float *data;                 // op-specific per-tile records
    unsigned long long wait_limit_ns;
    unsigned int max_polls;
    long long stall_tile;        // testing only: this tile never publishes (-1: none)
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" : : "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" : : "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_v2u64(unsigned long long *p, unsigned long long a,
                                                 unsigned long long b)
{
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" : : "l"(p), "l"(a), "l"(b)
                 : "memory");
}

__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long *p, unsigned long long &a,
                                                 unsigned long long &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p)
                 : "memory");
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr unsigned long long kFlagTag = 0xfff8000000000000ull;
constexpr unsigned long long kEpochMask = (1ull << 49) - 1;

// The flag word of `status` in the launch of `epoch`.
__device__ __forceinline__ unsigned long long flag_word(unsigned long long epoch, unsigned status)
{
    return kFlagTag | ((epoch & kEpochMask) << 2) | status;
}

// Status of a flag word for this launch (kStatusNone if stale or unset).
__device__ __forceinline__ unsigned flag_status(unsigned long long v, unsigned long long epoch)
{
    return ((v & ~3ull) == flag_word(epoch, 0)) ? unsigned(v & 3ull) : kStatusNone;
}

// Tagged record words.  Every float of a tile's record is stored as one
// 64-bit word: the high half tags the launch that wrote it, the low half holds
// the float's bits.  An aligned 64-bit access is single-copy atomic, so a
// reader whose relaxed load sees its own launch's tag in a word also sees the
// value written with it, without first acquiring the record's flag: a chunk
// can take its predecessor's inclusive prefix in one round trip as soon as the
// words land (the flags still serve every other look-back step).  The tag's
// top two bits are 01, so a tagged word never equals zero-filled memory or a
// flag word (top 13 bits set), and tags of different launches on the same
// workspace differ (the low 30 bits of the epoch).  The tile that the testing
// option stalls writes tag 0, which no reader accepts, so its successors wait
// on its flag as before.
__device__ __forceinline__ unsigned launch_tag(unsigned long long epoch)
{
    return 0x40000000u | unsigned(epoch & 0x3fffffffull);
}

// The tag `tile` writes into its records.
__device__ __forceinline__ unsigned record_tag(const Lookback &lb, unsigned long long epoch,
                                               unsigned tile)
{
    return (long long)tile == lb.stall_tile ? 0u : launch_tag(epoch);
}

__device__ __forceinline__ unsigned long long tag_word(unsigned tag, float x)
{
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(x);
}

// Record an error of the launch of `epoch` (any thread): the sticky bits,
// the first tile that gave up (if `tile` names one) and the launch tag.
__device__ __forceinline__ void raise_error(const Lookback &lb, unsigned long long epoch,
                                            unsigned bits, unsigned tile_plus1 = 0u)
{
    atomicOr(&lb.ctl->error, bits);
    if (tile_plus1 != 0u) atomicCAS(&lb.ctl->error_tile, 0u, tile_plus1);
    atomicMax(&lb.ctl->error_epoch, epoch + 1ull);
}

// Whether another CTA of the launch of `epoch` has already given up a wait.
__device__ __forceinline__ bool launch_failed(const Lookback &lb, unsigned long long epoch)
{
    return ld_relaxed_u64(&lb.ctl->error_epoch) == epoch + 1ull;
}

// Take a ticket and read the launch epoch (thread 0 of the CTA); all threads
// get both through shared memory.
__device__ __forceinline__ void take_ticket(const Lookback &lb, unsigned &tile,
                                            unsigned long long &epoch)
{
    __shared__ unsigned s_tile;
    __shared__ unsigned long long s_epoch;
    if (threadIdx.x == 0) {
        s_tile = atomicAdd(&lb.ctl->ticket, 1u);
        s_epoch = ld_relaxed_u64(&lb.ctl->epoch);
    }
    __syncthreads();
    tile = s_tile;
    epoch = s_epoch;
}

// Look at a record flag without waiting (warp-collective; lane 0 reads).
__device__ __forceinline__ unsigned peek_status(const Lookback &lb, size_t slot,
                                                unsigned long long epoch)
{
    unsigned st = 0;
    if ((threadIdx.x & 31) == 0)
        st = flag_status(ld_relaxed_u64(lb.flags + slot), epoch);
    return __shfl_sync(0xffffffffu, st, 0);
}

// Wait until record `slot` holds an aggregate or a prefix of this launch.
// Warp-collective.  Returns its status, or kStatusNone if the wait gave up.
// Lane 0 polls with acquire loads; the __syncwarp that follows orders every
// lane's later (L2) loads of the record's data after that acquire.
static __device__ __noinline__ unsigned wait_status(const Lookback &lb, size_t slot,
                                                    unsigned long long epoch, unsigned my_tile)
{
    const unsigned lane = threadIdx.x & 31;
    unsigned st = kStatusNone;
    if (lane == 0) {
        st = flag_status(ld_acquire_u64(lb.flags + slot), epoch);
        if (st == kStatusNone) {
            const unsigned long long t0 = global_timer_ns();
            unsigned sleep_ns = 20;
            for (unsigned it = 0;; ++it) {
                __nanosleep(sleep_ns);
                if (sleep_ns < 500) sleep_ns += sleep_ns;
                st = flag_status(ld_acquire_u64(lb.flags + slot), epoch);
                if (st != kStatusNone) break;
                if (it >= lb.max_polls || global_timer_ns() - t0 > lb.wait_limit_ns ||
                    launch_failed(lb, epoch)) {
                    raise_error(lb, epoch, kErrLookbackTimeout, my_tile + 1u);
                    break;
                }
            }
        }
    }
    st = __shfl_sync(0xffffffffu, st, 0);
    __syncwarp();
    return st;
}

// Parallel look-back window (warp-collective).  Chunk c of a chain whose
// records sit at slots q*stride + j looks at its 32 nearest predecessors at
// once: lane l polls chunk c-1-l.  The wait ends when the nearest predecessor
// holding an inclusive prefix is inside the window and every chunk between it
// and c holds at least an aggregate.  Returns that chunk p, or -1 if the wait
// gave up.  Lanes past chunk 0 read as "prefix" (a sentinel that can never
// be chosen: chunk 0 only ever publishes a prefix, so while it is unpublished
// an unset flag precedes the sentinel).  The __syncwarp before returning
// orders every lane's later record loads after the acquires.
static __device__ __noinline__ int wait_window(const Lookback &lb, size_t j, size_t stride, int c,
                                               unsigned long long epoch, unsigned my_tile)
{
    const int lane = threadIdx.x & 31;
    const int q = c - 1 - lane;
    const unsigned long long t0 = global_timer_ns();
    unsigned sleep_ns = 20;
    for (unsigned it = 0;; ++it) {
        unsigned st = kStatusPrefix;
        if (q >= 0) st = flag_status(ld_acquire_u64(lb.flags + size_t(q) * stride + j), epoch);
        const unsigned pmask = __ballot_sync(0xffffffffu, st == kStatusPrefix);
        const unsigned xmask = __ballot_sync(0xffffffffu, st == kStatusNone);
        if (pmask != 0u) {
            const int first = __ffs(pmask) - 1;
            const unsigned before = first == 0 ? 0u : (0xffffffffu >> (32 - first));
            if ((xmask & before) == 0u) {
                __syncwarp();
                return first <= c - 1 ? c - 1 - first : -1;
            }
        }
        int stop = 0;
        if (lane == 0 && (it >= lb.max_polls || global_timer_ns() - t0 > lb.wait_limit_ns ||
                          launch_failed(lb, epoch))) {
            raise_error(lb, epoch, kErrLookbackTimeout, my_tile + 1u);
            stop = 1;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return -1;
        __nanosleep(sleep_ns);
        if (sleep_ns < 400) sleep_ns += sleep_ns;
    }
}

// One poll of the window of wait_window, without waiting or raising errors:
// the chunk wait_window would return if the window resolves on this poll,
// else -2.  Warp-collective.
static __device__ __noinline__ int poll_window(const Lookback &lb, size_t j, size_t stride, int c,
                                               unsigned long long epoch)
{
    const int lane = threadIdx.x & 31;
    const int q = c - 1 - lane;
    unsigned st = kStatusPrefix;
    if (q >= 0) st = flag_status(ld_acquire_u64(lb.flags + size_t(q) * stride + j), epoch);
    const unsigned pmask = __ballot_sync(0xffffffffu, st == kStatusPrefix);
    const unsigned xmask = __ballot_sync(0xffffffffu, st == kStatusNone);
    int p = -2;
    if (pmask != 0u) {
        const int first = __ffs(pmask) - 1;
        const unsigned before = first == 0 ? 0u : (0xffffffffu >> (32 - first));
        if ((xmask & before) == 0u && first <= c - 1) p = c - 1 - first;
    }
    __syncwarp();
    return p;
}

// Publish record `slot` with `status` (warp-collective).  Every lane must have
// written its part of the record (.cg stores) before calling; the __syncwarp
// orders those writes before lane 0's release store, which is cumulative.
__device__ __forceinline__ void publish(const Lookback &lb, size_t slot, unsigned status,
                                        unsigned long long epoch, unsigned my_tile)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && (long long)my_tile != lb.stall_tile)
        st_release_u64(lb.flags + slot, flag_word(epoch, status));
}

// End of a CTA: count it; the launch's last CTA resets the ticket and done
// counters and advances the epoch for the next launch on this workspace.
__device__ __forceinline__ void finish_cta(const Lookback &lb, unsigned long long epoch)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&lb.ctl->done, 1u);
        if (prev == gridDim.x - 1) {
            lb.ctl->ticket = 0;
            lb.ctl->done = 0;
            lb.ctl->epoch = epoch + 1;
            __threadfence();
        }
    }
}

}  // namespace mg

// Partition kernel and circular-buffer tile-merge kernel for the stable
// co-rank merge on sm_103a.
//
// Method (web pages, cited by title and section):
//  * co-rank and its acceptance test, ties to A: "Co-rank Function 實作與
//    Basic Parallel Merge Kernel", §Co-rank Function 定義與不變式,
//    §Binary-Search Implementation, §Important (asymmetric <= / <).
//  * one co-rank per block-level output range, then block-cooperative
//    staging of the A and B windows: "Tiled 與 Circular Buffer Merge Kernel
//    (Memory Coalescing)", §Block-Level Co-Rank 與協同載入, §迭代式 Tile 載入與
//    Consumed 追蹤.
//  * circular buffer that keeps the unconsumed part of each window and
//    refills only consumed slots, with A_consumed / B_consumed / C_completed
//    bookkeeping: same page, §Circular Buffer Merge Kernel and §Simplified
//    Model 與 Circular 函式.
//
// GB300 design (what differs from the pages):
//  * The block-level co-rank of each CTA's output range is found inside the
//    tile-merge kernel by its two producer warps, one range end each, each
//    warp probing 32 points per round (higher radix).  A separate partition
//    kernel that writes the same splitters to an array serves the entry
//    point that keeps them in a fixed device array.
//  * Every search is a bounded form of the same co-rank: the largest i in
//    [max(0,k-n), min(k,m)] with i == lower bound or A[i-1] <= B[k-i].  On
//    sorted input it is the pages' i; on any input it stops.
//  * Ring slots are indexed by the element's 16-byte-aligned address
//    position (u), so every refill is a 16-byte-aligned 1-D bulk copy on the
//    TMA engine tracked by an mbarrier; the ring size is a power of two so
//    the pages' "% tile_size" wrap is a mask.
//  * Refills run ahead: a chunk is requested as soon as the slots it lands
//    in are consumed, so input for later sub-tiles is in flight while the
//    current one is merged; each ring has a 32-slot overhang that mirrors its
//    first slots, so a serial merge never wraps.
//  * The producers compute each sub-tile's co-rank themselves and publish
//    the next sub-tile's window while the consumers merge the current one.
//  * The kernel is warp-specialised: two producer threads (one per input
//    side) own all bulk copies and the consumed-count bookkeeping; consumer
//    warps only search, merge and stage, synchronised with the producers by
//    mbarriers.
//  * Each consumer thread merges VT (odd) outputs into registers; they pass
//    through a shared-memory stage that a producer writes to C with one
//    bulk store per sub-tile, instead of the pages' per-thread strided
//    writes.
#pragma once

#include <cstdint>

#include "om_ptx.cuh"

namespace om {

// Element size of a key type: E bytes, G = 16 / E elements per 16-byte group
// (the unit of every bulk copy's start, length and destination).
template <typename K>
struct KeyGeom {
    static constexpr int E = (int)sizeof(K);
    static constexpr int G = 16 / E;
    static_assert(E == 4 || E == 8, "keys of 4 or 8 bytes");
};

// Compare form of a key.  Integers and floats compare as themselves.  A
// double compares through an int64 with the same order, so the compares run
// on the integer pipes instead of the FP64 unit (a small fraction of the
// FP32 rate on this GPU): the sign-magnitude bits become two's complement,
// which maps -0.0 and +0.0 to the same integer 0 and orders every other
// non-NaN value as IEEE does.  Outputs keep the original bits.
template <typename K>
struct OrderKey {
    __device__ __forceinline__ static K of(K x) { return x; }
};
template <>
struct OrderKey<double> {
    // s = 0 (sign clear) or -1 (set): (b ^ (s & 0x7FF..F)) - s is b for a
    // non-negative value and -(b & 0x7FF..F) for a negative one.
    __device__ __forceinline__ static long long of(double x) {
        const long long b = __double_as_longlong(x);
        const long long s = b >> 63;
        return (b ^ (s & 0x7FFFFFFFFFFFFFFFLL)) - s;
    }
};

// The merge order on compare forms: x (from A) goes out no later than y
// (from B).  Ascending: x <= y; descending: x >= y.  Either way equal keys
// take A first, so the merge is stable.
template <bool DESC, typename O>
__device__ __forceinline__ bool ord_first(O x, O y) {
    return DESC ? (y <= x) : (x <= y);
}

// The same order on keys: a of A goes out no later than b of B.
template <bool DESC, typename K>
__device__ __forceinline__ bool a_first(K a, K b) {
    return ord_first<DESC>(OrderKey<K>::of(a), OrderKey<K>::of(b));
}

// ---------------------------------------------------------------- geometry --

// A merge problem cut into output ranges of `range_len` outputs.
//  run == 0: one merge, A = a_*, B = b_*, lengths m and n.
//  run  > 0: one pass of a bottom-up merge sort over a single buffer a_* of
//            m elements: segment s merges run 2s (A) with run 2s+1 (B),
//            each `run` long except at the end; b_* is unused.
template <typename K>
struct MergeGeom {
    const K* a_keys;
    const uint32_t* a_vals;
    const K* b_keys;
    const uint32_t* b_vals;
    K* c_keys;
    uint32_t* c_vals;
    int64_t m, n;
    int64_t run;
    int64_t range_len;
    int64_t ranges_per_seg;
    int64_t nranges;
};

template <typename K>
struct Segment {
    const K* ak;
    const uint32_t* av;
    int64_t m;
    const K* bk;
    const uint32_t* bv;
    int64_t n;
    K* ck;
    uint32_t* cv;
};

template <typename K, bool V>
__device__ __forceinline__ Segment<K> segment_of(const MergeGeom<K>& g, int64_t seg) {
    Segment<K> s;
    if (g.run == 0) {
        s.ak = g.a_keys;
        s.av = g.a_vals;
        s.m = g.m;
        s.bk = g.b_keys;
        s.bv = g.b_vals;
        s.n = g.n;
        s.ck = g.c_keys;
        s.cv = g.c_vals;
    } else {
        const int64_t base = seg * 2 * g.run;
        const int64_t rem = g.m - base;
        s.m = rem < g.run ? rem : g.run;
        const int64_t rb = rem - g.run;
        s.n = rb <= 0 ? 0 : (rb < g.run ? rb : g.run);
        s.ak = g.a_keys + base;
        s.bk = g.a_keys + base + s.m;
        s.ck = g.c_keys + base;
        if (V) {
            s.av = g.a_vals + base;
            s.bv = g.a_vals + base + s.m;
            s.cv = g.c_vals + base;
        } else {
            s.av = nullptr;
            s.bv = nullptr;
            s.cv = nullptr;
        }
    }
    return s;
}

// ------------------------------------------------------------- co-rank --

// co_rank(k) over global memory: the largest i in [max(0,k-n), min(k,m)]
// such that i is the lower bound or A[i-1] <= B[k-i].  At most
// ceil(log2(min(k,m) - max(0,k-n) + 1)) dependent loads.
template <typename K, bool DESC = false>
__device__ __forceinline__ int64_t corank_global(int64_t k, const K* __restrict__ A, int64_t m,
                                                 const K* __restrict__ B, int64_t n) {
    int64_t lo = k - n > 0 ? k - n : 0;
    int64_t hi = k < m ? k : m;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;  // lo < mid <= hi
        if (a_first<DESC>(__ldg(A + mid - 1), __ldg(B + k - mid))) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

// co_rank(k) by one warp, 33-way: while the interval [lo, hi] holds more
// than 32 candidates, the 32 lanes probe 32 evenly spaced points at once and
// a ballot keeps the sub-interval between the last probe that passed and the
// first that failed; the last <= 32 candidates are probed in one round.  This
// is the higher-radix form of the same search ("Co-rank Function 實作與
// Basic Parallel Merge Kernel", §Overview: binary search, or higher radix):
// about log33(range) + 1 rounds of parallel loads instead of log2(range)
// dependent loads.  Every lane returns the result.  On unsorted input the
// passing probes need not form a prefix; the interval still shrinks every
// round, so the loop always ends.
//
// The first round probes a ladder around the proportional estimate
// e = k * m / (m + n) instead (e -+ 1, 4, 16, ..., 4^15, clamped into the
// interval): on sorted data whose two inputs mix evenly the co-rank sits
// within a few hundred or thousand places of e, so one round brackets it
// tightly and the 33-way rounds start from a small interval (2-3 rounds
// fewer on large inputs).  Any sorted list of probes in (lo, hi] keeps the
// search exact: the passing probes are a prefix, and the interval becomes
// the gap between the last passing and the first failing one.  So e needs no
// exactness and is taken in fp32 (relative error about 2^-23, a few places
// on a 2^29-output merge): this GPU's FP64 rate is a small fraction of its
// FP32 rate, and a double division in every lane of every searching warp
// cost the one-wave merge about 1.7 us at its start.
template <typename K, bool DESC = false>
__device__ __forceinline__ int64_t corank_warp(int64_t k, const K* __restrict__ A, int64_t m,
                                               const K* __restrict__ B, int64_t n, int lane) {
    int64_t lo = k - n > 0 ? k - n : 0;
    int64_t hi = k < m ? k : m;
    if (hi - lo > 64) {
        // 0 <= e <= about k (m + n > 0 here); the clamp below keeps every probe in (lo, hi]
        const int64_t e = (int64_t)((float)k * __fdividef((float)m, (float)(m + n)));
        const int j = lane < 16 ? 15 - lane : lane - 16;  // ladder step 4^j
        const int64_t off = (int64_t)1 << (2 * j);
        int64_t c = lane < 16 ? e - off + 1 : e + off;   // e-4^15+1 .. e, e+1 .. e+4^15
        c = c <= lo ? lo + 1 : (c > hi ? hi : c);        // sorted, in (lo, hi]
        const bool pass = a_first<DESC>(__ldg(A + c - 1), __ldg(B + k - c));
        const unsigned bal = __ballot_sync(0xffffffffu, pass);
        const int t = __popc(bal);
        const int64_t c_prev = __shfl_sync(0xffffffffu, c, t > 0 ? t - 1 : 0);
        const int64_t c_next = __shfl_sync(0xffffffffu, c, t < 32 ? t : 31);
        const int64_t new_lo = t == 0 ? lo : c_prev;
        const int64_t new_hi = t == 32 ? hi : c_next - 1;
        lo = new_lo;
        hi = new_hi > lo ? new_hi : lo;  // (on unsorted input the probes need not form a prefix)
    }
    while (hi - lo > 32) {
        const int64_t span = hi - lo;
        const int64_t c = lo + (span * (lane + 1)) / 33;  // lo < c < hi
        const bool pass = a_first<DESC>(__ldg(A + c - 1), __ldg(B + k - c));
        const int t = __popc(__ballot_sync(0xffffffffu, pass));
        const int64_t new_lo = (t == 0) ? lo : lo + (span * t) / 33;
        const int64_t new_hi = (t == 32) ? hi : lo + (span * (t + 1)) / 33 - 1;
        lo = new_lo;
        hi = new_hi;
    }
    const int64_t c = lo + 1 + lane;
    bool pass = false;
    if (c <= hi) pass = a_first<DESC>(__ldg(A + c - 1), __ldg(B + k - c));
    return lo + __popc(__ballot_sync(0xffffffffu, pass));
}

// Partition kernel: split[r] = co-rank of the first output of range r within
// its segment.  One warp per range.
template <typename K, bool V, bool DESC = false>
__global__ void __launch_bounds__(128) partition_kernel(MergeGeom<K> g, int64_t* __restrict__ split) {
    const int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= g.nranges) return;  // whole warp
    const int64_t seg = r / g.ranges_per_seg;
    const int64_t local = r - seg * g.ranges_per_seg;
    const Segment<K> s = segment_of<K, V>(g, seg);
    const int64_t len = s.m + s.n;
    // local * range_len, clamped to len without overflowing
    const int64_t k = (local > len / g.range_len) ? len : (local * g.range_len < len ? local * g.range_len : len);
    const int64_t i = corank_warp<K, DESC>(k, s.ak, s.m, s.bk, s.n, lane);
    if (lane == 0) split[r] = i;
}

// One co-rank by one warp.
template <typename K, bool DESC = false>
__global__ void __launch_bounds__(32) corank_one_kernel(int64_t k, const K* __restrict__ A, int64_t m,
                                                        const K* __restrict__ B, int64_t n, int64_t* out) {
    const int64_t i = corank_warp<K, DESC>(k, A, m, B, n, threadIdx.x & 31);
    if (threadIdx.x == 0) *out = i;
}

// Batched co-rank of one merge (device ks -> device i).
template <typename K, bool DESC = false>
__global__ void __launch_bounds__(128) corank_batch_kernel(const int64_t* __restrict__ ks, int64_t count,
                                                           const K* __restrict__ A, int64_t m,
                                                           const K* __restrict__ B, int64_t n,
                                                           int64_t* __restrict__ out) {
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t >= count) return;
    int64_t k = ks[t];
    k = k < 0 ? 0 : (k > m + n ? m + n : k);
    out[t] = corank_global<K, DESC>(k, A, m, B, n);
}

// ------------------------------------------------------------ tile merge --

template <int NT_, int VT_, int RING_LOG2_, int CH_LOG2_, int MIN_CTAS_ = 5>
struct TileCfg {
    static constexpr int NT = NT_;          // consumer threads
    static constexpr int THREADS = NT + 64;  // plus two producer warps
    // CTAs per SM the shape is sized for (by its shared memory): the register
    // budget the compiler must keep to
    static constexpr int MIN_CTAS = MIN_CTAS_;
    static constexpr int VT = VT_;
    static constexpr int T = NT * VT;  // outputs per sub-tile
    static constexpr int RING_LOG2 = RING_LOG2_;
    static constexpr int RING = 1 << RING_LOG2;
    static constexpr uint32_t RMASK = RING - 1;
    static constexpr int CH_LOG2 = CH_LOG2_;
    static constexpr int CH = 1 << CH_LOG2;  // elements per refill chunk
    static constexpr int NCH_LOG2 = RING_LOG2 - CH_LOG2;
    static constexpr int NCH = 1 << NCH_LOG2;
    static constexpr int STAGE = T + 8;
    // Each side's ring region is RING slots plus an overhang of OVH slots
    // that mirrors slots [0, OVH): a head placed at slot x < RING can walk
    // VT - 1 slots on without wrapping, so the serial merge needs no mask.
    static constexpr int OVH = 32;
    static constexpr int RSTRIDE = RING + OVH;  // elements per side region (A, then B)
    // largest power of two <= T: the first step of the fixed-step search
    static constexpr int SEARCH_TOP = (T >= 4096) ? 4096 : (T >= 2048) ? 2048 : (T >= 1024) ? 1024
                                    : (T >= 512) ? 512 : (T >= 256) ? 256 : 128;
    static_assert(VT % 2 == 1, "an odd VT keeps the register->stage writes and the search's first probes free "
                               "of bank conflicts");
    static_assert(T % 4 == 0, "sub-tile boundaries stay 16-byte aligned in C");
    static_assert(T + CH <= RING, "a window of T plus one chunk must fit in the ring");
    static_assert(CH >= 4 && NCH >= 2, "chunks are whole 16-byte groups");
    static_assert(2 * SEARCH_TOP > T, "the fixed-step search must reach every co-rank");
    static_assert(OVH >= VT && OVH % 4 == 0 && OVH <= CH, "the overhang covers one serial merge, in 16-byte groups");
};

// Streaming state of one input side (A or B) of one CTA's output range.
// Positions are in "u" units: u = element index + (address / E) mod G of
// the side's first element (E-byte keys, G = 16 / E), so u % G == 0 exactly
// at 16-byte boundaries.
struct SideStream {
    const char* base16;       // 16-byte aligned address of u = 0 (keys)
    const char* vbase16;      // same for values
    int64_t arr_lo, arr_hi;   // u extent of the whole side array
    int64_t arr_lo4, arr_hi4; // its 16-byte-aligned interior
    int64_t u_lo, u_hi;       // u extent of this CTA's part
    int64_t head;             // next unconsumed u (A_consumed / B_consumed)
    int64_t c_first, c_last;  // chunk indices covering [u_lo, u_hi)
    int64_t next_issue;       // next chunk to request (thread 0)
    int next_wait;            // next chunk (relative to c_first) not yet waited for
};

template <typename Cfg, typename K>
__device__ __forceinline__ void side_init(SideStream& s, const void* keys, const void* vals, int64_t len,
                                          int64_t lo, int64_t hi) {
    constexpr int E = KeyGeom<K>::E, G = KeyGeom<K>::G;
    const uintptr_t a = reinterpret_cast<uintptr_t>(keys);
    const int64_t mis = (int64_t)((a / E) & (G - 1));
    s.base16 = reinterpret_cast<const char*>(a & ~uintptr_t(15));
    s.vbase16 = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(vals) & ~uintptr_t(15));
    s.arr_lo = mis;
    s.arr_hi = mis + len;
    s.arr_lo4 = (s.arr_lo + G - 1) & ~int64_t(G - 1);
    s.arr_hi4 = s.arr_hi & ~int64_t(G - 1);
    s.u_lo = mis + lo;
    s.u_hi = mis + hi;
    s.head = s.u_lo;
    s.c_first = s.u_lo >> Cfg::CH_LOG2;
    s.c_last = (s.u_hi > s.u_lo) ? ((s.u_hi - 1) >> Cfg::CH_LOG2) : s.c_first - 1;
    s.next_issue = s.c_first;
    s.next_wait = 0;
}

// Thread 0 only: request chunk c of side s into its ring slots.  A chunk
// that lies wholly inside the CTA's part and the array's aligned interior is
// one bulk copy per array.  Otherwise the 16-byte aligned body goes through
// a bulk copy and the at most (G - 1) + (G - 1) elements at the two ends of
// the side array that do not fill a 16-byte group are loaded with plain
// loads; those
// stores are published to the other threads by the barrier's arrive
// (release) and their wait (acquire).
template <typename Cfg, typename K, bool V>
__device__ __forceinline__ void issue_chunk(SideStream& s, int64_t c, K* ring_k, uint32_t* ring_v,
                                            uint64_t* bars, uint64_t policy) {
    constexpr int E = KeyGeom<K>::E, G = KeyGeom<K>::G;
    static_assert(!V || E == 4, "values are 32-bit and share the keys' u positions");
    const int64_t cs = c << Cfg::CH_LOG2;
    const int64_t ce = cs + Cfg::CH;
    uint64_t* bar = &bars[(int)(c - s.c_first) & (Cfg::NCH - 1)];
    // A chunk that lands at slot 0 also fills the overhang (its first OVH
    // elements again at slot RING), in the same barrier transaction.
    const bool first_slot = ((uint32_t)cs & Cfg::RMASK) == 0;
    if (cs >= s.u_lo && ce <= s.u_hi && cs >= s.arr_lo4 && ce <= s.arr_hi4) {
        const uint32_t slot = (uint32_t)cs & Cfg::RMASK;
        const uint32_t ovh = first_slot ? (uint32_t)Cfg::OVH : 0u;
        mbar_arrive_expect_tx(bar, ((uint32_t)Cfg::CH + ovh) * (uint32_t)E * (V ? 2u : 1u));
        bulk_copy_g2s(ring_k + slot, s.base16 + E * cs, Cfg::CH * E, bar, policy);
        if (V) bulk_copy_g2s(ring_v + slot, s.vbase16 + 4 * cs, Cfg::CH * 4, bar, policy);
        if (first_slot) {
            bulk_copy_g2s(ring_k + Cfg::RING, s.base16 + E * cs, Cfg::OVH * E, bar, policy);
            if (V) bulk_copy_g2s(ring_v + Cfg::RING, s.vbase16 + 4 * cs, Cfg::OVH * 4, bar, policy);
        }
        return;
    }
    const int64_t s0 = cs > s.u_lo ? cs : s.u_lo;
    const int64_t e0 = ce < s.u_hi ? ce : s.u_hi;
    int64_t bs = s0 & ~int64_t(G - 1);
    if (bs < s.arr_lo4) bs = s.arr_lo4;
    int64_t be = (e0 + G - 1) & ~int64_t(G - 1);
    if (be > s.arr_hi4) be = s.arr_hi4;
    const K* gk = reinterpret_cast<const K*>(s.base16);
    const uint32_t* gv = reinterpret_cast<const uint32_t*>(s.vbase16);
    bool plain = false;
    uint32_t bytes = 0;
    int64_t p0 = s0, p1 = e0, q0 = e0, q1 = e0;  // plain-load intervals [p0,p1) and [q0,q1)
    if (be > bs) {
        p1 = bs;
        q0 = be;
        bytes = (uint32_t)(be - bs) * (uint32_t)E;
    }
    for (int64_t u = p0; u < p1; ++u) {
        const uint32_t slot = (uint32_t)u & Cfg::RMASK;
        ring_k[slot] = gk[u];
        if (V) ring_v[slot] = gv[u];
        if (slot < (uint32_t)Cfg::OVH) {
            ring_k[Cfg::RING + slot] = gk[u];
            if (V) ring_v[Cfg::RING + slot] = gv[u];
        }
        plain = true;
    }
    for (int64_t u = q0; u < q1; ++u) {
        const uint32_t slot = (uint32_t)u & Cfg::RMASK;
        ring_k[slot] = gk[u];
        if (V) ring_v[slot] = gv[u];
        if (slot < (uint32_t)Cfg::OVH) {
            ring_k[Cfg::RING + slot] = gk[u];
            if (V) ring_v[Cfg::RING + slot] = gv[u];
        }
        plain = true;
    }
    // the bulk body's part inside the first OVH elements of a slot-0 chunk
    int64_t ms = bs > cs ? bs : cs;
    int64_t me = be < cs + Cfg::OVH ? be : cs + Cfg::OVH;
    const uint32_t mirror = (first_slot && bytes && me > ms) ? (uint32_t)(me - ms) * (uint32_t)E : 0u;
    if (plain) fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, V ? 2 * (bytes + mirror) : bytes + mirror);
    if (bytes) {
        const uint32_t slot = (uint32_t)bs & Cfg::RMASK;
        bulk_copy_g2s(ring_k + slot, s.base16 + E * bs, bytes, bar, policy);
        if (V) bulk_copy_g2s(ring_v + slot, s.vbase16 + 4 * bs, bytes, bar, policy);
    }
    if (mirror) {
        const uint32_t slot = (uint32_t)(ms - cs);
        bulk_copy_g2s(ring_k + Cfg::RING + slot, s.base16 + E * ms, mirror, bar, policy);
        if (V) bulk_copy_g2s(ring_v + Cfg::RING + slot, s.vbase16 + 4 * ms, mirror, bar, policy);
    }
}

// Thread 0 only: request every chunk whose ring slots are free, i.e. whose
// previous occupant (chunk - NCH) lies entirely below the consumed head.
template <typename Cfg, typename K, bool V>
__device__ __forceinline__ void refill(SideStream& s, K* ring_k, uint32_t* ring_v, uint64_t* bars,
                                       uint64_t policy) {
    const int64_t head_chunk = s.head >> Cfg::CH_LOG2;
    while (s.next_issue <= s.c_last && s.next_issue - Cfg::NCH + 1 <= head_chunk) {
        issue_chunk<Cfg, K, V>(s, s.next_issue, ring_k, ring_v, bars, policy);
        ++s.next_issue;
    }
}

// Every thread: wait until all chunks covering u < need_end have landed.
template <typename Cfg>
__device__ __forceinline__ bool wait_window(SideStream& s, int64_t need_end, uint64_t* bars, uint32_t* err) {
    if (need_end <= s.head) return true;
    const int need = (int)(((need_end - 1) >> Cfg::CH_LOG2) - s.c_first);
    for (; s.next_wait <= need; ++s.next_wait) {
        if (!mbar_wait_bounded(&bars[s.next_wait & (Cfg::NCH - 1)], (uint32_t)(s.next_wait >> Cfg::NCH_LOG2) & 1u,
                               err))
            return false;
    }
    return true;
}

// co_rank(d) of the two ring windows, A = ring[(ha + x) & mask] and
// B = ring[RSTRIDE + ((hb + x) & mask)]: the largest i in [lo, hi] with i == lo
// or A[i-1] <= B[d-i] (in the merge order), by a fixed sequence of
// power-of-two steps (no data dependent trip count, so a warp never diverges
// on it).  Offsets are kept in bytes, so each probe is two adds, two masks
// and two loads.
template <typename Cfg, typename K, bool DESC = false>
__device__ __forceinline__ int corank_ring(int d, int lo, int hi, const K* ring, uint32_t ha, uint32_t hb) {
    constexpr uint32_t E = sizeof(K);
    constexpr uint32_t MB = (uint32_t)Cfg::RING * E - 1;  // byte mask of one ring
    const char* rk = reinterpret_cast<const char*>(ring);
    const char* rb = rk + (size_t)Cfg::RSTRIDE * E;       // B region
    const uint32_t xa = ha * E - E;                      // + cand*E: byte of A[cand-1]
    const uint32_t xb = (hb + (uint32_t)d) * E;          // - cand*E: byte of B[d-cand]
    const uint32_t hiE = (uint32_t)hi * E;
    uint32_t loE = (uint32_t)lo * E;
#pragma unroll
    for (int step = Cfg::SEARCH_TOP; step > 0; step >>= 1) {
        const uint32_t candE = loE + (uint32_t)step * E;
        if (candE <= hiE) {
            const K x = *reinterpret_cast<const K*>(rk + ((xa + candE) & MB));
            const K y = *reinterpret_cast<const K*>(rb + ((xb - candE) & MB));
            if (a_first<DESC>(x, y)) loE = candE;
        }
    }
    return (int)(loE / E);
}

// Serial merge of VT outputs from the split (a, b) of the two windows, with
// selects instead of branches: take A unless B's head comes strictly before
// it (ties go to A).  GUARD adds the exhaustion tests needed when a window
// ends before the sub-tile does (the last sub-tile of a range); without GUARD
// all VT steps run.  The heads walk linearly through their side's region (the
// overhang covers the wrap) as byte offsets, and only A's is kept: after v
// steps B's head is at pa0 + pb0 + v * E - pa.  Returns the A position after
// the last step.
template <typename Cfg, typename K, bool V, bool GUARD, bool DESC = false>
__device__ __forceinline__ uint32_t merge_serial(int a, int b, int cnt, int wa, int wb, const K* ring,
                                                 const uint32_t* vring, uint32_t ha, uint32_t hb, K (&keys)[Cfg::VT],
                                                 uint32_t (&vals)[Cfg::VT]) {
    constexpr uint32_t M = Cfg::RMASK;
    constexpr uint32_t E = sizeof(K);
    static_assert(!V || E == 4, "values share the keys' byte offsets");
    const char* rk = reinterpret_cast<const char*>(ring);
    const char* rv = reinterpret_cast<const char*>(vring);
    const uint32_t pa0 = ((ha + (uint32_t)a) & M) * E;
    const uint32_t pb0 = ((uint32_t)Cfg::RSTRIDE + ((hb + (uint32_t)b) & M)) * E;
    const uint32_t sum0 = pa0 + pb0;
    const uint32_t pa_end = pa0 + (uint32_t)(wa - a) * E;
    const uint32_t pb_end = pb0 + (uint32_t)(wb - b) * E;
    uint32_t pa = pa0;
    K ak = *reinterpret_cast<const K*>(rk + pa0);
    K bk = *reinterpret_cast<const K*>(rk + pb0);
    // compare forms of the two heads, each computed once when its key is read
    auto ao = OrderKey<K>::of(ak);
    auto bo = OrderKey<K>::of(bk);
    uint32_t av = 0, bv = 0;
    if (V) {
        av = *reinterpret_cast<const uint32_t*>(rv + pa0);
        bv = *reinterpret_cast<const uint32_t*>(rv + pb0);
    }
#pragma unroll
    for (int v = 0; v < Cfg::VT; ++v) {
        if (!GUARD || v < cnt) {
            const uint32_t pb = sum0 + (uint32_t)v * E - pa;
            const bool p = GUARD ? ((pb >= pb_end) || ((pa < pa_end) && ord_first<DESC>(ao, bo)))
                                 : ord_first<DESC>(ao, bo);
            keys[v] = p ? ak : bk;
            if (V) vals[v] = p ? av : bv;
            const uint32_t pa_next = pa + E;
            const uint32_t off = p ? pa_next : pb + E;  // the next head of the side just taken
            pa = p ? pa_next : pa;
            if (v + 1 < Cfg::VT) {
                const K nk = *reinterpret_cast<const K*>(rk + off);
                const auto no = OrderKey<K>::of(nk);
                ak = p ? nk : ak;
                bk = p ? bk : nk;
                ao = p ? no : ao;
                bo = p ? bo : no;
                if (V) {
                    const uint32_t nv = *reinterpret_cast<const uint32_t*>(rv + off);
                    av = p ? nv : av;
                    bv = p ? bv : nv;
                }
            }
        }
    }
    return (uint32_t)a + (pa - pa0) / E;
}

// A producer publishes a window cut to the data already requested when the
// previous sub-tile's use of its side plus this margin fits in it.
constexpr int kPartialMargin = 128;

// Whether a key type takes the one-sided path below.  Not float64: its
// merges are bound by the consumers' compare conversions, and the extra
// branch measured 3.6 % slower on interleaved float64 data (0.893 -> 0.926
// ms for 2^28 outputs); every other type gained or stayed even.
template <typename K>
struct OneSidedPath {
    static constexpr bool on = true;
};
template <>
struct OneSidedPath<double> {
    static constexpr bool on = false;
};

// Whether the sub-tile's teff outputs all come from one side, decided from
// the windows' ends alone: 1 when A's window holds teff elements and its
// teff-th goes out no later than B's first (or B's window is empty: its
// range is used up); 2 when the same holds for B with B strictly first;
// 0 otherwise.  Long runs of one input (a much shorter other input, runs of
// equal keys) give such sub-tiles; their co-rank is then teff or 0 with no
// search, and the merge is a copy of that side's window.  A cut window is
// never empty, so an empty window means the side has no more data.
template <typename Cfg, typename K, bool DESC>
__device__ __forceinline__ int one_sided(const K* ring, uint32_t ha, uint32_t hb, int wa, int wb, int teff) {
    constexpr uint32_t M = Cfg::RMASK;
    const K* rb = ring + Cfg::RSTRIDE;
    if (wa >= teff && (wb == 0 || a_first<DESC>(ring[(ha + (uint32_t)teff - 1) & M], rb[hb & M]))) return 1;
    if (wb >= teff && (wa == 0 || !a_first<DESC>(ring[ha & M], rb[(hb + (uint32_t)teff - 1) & M]))) return 2;
    return 0;
}

// Copy of cnt (<= VT) consecutive elements of one ring window, from slot
// `from` on, into the thread's output registers (keys and values); the
// overhang past the ring end means the walk needs no wrap mask.
template <typename Cfg, typename K, bool V>
__device__ __forceinline__ void copy_window(const K* rk, const uint32_t* rv, uint32_t from, int cnt,
                                            K (&keys)[Cfg::VT], uint32_t (&vals)[Cfg::VT]) {
    const uint32_t p0 = from & Cfg::RMASK;
#pragma unroll
    for (int v = 0; v < Cfg::VT; ++v) {
        if (v < cnt) {
            keys[v] = rk[p0 + v];
            if (V) vals[v] = rv[p0 + v];
        }
    }
}

// Shared memory of the tile-merge kernel: keys of both rings back to back
// (A ring, then B ring, so one masked index addresses either), values
// likewise, the output stage, the chunk barriers of both sides, the
// producer/consumer barriers and the per-sub-tile window descriptors.
template <typename Cfg, bool V, int E = 4>
struct TileSmem {
    static constexpr size_t ring_bytes = (size_t)2 * Cfg::RSTRIDE * (E + (V ? 4 : 0));
    static constexpr size_t stage_bytes = (size_t)Cfg::STAGE * (E + (V ? 4 : 0));
    // chunk barriers of A and B, ready[2], done[2], stage_free
    static constexpr size_t bar_bytes = (size_t)(2 * Cfg::NCH + 5) * 8;
    // window descriptors: 2 x {ha, hb, wa, wb, teff, partial_a, partial_b, hint},
    // then the abort flag and padding
    static constexpr size_t info_bytes = 2 * 8 * 4 + 8 * 4;
    // the range's two co-ranks when the producer warps search them (int64 x 2)
    static constexpr size_t bound_bytes = 16;
    static constexpr size_t total = ring_bytes + stage_bytes + bar_bytes + info_bytes + bound_bytes;
};

// The tile-merge kernel.  CTA r merges output range r of the geometry,
// C[k0, k1) from A[i0, i1) and B[j0, j1), in sub-tiles of T outputs.  i0 and
// i1 are the co-ranks of k0 and k1: read from `split` when the partition
// kernel wrote them there, else (split == nullptr) found by the two producer
// warps at the start, one rank each (corank_warp), so the merge needs no
// separate launch and no scratch.  Neighbouring CTAs search the rank they
// share the same way, so their ranges meet exactly.  It is warp-specialised: NT
// consumer threads merge; two producer threads (lane 0 of two extra warps)
// own the bulk copies, one per input side.  Per sub-tile s:
//   producers: (window s is published) the A producer releases the stage
//             once the store of s-1 has read it (stage_free) -> find the
//             sub-tile's co-rank r on the two windows -> publish window s+1
//             from data already requested, when it serves (ready[s+1],
//             count 2) -> wait for the consumers (done[s]) -> advance the side's head by
//             its share of r, request freed chunks; the A producer
//             bulk-stores the stage -> publish window s+1 now if it could not
//             be published early
//   consumers: wait ready[s] -> co-rank + serial merge -> wait stage_free
//             (s-1) -> write the stage -> arrive done[s]
// Consumers never run a CTA-wide barrier and keep no streaming state; with
// the next window published while they merge, they rarely wait for it.
template <typename Cfg, typename K, bool V, bool DESC = false>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_CTAS) tile_merge_kernel(MergeGeom<K> g,
                                                                    const int64_t* __restrict__ split,
                                                                    uint32_t* err) {
    constexpr int NT = Cfg::NT;
    constexpr int VT = Cfg::VT;
    constexpr int T = Cfg::T;
    constexpr int E = KeyGeom<K>::E, G = KeyGeom<K>::G;
    using Smem = TileSmem<Cfg, V, E>;

    extern __shared__ __align__(128) unsigned char smem[];
    K* ring = reinterpret_cast<K*>(smem);
    uint32_t* vring = V ? reinterpret_cast<uint32_t*>(ring + 2 * Cfg::RSTRIDE) : nullptr;
    K* stage_k = reinterpret_cast<K*>(smem + Smem::ring_bytes);
    uint32_t* stage_v = V ? reinterpret_cast<uint32_t*>(stage_k + Cfg::STAGE) : nullptr;
    uint64_t* bars_a = reinterpret_cast<uint64_t*>(smem + Smem::ring_bytes + Smem::stage_bytes);
    uint64_t* bars_b = bars_a + Cfg::NCH;
    uint64_t* ready = bars_b + Cfg::NCH;  // [2]
    uint64_t* done = ready + 2;          // [2]
    uint64_t* stage_free = done + 2;     // [1]
    int* info = reinterpret_cast<int*>(stage_free + 1);  // [2][8]: ha, hb, wa, wb, teff, partial a/b, hint
    volatile int* abort_flag = info + 20;
    int64_t* bound_slot = reinterpret_cast<int64_t*>(smem + Smem::ring_bytes + Smem::stage_bytes +
                                                     Smem::bar_bytes + Smem::info_bytes);  // [2]

    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const int64_t seg = r / g.ranges_per_seg;
    const int64_t local = r - seg * g.ranges_per_seg;
    const Segment<K> s = segment_of<K, V>(g, seg);
    const int64_t len = s.m + s.n;
    const int64_t k0 = local * g.range_len;
    if (k0 >= len) return;  // whole CTA
    const int64_t k1 = (k0 + g.range_len < len) ? k0 + g.range_len : len;
    const bool have_split = split != nullptr;
    int64_t i0 = 0, i1 = 0;
    if (have_split) {
        i0 = split[r];
        i1 = (k1 == len) ? s.m : split[r + 1];
        const int64_t j0 = k0 - i0, j1 = k1 - i1;
        if (i0 < 0 || i1 < i0 || i1 > s.m || j0 < 0 || j1 < j0 || j1 > s.n) {
            if (tid == 0) atomicOr(err, kErrBadRange);
            return;  // whole CTA
        }
    }
    const uintptr_t caddr = reinterpret_cast<uintptr_t>(s.ck);
    const int misc = (int)((caddr / E) & (G - 1));

    if (tid == 0) {
        for (int c = 0; c < Cfg::NCH; ++c) {
            mbar_init(&bars_a[c], 1);
            mbar_init(&bars_b[c], 1);
        }
        mbar_init(&ready[0], 2);  // both producers
        mbar_init(&ready[1], 2);
        mbar_init(&done[0], NT + 2);  // the consumers, and both producers once they have read the windows
        mbar_init(&done[1], NT + 2);
        mbar_init(stage_free, 1);
        fence_barrier_init();
        *abort_flag = 0;
    }
    __syncthreads();  // the last CTA-wide barrier: barriers initialised

    if (tid >= NT) {
        // ----------------------------------------------------- producers --
        // Lane 0 of each extra warp: the first streams A, the second B, so
        // the two sides' refills and chunk waits run side by side.  The A
        // producer also owns the stage: it bulk-stores it and hands it back.
        int64_t kend = k1;  // end of the outputs this CTA merges
        if (!have_split) {
            // The first producer warp finds co_rank(k0), the second
            // co_rank(k1); they swap results through shared memory.  Each
            // result lies in its rank's legal interval; on unsorted input the
            // two may still cross, and then the range is dropped (the error
            // word says so) by publishing no sub-tile.
            const bool first = tid < NT + 32;
            const int64_t kk = first ? k0 : k1;
            const int64_t ii = corank_warp<K, DESC>(kk, s.ak, s.m, s.bk, s.n, tid & 31);
            if ((tid & 31) == 0) bound_slot[first ? 0 : 1] = ii;
            named_barrier_sync(1, 64);  // the two producer warps
            i0 = bound_slot[0];
            i1 = bound_slot[1];
            if (i1 < i0 || k1 - i1 < k0 - i0) {
                if (tid == NT) atomicOr(err, kErrBadRange);
                i0 = i1 = 0;
                kend = k0;
            }
        }
        if ((tid & 31) != 0) return;
        const int64_t j0 = (kend == k0) ? 0 : k0 - i0;
        const int64_t j1 = (kend == k0) ? 0 : k1 - i1;
        const bool side_a = tid == NT;
        SideStream S;
        if (side_a) {
            side_init<Cfg, K>(S, s.ak, s.av, s.m, i0, i1);
        } else {
            side_init<Cfg, K>(S, s.bk, s.bv, s.n, j0, j1);
        }
        K* rk = side_a ? ring : ring + Cfg::RSTRIDE;
        uint32_t* rv = V ? (side_a ? vring : vring + Cfg::RSTRIDE) : nullptr;
        uint64_t* bars = side_a ? bars_a : bars_b;
        char* cbase16 = reinterpret_cast<char*>(caddr & ~uintptr_t(15));
        char* cvbase16 = V ? reinterpret_cast<char*>(reinterpret_cast<uintptr_t>(s.cv) & ~uintptr_t(15)) : nullptr;
        const uint64_t policy = l2_policy_evict_first();
        refill<Cfg, K, V>(S, rk, rv, bars, policy);
        int64_t kdone = k0;
        bool failed = false;
        int64_t first_new = S.c_first;  // chunks from here on were requested by the latest refill

        // Publish this side's window of the sub-tile merged in iteration `it`
        // (outputs from kd; this side's data from head).  A whole window
        // covers min(T, rest of the range) elements.  A cut window covers only
        // the part requested before `avail_chunk` (landed by now or soon):
        // used when it still holds `prev_used` (this side's use in the sub-tile
        // before) plus a margin, and checked for exactness by both producers
        // before the sub-tile counts.  early: publishing before the previous
        // sub-tile's consumers are done, from data already requested; returns
        // 0 when that data cannot serve, 1 when published, -1 on a timeout.
        //
        // hint: whether the consumers should test the sub-tile for being
        // one-sided (one_sided): set after a sub-tile whose outputs all came
        // from one side (a run of one side usually goes on), and for the
        // first and any redone sub-tile.  Interleaved data then never pays
        // for the test; a run that starts inside a sub-tile is merged there
        // and copied from the next sub-tile on.
        auto publish = [&](int it, int64_t kd, int64_t head, int64_t avail_chunk, int prev_used, bool force_full,
                           bool early, int hint) -> int {
            const int teff = (int)((kend - kd) < T ? (kend - kd) : T);
            int* inf = info + 8 * (it & 1);
            if (teff == 0) {  // every sub-tile is merged: tell the consumers to stop
                if (side_a) inf[4] = 0;
                mbar_arrive(&ready[it & 1]);
                return 1;
            }
            const int need = (int)((S.u_hi - head) < T ? (S.u_hi - head) : T);
            const int64_t avail_end = (avail_chunk << Cfg::CH_LOG2) < S.u_hi ? (avail_chunk << Cfg::CH_LOG2) : S.u_hi;
            const int landed = (int)(avail_end - head < need ? avail_end - head : need);
            int w = need;
            int partial = 0;
            const bool can_cut = !force_full && teff == T && prev_used >= 0 && prev_used + kPartialMargin <= landed;
            if (landed < need) {
                if (can_cut) {
                    w = landed;
                    partial = 1;
                } else if (early) {
                    return 0;
                }
            }
            const bool ok = wait_window<Cfg>(S, head + w, bars, err);
            inf[side_a ? 0 : 1] = (int)((uint32_t)head & Cfg::RMASK);
            inf[side_a ? 2 : 3] = w;
            inf[side_a ? 5 : 6] = partial;
            if (side_a) {
                inf[4] = teff;
                inf[7] = hint;
            }
            if (!ok) *abort_flag = 1;
            mbar_arrive(&ready[it & 1]);  // release: this side's window and descriptor
            return ok ? 1 : -1;
        };

        if (publish(0, kdone, S.head, S.c_first, -1, true, false, 1) < 0) failed = true;
        for (int it = 0; !failed; ++it) {
            // Sub-tile `it` is published; the consumers may be merging it.
            const int teff = (int)((kend - kdone) < T ? (kend - kdone) : T);
            if (teff == 0) break;  // the stop mark was published
            if (side_a && it > 0) {
                bulk_wait_read_all();  // the previous sub-tile's store has read the stage
                mbar_arrive(stage_free);
            }
            const int* inf = info + 8 * (it & 1);
            if (!mbar_wait_bounded(&ready[it & 1], (uint32_t)(it >> 1) & 1u, err)) {
                *abort_flag = 1;
                failed = true;
                break;
            }
            // Both windows are visible: each producer finds the sub-tile's
            // co-rank r on them itself.  A cut window is exact only when
            // r < wa and T - r < wb (every output's two heads lie inside the
            // windows, so r is the true co-rank); otherwise the sub-tile is
            // merged again with whole windows.  This runs while the consumers
            // merge.
            // When the hint asks for it, a one-sided sub-tile (one_sided) is
            // recognised here exactly as the consumers recognise it: it needs
            // no search, they copy it, and it is exact whatever the windows
            // were cut to.
            const int wa_ = inf[2], wb_ = inf[3];
            const int side = (OneSidedPath<K>::on && inf[7])
                                 ? one_sided<Cfg, K, DESC>(ring, (uint32_t)inf[0], (uint32_t)inf[1], wa_, wb_, teff)
                                 : 0;
            const int r = side == 1   ? teff
                          : side == 2 ? 0
                                      : corank_ring<Cfg, K, DESC>(teff, teff - wb_ > 0 ? teff - wb_ : 0,
                                                                  teff < wa_ ? teff : wa_, ring, (uint32_t)inf[0],
                                                                  (uint32_t)inf[1]);
            const bool redo = side == 0 && (inf[5] | inf[6]) && !(r < wa_ && teff - r < wb_);
            const int used = side_a ? r : teff - r;
            const int hint = (r == teff || r == 0) ? 1 : 0;
            // This producer has read the windows: `done` (which both refills
            // wait for) may now complete, so no refill overwrites a window
            // slot that the other producer is still searching.
            mbar_arrive(&done[it & 1]);
            // Publish the next sub-tile now from what is already requested, so
            // that the consumers find it ready when they finish this one.
            int next = 0;
            if (!redo) {
                next = publish(it + 1, kdone + teff, S.head + used, S.next_issue, used, false, true, hint);
                if (next < 0) {
                    failed = true;
                    break;
                }
            }
            if (!mbar_wait_bounded(&done[it & 1], (uint32_t)(it >> 1) & 1u, err)) {
                *abort_flag = 1;
                failed = true;
                break;
            }
            if (redo) {  // same sub-tile again, with whole windows; nothing stored
                if (publish(it + 1, kdone, S.head, S.next_issue, -1, true, false, 1) < 0) failed = true;
                continue;
            }
            S.head += used;
            first_new = S.next_issue;
            refill<Cfg, K, V>(S, rk, rv, bars, policy);
            if (side_a) {
                // C[kdone, kdone + teff) <- stage.  u = misc + k; stage slot = u - (u0 & ~(G-1)).
                const int64_t cu0 = misc + kdone, cu1 = cu0 + teff;
                const int64_t g0 = cu0 & ~int64_t(G - 1);
                const int64_t bs = (cu0 + G - 1) & ~int64_t(G - 1);
                const int64_t be = cu1 & ~int64_t(G - 1);
                int64_t p1 = cu1, q0 = cu1;
                if (be > bs) {
                    bulk_copy_s2g(cbase16 + E * bs, stage_k + (bs - g0), (uint32_t)(be - bs) * (uint32_t)E, policy);
                    if (V) bulk_copy_s2g(cvbase16 + 4 * bs, stage_v + (bs - g0), (uint32_t)(be - bs) * 4u, policy);
                    p1 = bs;
                    q0 = be;
                }
                K* ck = reinterpret_cast<K*>(cbase16);
                uint32_t* cv = reinterpret_cast<uint32_t*>(cvbase16);
                for (int64_t u = cu0; u < p1; ++u) {
                    ck[u] = stage_k[u - g0];
                    if (V) cv[u] = stage_v[u - g0];
                }
                for (int64_t u = q0; u < cu1; ++u) {
                    ck[u] = stage_k[u - g0];
                    if (V) cv[u] = stage_v[u - g0];
                }
                bulk_commit();
            }
            kdone += teff;
            if (next == 0 && publish(it + 1, kdone, S.head, first_new, used, false, false, hint) < 0) failed = true;
        }
        if (failed) {
            // Let every requested chunk land (bounded) before the CTA's shared
            // memory is released; only the last NCH requests can be pending.
            const int64_t c0 = S.next_issue - Cfg::NCH > S.c_first ? S.next_issue - Cfg::NCH : S.c_first;
            for (int64_t c = c0; c < S.next_issue; ++c) {
                const int rel = (int)(c - S.c_first);
                mbar_wait_bounded(&bars[rel & (Cfg::NCH - 1)], (uint32_t)(rel >> Cfg::NCH_LOG2) & 1u, err);
            }
        }
        if (side_a) bulk_wait_all();
        return;
    }

    // -------------------------------------------------------- consumers --
    const int dthr = tid * VT;
    for (int it = 0;; ++it) {
        if (!mbar_wait_bounded(&ready[it & 1], (uint32_t)(it >> 1) & 1u, err) || *abort_flag) {
            *abort_flag = 1;
            return;
        }
        const int* inf = info + 8 * (it & 1);
        const int teff = inf[4];
        if (teff == 0) return;  // the producers have published the last sub-tile
        const uint32_t ha = (uint32_t)inf[0];
        const uint32_t hb = (uint32_t)inf[1];
        const int wa = inf[2];
        const int wb = inf[3];
        const bool partial = (inf[5] | inf[6]) != 0;
        const int d = dthr < teff ? dthr : teff;
        K keys[VT];
        uint32_t vals[VT];
        const bool full = (teff == T) && (wa == T) && (wb == T);
        const int side = (OneSidedPath<K>::on && inf[7]) ? one_sided<Cfg, K, DESC>(ring, ha, hb, wa, wb, teff) : 0;
        int cnt = VT;
        if (side != 0) {
            // every output of the sub-tile comes from one side: copy it
            cnt = (teff - d < VT) ? teff - d : VT;
            if (side == 1) {
                copy_window<Cfg, K, V>(ring, vring, ha + (uint32_t)d, cnt, keys, vals);
            } else {
                copy_window<Cfg, K, V>(ring + Cfg::RSTRIDE, V ? vring + Cfg::RSTRIDE : nullptr, hb + (uint32_t)d,
                                       cnt, keys, vals);
            }
        } else if (full) {
            const int a = corank_ring<Cfg, K, DESC>(d, 0, d, ring, ha, hb);
            merge_serial<Cfg, K, V, false, DESC>(a, d - a, VT, wa, wb, ring, vring, ha, hb, keys, vals);
        } else if (partial) {
            // Windows cut to the data already requested (teff == T).
            // Searches stay inside them and the merge runs without
            // exhaustion tests; the producers check that the result is exact
            // and, if not, the sub-tile is discarded and published again with
            // whole windows.
            const int lo = d - wb > 0 ? d - wb : 0;
            const int hi = d < wa ? d : wa;
            const int a = corank_ring<Cfg, K, DESC>(d, lo, hi, ring, ha, hb);
            merge_serial<Cfg, K, V, false, DESC>(a, d - a, VT, wa, wb, ring, vring, ha, hb, keys, vals);
        } else {
            cnt = (teff - d < VT) ? teff - d : VT;
            const int lo = d - wb > 0 ? d - wb : 0;
            const int hi = d < wa ? d : wa;
            const int a = corank_ring<Cfg, K, DESC>(d, lo, hi, ring, ha, hb);
            merge_serial<Cfg, K, V, true, DESC>(a, d - a, cnt, wa, wb, ring, vring, ha, hb, keys, vals);
        }
        if (it > 0 && !mbar_wait_bounded(stage_free, (uint32_t)(it - 1) & 1u, err)) {
            *abort_flag = 1;
            return;
        }
        if (cnt == VT) {
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                stage_k[misc + d + v] = keys[v];
                if (V) stage_v[misc + d + v] = vals[v];
            }
        } else {
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                if (v < cnt) {
                    stage_k[misc + d + v] = keys[v];
                    if (V) stage_v[misc + d + v] = vals[v];
                }
            }
        }
        fence_proxy_async_smem();  // stage writes -> visible to the bulk store
        mbar_arrive(&done[it & 1]);  // release: stage written, ring reads done
    }
}

}  // namespace om

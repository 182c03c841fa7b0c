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
//  * The grid-level co-rank is a separate partition kernel that writes one
//    splitter per output range (the pages' thread 0 search per block).
//  * The search is the bounded bisection form of the same co-rank: the
//    largest i in [max(0,k-n), min(k,m)] with i == lower bound or
//    A[i-1] <= B[k-i].  On sorted input it is the pages' i; on any input it
//    stops after ceil(log2(range + 1)) steps.
//  * Ring slots are indexed by the element's 16-byte-aligned address
//    position (u), so every refill is a 16-byte-aligned 1-D bulk copy issued
//    by one thread on the TMA engine and tracked by an mbarrier; the ring
//    size is a power of two so the pages' "% tile_size" wrap is a mask.
//  * Refills run ahead: a chunk is requested as soon as the slots it lands
//    in are consumed, so several sub-tiles of input are in flight while the
//    current one is merged.
//  * Each thread merges VT (odd) outputs into registers; they pass through a
//    shared-memory stage so C is written with coalesced 128-bit streaming
//    stores instead of the pages' per-thread strided writes.
#pragma once

#include <cstdint>

#include "om_ptx.cuh"

namespace om {

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
template <typename K>
__device__ __forceinline__ int64_t corank_global(int64_t k, const K* __restrict__ A, int64_t m,
                                                 const K* __restrict__ B, int64_t n) {
    int64_t lo = k - n > 0 ? k - n : 0;
    int64_t hi = k < m ? k : m;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;  // lo < mid <= hi
        if (__ldg(A + mid - 1) <= __ldg(B + k - mid)) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

// Partition kernel: split[r] = co-rank of the first output of range r within
// its segment.  One thread per range.
template <typename K, bool V>
__global__ void __launch_bounds__(128) partition_kernel(MergeGeom<K> g, int64_t* __restrict__ split) {
    const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (r >= g.nranges) return;
    const int64_t seg = r / g.ranges_per_seg;
    const int64_t local = r - seg * g.ranges_per_seg;
    const Segment<K> s = segment_of<K, V>(g, seg);
    const int64_t len = s.m + s.n;
    int64_t k = local * g.range_len;
    if (k > len) k = len;
    split[r] = corank_global(k, s.ak, s.m, s.bk, s.n);
}

// Batched co-rank of one merge (device ks -> device i).
template <typename K>
__global__ void __launch_bounds__(128) corank_batch_kernel(const int64_t* __restrict__ ks, int64_t count,
                                                           const K* __restrict__ A, int64_t m,
                                                           const K* __restrict__ B, int64_t n,
                                                           int64_t* __restrict__ out) {
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t >= count) return;
    int64_t k = ks[t];
    k = k < 0 ? 0 : (k > m + n ? m + n : k);
    out[t] = corank_global(k, A, m, B, n);
}

// ------------------------------------------------------------ tile merge --

template <int NT_, int VT_, int RING_LOG2_, int CH_LOG2_>
struct TileCfg {
    static constexpr int NT = NT_;
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
    static_assert(VT % 2 == 1, "odd VT keeps the register->stage writes free of bank conflicts");
    static_assert(T % 4 == 0, "sub-tile boundaries stay 16-byte aligned in C");
    static_assert(T + CH <= RING, "a window of T plus one chunk must fit in the ring");
    static_assert(CH >= 4 && NCH >= 2, "chunks are whole 16-byte groups");
};

template <typename Cfg, bool V>
struct TileSmem {
    static constexpr size_t ring_bytes = (size_t)Cfg::RING * 4 * (V ? 4 : 2);
    static constexpr size_t stage_bytes = (size_t)Cfg::STAGE * 4 * (V ? 2 : 1);
    static constexpr size_t bar_bytes = (size_t)2 * Cfg::NCH * 8;
    static constexpr size_t total = ring_bytes + stage_bytes + bar_bytes + 16;
};

// Streaming state of one input side (A or B) of one CTA's output range.
// Positions are in "u" units: u = element index + (address / 4) mod 4 of
// the segment's first element, so u % 4 == 0 exactly at 16-byte boundaries.
struct SideStream {
    const char* base16;   // 16-byte aligned address of u = 0 (keys)
    const char* vbase16;  // same for values
    int64_t arr_lo, arr_hi;  // u extent of the whole side array
    int64_t u_lo, u_hi;      // u extent of this CTA's part
    int64_t head;            // next unconsumed u (A_consumed / B_consumed)
    int64_t c_first, c_last; // chunk indices covering [u_lo, u_hi)
    int64_t next_issue;      // next chunk to request (thread 0)
    int64_t next_wait;       // next chunk this thread has not yet waited for
};

template <typename Cfg>
__device__ __forceinline__ void side_init(SideStream& s, const void* keys, const void* vals, int64_t len,
                                          int64_t lo, int64_t hi) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(keys);
    const int64_t mis = (int64_t)((a >> 2) & 3);
    s.base16 = reinterpret_cast<const char*>(a & ~uintptr_t(15));
    s.vbase16 = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(vals) & ~uintptr_t(15));
    s.arr_lo = mis;
    s.arr_hi = mis + len;
    s.u_lo = mis + lo;
    s.u_hi = mis + hi;
    s.head = s.u_lo;
    s.c_first = s.u_lo >> Cfg::CH_LOG2;
    s.c_last = (s.u_hi > s.u_lo) ? ((s.u_hi - 1) >> Cfg::CH_LOG2) : s.c_first - 1;
    s.next_issue = s.c_first;
    s.next_wait = s.c_first;
}

// Thread 0 only: request chunk c of side s into its ring slots.  The 16-byte
// aligned body goes through one bulk copy per array; the at most 3 + 3
// elements at the two ends of the side array that do not fill a 16-byte group
// are loaded with plain loads.
template <typename Cfg, typename K, bool V>
__device__ __forceinline__ void issue_chunk(SideStream& s, int64_t c, K* ring_k, uint32_t* ring_v,
                                            uint64_t* bars, uint64_t policy) {
    const int64_t s0 = (c << Cfg::CH_LOG2) > s.u_lo ? (c << Cfg::CH_LOG2) : s.u_lo;
    const int64_t e0 = ((c + 1) << Cfg::CH_LOG2) < s.u_hi ? ((c + 1) << Cfg::CH_LOG2) : s.u_hi;
    const int64_t arr_lo4 = (s.arr_lo + 3) & ~int64_t(3);
    const int64_t arr_hi4 = s.arr_hi & ~int64_t(3);
    int64_t bs = s0 & ~int64_t(3);
    if (bs < arr_lo4) bs = arr_lo4;
    int64_t be = (e0 + 3) & ~int64_t(3);
    if (be > arr_hi4) be = arr_hi4;
    uint64_t* bar = &bars[(c - s.c_first) & (Cfg::NCH - 1)];
    const K* gk = reinterpret_cast<const K*>(s.base16);
    const uint32_t* gv = reinterpret_cast<const uint32_t*>(s.vbase16);
    bool plain = false;
    auto load_plain = [&](int64_t u) {
        ring_k[(uint32_t)u & Cfg::RMASK] = gk[u];
        if (V) ring_v[(uint32_t)u & Cfg::RMASK] = gv[u];
        plain = true;
    };
    uint32_t bytes = 0;
    if (be > bs) {
        for (int64_t u = s0; u < bs; ++u) load_plain(u);
        for (int64_t u = be; u < e0; ++u) load_plain(u);
        bytes = (uint32_t)(be - bs) * 4u;
    } else {
        for (int64_t u = s0; u < e0; ++u) load_plain(u);
    }
    if (plain) fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, V ? 2 * bytes : bytes);
    if (bytes) {
        const uint32_t slot = (uint32_t)bs & Cfg::RMASK;
        bulk_copy_g2s(ring_k + slot, s.base16 + 4 * bs, bytes, bar, policy);
        if (V) bulk_copy_g2s(ring_v + slot, s.vbase16 + 4 * bs, bytes, bar, policy);
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
__device__ __forceinline__ bool wait_window(SideStream& s, int64_t need_end, uint64_t* bars,
                                            uint32_t* err) {
    if (need_end <= s.head) return true;
    const int64_t c_need = (need_end - 1) >> Cfg::CH_LOG2;
    for (; s.next_wait <= c_need; ++s.next_wait) {
        const int64_t rel = s.next_wait - s.c_first;
        if (!mbar_wait_bounded(&bars[rel & (Cfg::NCH - 1)], (uint32_t)(rel >> Cfg::NCH_LOG2) & 1u, err))
            return false;
    }
    return true;
}

// co_rank(d) of two ring windows: A window = ring_a[(ha + x) & mask] for
// x < wa, B window likewise.  Same bounded bisection as corank_global.
template <typename Cfg, typename K>
__device__ __forceinline__ int corank_ring(int d, const K* ra, uint32_t ha, int wa, const K* rb,
                                           uint32_t hb, int wb) {
    int lo = d - wb > 0 ? d - wb : 0;
    int hi = d < wa ? d : wa;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const K x = ra[(ha + (uint32_t)(mid - 1)) & Cfg::RMASK];
        const K y = rb[(hb + (uint32_t)(d - mid)) & Cfg::RMASK];
        if (x <= y) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

// The tile-merge kernel.  CTA r merges output range r of the geometry:
// C[k0, k1) from A[i0, i1) and B[j0, j1), where i0 / i1 come from the
// partition kernel.  It walks the range in sub-tiles of T outputs:
//   wait for the window chunks -> per-thread co-rank in the ring -> serial
//   merge of VT outputs -> stage -> barrier -> advance A/B heads by the
//   sub-tile's co-rank, request freed chunks -> 128-bit stores of the stage.
template <typename Cfg, typename K, bool V>
__global__ void __launch_bounds__(Cfg::NT) tile_merge_kernel(MergeGeom<K> g, const int64_t* __restrict__ split,
                                                             uint32_t* err) {
    constexpr int NT = Cfg::NT;
    constexpr int VT = Cfg::VT;
    constexpr int T = Cfg::T;
    constexpr uint32_t RMASK = Cfg::RMASK;
    using Smem = TileSmem<Cfg, V>;

    extern __shared__ __align__(128) unsigned char smem[];
    K* ring_a = reinterpret_cast<K*>(smem);
    K* ring_b = ring_a + Cfg::RING;
    uint32_t* ring_av = V ? reinterpret_cast<uint32_t*>(ring_b + Cfg::RING) : nullptr;
    uint32_t* ring_bv = V ? ring_av + Cfg::RING : nullptr;
    K* stage_k = reinterpret_cast<K*>(smem + Smem::ring_bytes);
    uint32_t* stage_v = V ? reinterpret_cast<uint32_t*>(stage_k + Cfg::STAGE) : nullptr;
    uint64_t* bars_a = reinterpret_cast<uint64_t*>(smem + Smem::ring_bytes + Smem::stage_bytes);
    uint64_t* bars_b = bars_a + Cfg::NCH;
    int* s_misc = reinterpret_cast<int*>(bars_b + Cfg::NCH);  // [0] a_used, [1] abort

    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const int64_t seg = r / g.ranges_per_seg;
    const int64_t local = r - seg * g.ranges_per_seg;
    const Segment<K> s = segment_of<K, V>(g, seg);
    const int64_t len = s.m + s.n;
    const int64_t k0 = local * g.range_len;
    if (k0 >= len) return;  // whole CTA: empty range of a short last segment
    const int64_t k1 = (k0 + g.range_len < len) ? k0 + g.range_len : len;
    const int64_t i0 = split[r];
    const int64_t i1 = (k1 == len) ? s.m : split[r + 1];
    const int64_t j0 = k0 - i0, j1 = k1 - i1;
    if (i0 < 0 || i1 < i0 || i1 > s.m || j0 < 0 || j1 < j0 || j1 > s.n) {
        if (tid == 0) atomicOr(err, kErrBadRange);
        return;  // whole CTA
    }

    SideStream A, B;
    side_init<Cfg>(A, s.ak, s.av, s.m, i0, i1);
    side_init<Cfg>(B, s.bk, s.bv, s.n, j0, j1);
    const uintptr_t caddr = reinterpret_cast<uintptr_t>(s.ck);
    const int64_t misc = (int64_t)((caddr >> 2) & 3);
    K* cbase16 = reinterpret_cast<K*>(caddr & ~uintptr_t(15));
    uint32_t* cvbase16 = V ? reinterpret_cast<uint32_t*>(reinterpret_cast<uintptr_t>(s.cv) & ~uintptr_t(15))
                           : nullptr;

    uint64_t policy = 0;
    if (tid == 0) {
        for (int c = 0; c < Cfg::NCH; ++c) {
            mbar_init(&bars_a[c], 1);
            mbar_init(&bars_b[c], 1);
        }
        fence_barrier_init();
        s_misc[1] = 0;
        policy = l2_policy_evict_first();
    }
    __syncthreads();
    if (tid == 0) {
        refill<Cfg, K, V>(A, ring_a, ring_av, bars_a, policy);
        refill<Cfg, K, V>(B, ring_b, ring_bv, bars_b, policy);
    }
    __syncthreads();  // publishes plain-loaded ragged elements

    bool aborted = false;
    for (int64_t kdone = k0; kdone < k1;) {
        const int teff = (int)((k1 - kdone) < T ? (k1 - kdone) : T);
        const int wa = (int)((A.u_hi - A.head) < T ? (A.u_hi - A.head) : T);
        const int wb = (int)((B.u_hi - B.head) < T ? (B.u_hi - B.head) : T);
        bool ok = wait_window<Cfg>(A, A.head + wa, bars_a, err);
        ok = wait_window<Cfg>(B, B.head + wb, bars_b, err) && ok;
        if (!ok) s_misc[1] = 1;

        const uint32_t ha = (uint32_t)A.head & RMASK;
        const uint32_t hb = (uint32_t)B.head & RMASK;
        const int d = (tid * VT < teff) ? tid * VT : teff;
        const int cnt = (teff - d < VT) ? teff - d : VT;
        int a = corank_ring<Cfg, K>(d, ring_a, ha, wa, ring_b, hb, wb);
        int b = d - a;

        // Serial merge of cnt outputs: take A unless A is exhausted or B's
        // head is strictly smaller (ties go to A).
        K keys[VT];
        uint32_t vals[VT];
        K ak = (a < wa) ? ring_a[(ha + a) & RMASK] : K(0);
        K bk = (b < wb) ? ring_b[(hb + b) & RMASK] : K(0);
#pragma unroll
        for (int v = 0; v < VT; ++v) {
            if (v < cnt) {
                const bool take_a = (b >= wb) || (a < wa && ak <= bk);
                if (take_a) {
                    keys[v] = ak;
                    if (V) vals[v] = ring_av[(ha + a) & RMASK];
                    ++a;
                    if (a < wa) ak = ring_a[(ha + a) & RMASK];
                } else {
                    keys[v] = bk;
                    if (V) vals[v] = ring_bv[(hb + b) & RMASK];
                    ++b;
                    if (b < wb) bk = ring_b[(hb + b) & RMASK];
                }
            }
        }
        if (tid == NT - 1) s_misc[0] = a;  // = co_rank(teff): the A elements this sub-tile used

        const int off = (int)((misc + kdone) & 3);
#pragma unroll
        for (int v = 0; v < VT; ++v) {
            if (v < cnt) {
                stage_k[off + d + v] = keys[v];
                if (V) stage_v[off + d + v] = vals[v];
            }
        }
        __syncthreads();  // ring reads done, stage written, a_used published
        if (s_misc[1]) {
            aborted = true;
            break;
        }
        const int a_used = s_misc[0];
        A.head += a_used;
        B.head += teff - a_used;
        if (tid == 0) {
            refill<Cfg, K, V>(A, ring_a, ring_av, bars_a, policy);
            refill<Cfg, K, V>(B, ring_b, ring_bv, bars_b, policy);
        }

        // C[kdone, kdone + teff) <- stage; u = misc + k, stage slot = u - g0.
        const int64_t cu0 = misc + kdone;
        const int64_t g0 = cu0 & ~int64_t(3);
        const int ngroups = (int)((((cu0 + teff + 3) & ~int64_t(3)) - g0) >> 2);
        for (int q = tid; q < ngroups; q += NT) {
            const int64_t gu = g0 + 4 * q;
            if (gu >= cu0 && gu + 4 <= cu0 + teff) {
                st_global_cs_v4(cbase16 + gu, *reinterpret_cast<const uint4*>(stage_k + 4 * q));
                if (V) st_global_cs_v4(cvbase16 + gu, *reinterpret_cast<const uint4*>(stage_v + 4 * q));
            } else {
                for (int e = 0; e < 4; ++e) {
                    const int64_t u = gu + e;
                    if (u >= cu0 && u < cu0 + teff) {
                        cbase16[u] = stage_k[4 * q + e];
                        if (V) cvbase16[u] = stage_v[4 * q + e];
                    }
                }
            }
        }
        kdone += teff;
        __syncthreads();  // stage reads done before the next sub-tile writes it
    }

    if (aborted && tid == 0) {
        // Let every requested copy land (bounded) before the CTA's shared
        // memory is released.
        for (int side = 0; side < 2; ++side) {
            SideStream* sp = side == 0 ? &A : &B;
            uint64_t* bars = side == 0 ? bars_a : bars_b;
            for (int64_t c = sp->next_wait; c < sp->next_issue; ++c) {
                const int64_t rel = c - sp->c_first;
                mbar_wait_bounded(&bars[rel & (Cfg::NCH - 1)], (uint32_t)(rel >> Cfg::NCH_LOG2) & 1u, err);
            }
        }
    }
}

}  // namespace om

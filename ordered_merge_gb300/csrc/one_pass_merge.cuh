// One-pass tiled merge for merges small enough to finish in one wave of CTAs.
//
// "Tiled 與 Circular Buffer Merge Kernel (Memory Coalescing)", §Block-Level
// Co-Rank 與協同載入: each block finds the co-ranks of its output tile's two
// ends, loads its A and B windows into shared memory cooperatively
// (coalesced), and merges them there with one co-rank search and one short
// sequential merge per thread.  This is that tiled kernel with one tile per
// CTA, no iteration and no circular buffer: when the whole merge fits in one
// wave, a CTA that has only one tile to merge gains nothing from streaming
// it through a ring, and merging all of it at once with every warp is
// quicker than the ring kernel's producer/consumer hand-offs (the merge is
// then bound by latency: the range search, one DRAM round trip for the
// windows, the merge, the stores).
//
// Each thread merges VT (odd) outputs into registers; the outputs go back
// into the shared window (every read of it is done by then) and leave with
// coalesced stores.  Ties take A first, in either order (a_first).
#pragma once

#include <cstdint>

#include "merge_kernels.cuh"
#include "om_ptx.cuh"

namespace om {

template <int NT_, int VT_, int MIN_CTAS_>
struct OnePassCfg {
    static constexpr int NT = NT_;  // threads; the first two warps search the tile's ends
    static constexpr int VT = VT_;
    static constexpr int T = NT * VT;  // outputs per CTA
    static constexpr int MIN_CTAS = MIN_CTAS_;
    static_assert(VT % 2 == 1, "an odd VT keeps the VT-strided shared stores free of bank conflicts");
    static_assert(NT >= 64 && NT % 32 == 0, "two searching warps at least");
};

// Shared memory: T keys (+ T values) for the windows, later the outputs,
// plus 8 spare slots (a head may be read one past its window), then the two
// co-ranks.
template <typename Cfg, typename K, bool V>
constexpr size_t one_pass_smem_bytes() {
    return (size_t)(Cfg::T + 8) * (sizeof(K) + (V ? 4 : 0)) + 16;
}

// Merges C[k0, k1) of one merge (g.run == 0), k0 = blockIdx.x * T.  Launch:
// Cfg::NT threads, one_pass_smem_bytes() of dynamic shared memory,
// ceil((m + n) / T) CTAs.
template <typename Cfg, typename K, bool V, bool DESC = false>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MIN_CTAS) one_pass_merge_kernel(MergeGeom<K> g, uint32_t* err) {
    constexpr int NT = Cfg::NT, VT = Cfg::VT, T = Cfg::T;
    extern __shared__ __align__(16) unsigned char op_smem[];
    K* wk = reinterpret_cast<K*>(op_smem);
    uint32_t* wv = V ? reinterpret_cast<uint32_t*>(wk + T + 8) : nullptr;
    int64_t* bound = reinterpret_cast<int64_t*>(op_smem + (size_t)(T + 8) * (sizeof(K) + (V ? 4 : 0)));

    const int tid = threadIdx.x;
    const int64_t len = g.m + g.n;
    const int64_t k0 = (int64_t)blockIdx.x * T;
    if (k0 >= len) return;  // whole CTA
    const int64_t k1 = k0 + T < len ? k0 + T : len;
    if (tid < 64) {  // warp 0: co_rank(k0); warp 1: co_rank(k1)
        const int64_t kk = tid < 32 ? k0 : k1;
        const int64_t ii = corank_warp<K, DESC>(kk, g.a_keys, g.m, g.b_keys, g.n, tid & 31);
        if ((tid & 31) == 0) bound[tid >> 5] = ii;
    }
    __syncthreads();
    const int64_t i0 = bound[0], i1 = bound[1];
    const int64_t j0 = k0 - i0, j1 = k1 - i1;
    if (i1 < i0 || j1 < j0) {  // only on unsorted input: the two searches crossed
        if (tid == 0) atomicOr(err, kErrBadRange);
        return;  // whole CTA
    }
    const int la = (int)(i1 - i0), lb = (int)(j1 - j0);  // la + lb = k1 - k0 <= T

    // both windows into shared memory, coalesced: A at [0, la), B at
    // [la, la + lb); asynchronous copies, so every element a thread fetches
    // is in flight at once (one DRAM round trip, not one per load)
    for (int x = tid; x < la; x += NT) {
        cp_async_elem<sizeof(K)>(wk + x, g.a_keys + i0 + x);
        if (V) cp_async_elem<4>(wv + x, g.a_vals + i0 + x);
    }
    for (int x = tid; x < lb; x += NT) {
        cp_async_elem<sizeof(K)>(wk + la + x, g.b_keys + j0 + x);
        if (V) cp_async_elem<4>(wv + la + x, g.b_vals + j0 + x);
    }
    cp_async_wait_all();
    __syncthreads();

    const int total = la + lb;
    const int d = tid * VT;
    int cnt = 0;
    K keys[VT];
    uint32_t vals[VT];
    if (d < total) {
        cnt = total - d < VT ? total - d : VT;
        // co_rank(d) of the windows: the largest a in [max(0, d - lb), min(d, la)]
        // with a at the lower bound or A[a-1] <= B[d-a] (in the order)
        int lo = d - lb > 0 ? d - lb : 0;
        int hi = d < la ? d : la;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a_first<DESC>(wk[mid - 1], wk[la + d - mid])) {
                lo = mid;
            } else {
                hi = mid - 1;
            }
        }
        // serial merge of cnt outputs with exhaustion tests; a head read one
        // past its window stays inside the buffer (B's start, or a spare
        // slot) and is never taken
        int ia = lo, ib = la + d - lo;
        const int ea = la, eb = la + lb;
        K ak = wk[ia], bk = wk[ib];
        auto ao = OrderKey<K>::of(ak);
        auto bo = OrderKey<K>::of(bk);
        uint32_t av = V ? wv[ia] : 0u, bv = V ? wv[ib] : 0u;
#pragma unroll
        for (int v = 0; v < VT; ++v) {
            if (v < cnt) {
                const bool p = (ib >= eb) || (ia < ea && ord_first<DESC>(ao, bo));
                keys[v] = p ? ak : bk;
                if (V) vals[v] = p ? av : bv;
                ia += p ? 1 : 0;
                ib += p ? 0 : 1;
                if (v + 1 < VT) {
                    const int nx = p ? ia : ib;  // <= T: inside the buffer
                    const K nk = wk[nx];
                    const auto no = OrderKey<K>::of(nk);
                    ak = p ? nk : ak;
                    bk = p ? bk : nk;
                    ao = p ? no : ao;
                    bo = p ? bo : no;
                    if (V) {
                        const uint32_t nv = wv[nx];
                        av = p ? nv : av;
                        bv = p ? bv : nv;
                    }
                }
            }
        }
    }
    __syncthreads();  // every window read is done: the buffer takes the outputs
#pragma unroll
    for (int v = 0; v < VT; ++v) {
        if (v < cnt) {
            wk[d + v] = keys[v];
            if (V) wv[d + v] = vals[v];
        }
    }
    __syncthreads();
#pragma unroll 4
    for (int x = tid; x < total; x += NT) {
        g.c_keys[k0 + x] = wk[x];
        if (V) g.c_vals[k0 + x] = wv[x];
    }
}

}  // namespace om

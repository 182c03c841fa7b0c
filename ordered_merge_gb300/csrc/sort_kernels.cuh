// Block-level kernels of the stable merge sort on sm_103a.
//
// "排序 (Sorting) 練習題 (Practice - Sorting Foundations and Parallel Radix
// Sort)", merge-sort stages: early stages have many small independent merges
// (parallelism across merges: give different merges to different thread
// blocks); late stages have few large merges (parallelism inside one merge:
// cut it with the co-rank function).  The same page notes that sorting
// networks are often fastest on short sequences.
//
// block_sort_kernel covers the early stages.  One CTA owns a tile of NT*VT
// consecutive elements and, in shared memory, takes every run of length
// run_from inside the tile to length run_to by pairwise merges:
//  * run_from == 1: each thread first sorts its VT consecutive elements in
//    registers with an odd-even transposition network that only swaps when
//    the left key comes strictly after the right one (so equal keys keep
//    their order), then merges upward from runs of VT.
//  * each merge step: thread t produces outputs [t*VT, t*VT + VT) of the
//    merge its slice falls in (VT and the run lengths are powers of two, so a
//    slice never straddles two merges), by a co-rank search in shared memory
//    and a serial merge of VT outputs into registers (ties: earlier run
//    first).
// The kernel may run in place (out == in): a CTA reads its whole tile before
// it writes any of it, and tiles do not overlap.
// Shared memory indices are padded by one element per 128 bytes so that the
// register -> shared writes of VT consecutive elements per thread hit
// distinct banks (4-byte keys: one per 32 elements; 8-byte keys: one per 16).
// Keys of any type of merge_kernels.cuh sort in either order (the order and
// compare forms come from there); values are 32-bit.
#pragma once

#include <cstdint>
#include <limits>

#include "merge_kernels.cuh"
#include "om_ptx.cuh"

namespace om {

__device__ __forceinline__ int pad32(int x) { return x + (x >> 5); }

// Padded index of an E-byte element (x >= 0): one element of padding per
// 128 bytes, i.e. per 32 four-byte or 16 eight-byte elements.
template <typename K>
__device__ __forceinline__ int padk(int x) {
    static_assert(sizeof(K) == 4 || sizeof(K) == 8, "keys of 4 or 8 bytes");
    return x + (x >> (sizeof(K) == 4 ? 5 : 4));
}

// A key that no key comes strictly after in the order: the type's maximum
// (ascending) or lowest value (descending); infinities for floats.
template <typename K, bool DESC>
__device__ __forceinline__ K last_key() {
    if (std::numeric_limits<K>::has_infinity) {
        return DESC ? -std::numeric_limits<K>::infinity() : std::numeric_limits<K>::infinity();
    }
    return DESC ? std::numeric_limits<K>::lowest() : std::numeric_limits<K>::max();
}

template <int NT_, int VT_>
struct BlockSortCfg {
    static constexpr int NT = NT_;
    static constexpr int VT = VT_;
    static constexpr int TILE = NT * VT;
    static constexpr int PADDED = TILE + TILE / 32;
    // CTAs per SM to hold the registers to: 1024 threads' worth (with the
    // shared-memory carveout set to its maximum, that many tiles fit)
    static constexpr int MIN_CTAS = NT >= 1024 ? 1 : 1024 / NT;
    static_assert((VT & (VT - 1)) == 0, "VT must be a power of two");
    static_assert(TILE % 32 == 0, "tile is whole bank rows");
};

// Padded keys (and values) of one tile, plus one 16-byte group so that a
// merge may read the element one past the tile's last without a clamp.
template <typename Cfg, typename K>
constexpr int block_sort_key_slots() {
    return Cfg::TILE + Cfg::TILE / (128 / (int)sizeof(K)) + 16 / (int)sizeof(K);
}

template <typename Cfg, typename K, bool V>
constexpr size_t block_sort_smem_bytes() {
    return (size_t)block_sort_key_slots<Cfg, K>() * sizeof(K) + (V ? (size_t)(Cfg::PADDED + 4) * 4 : 0);
}

// co_rank(d) of A = s[pad(a0 + x)], x < m and B = s[pad(b0 + x)], x < n:
// the largest i in [max(0,d-n), min(d,m)] with i at the lower bound or
// A[i-1] <= B[d-i] (in the order), by power-of-two steps from `top` (a
// power of two with 2 * top > min(d,m) - max(0,d-n)), so every thread of a
// pass takes the same number of steps.
template <typename K, bool DESC>
__device__ __forceinline__ int corank_padded(int d, const K* s, int a0, int m, int b0, int n, int top) {
    int lo = d - n > 0 ? d - n : 0;
    const int hi = d < m ? d : m;
    for (int step = top; step > 0; step >>= 1) {
        const int cand = lo + step;
        if (cand <= hi && a_first<DESC>(s[padk<K>(a0 + cand - 1)], s[padk<K>(b0 + d - cand)])) lo = cand;
    }
    return lo;
}

// One merge step of the block sort: thread outputs [p0, p0 + VT) of the merge
// of the two runs of length w its slice falls in, into k / v (registers);
// returns how many of them exist (VT unless the tile is short).  FULL: the
// tile holds TILE elements, so both runs are whole and every thread has VT
// outputs (no length clamps or per-output guards).
template <int VT, typename K, bool V, bool DESC, bool FULL>
__device__ __forceinline__ int block_merge_step(const K* sk, const uint32_t* sv, int p0, int count, int w, K (&k)[VT],
                                                uint32_t (&v)[VT]) {
    if (!FULL && p0 >= count) return 0;
    const int a0 = p0 & ~(2 * w - 1);
    const int d = p0 - a0;
    const int m = FULL ? w : ((count - a0) < w ? (count - a0) : w);
    const int nb_raw = count - a0 - w;
    const int nb = FULL ? w : (nb_raw <= 0 ? 0 : (nb_raw < w ? nb_raw : w));
    const int b0 = a0 + w;
    const int cnt = FULL ? VT : ((m + nb - d) < VT ? (m + nb - d) : VT);
    const int a = corank_padded<K, DESC>(d, sk, a0, m, b0, nb, w);
    // Serial merge with selects: A and B are adjacent runs, so one index
    // reaches either head (at most one past the tile's last element: the
    // spare slot).  Take A unless A is exhausted or B's head comes strictly
    // before it.
    int ia = a0 + a, ib = b0 + (d - a);
    const int ea = a0 + m, eb = b0 + nb;
    K ak = sk[padk<K>(ia)], bk = sk[padk<K>(ib)];
    auto ao = OrderKey<K>::of(ak);
    auto bo = OrderKey<K>::of(bk);
    uint32_t av = V ? sv[pad32(ia)] : 0u, bv = V ? sv[pad32(ib)] : 0u;
#pragma unroll
    for (int i = 0; i < VT; ++i) {
        if (FULL || i < cnt) {
            const bool p = (ib >= eb) || (ia < ea && ord_first<DESC>(ao, bo));
            k[i] = p ? ak : bk;
            if (V) v[i] = p ? av : bv;
            ia += p ? 1 : 0;
            ib += p ? 0 : 1;
            if (i + 1 < VT) {
                const int idx = p ? ia : ib;  // at most TILE: the spare slot
                const K nk = sk[padk<K>(idx)];
                const auto no = OrderKey<K>::of(nk);
                ak = p ? nk : ak;
                bk = p ? bk : nk;
                ao = p ? no : ao;
                bo = p ? bo : no;
                if (V) {
                    const uint32_t nv = sv[pad32(idx)];
                    av = p ? nv : av;
                    bv = p ? bv : nv;
                }
            }
        }
    }
    return cnt;
}

// The work of one CTA on its tile of `count` elements.  FULL (count ==
// TILE, every tile but the last): the loops over the tile are unrolled and
// carry no bounds tests.
template <typename Cfg, typename K, bool V, bool DESC, bool FULL>
__device__ __forceinline__ void block_sort_tile(const K* in_k, const uint32_t* in_v, K* out_k, uint32_t* out_v,
                                                int64_t base, int count, int run_from, int run_to, K* sk,
                                                uint32_t* sv) {
    constexpr int NT = Cfg::NT;
    constexpr int VT = Cfg::VT;
    const int tid = threadIdx.x;

    if (FULL) {
#pragma unroll
        for (int j = 0; j < VT; ++j) {
            const int p = tid + j * NT;
            sk[padk<K>(p)] = in_k[base + p];
            if (V) sv[pad32(p)] = in_v[base + p];
        }
    } else {
        for (int p = tid; p < count; p += NT) {
            sk[padk<K>(p)] = in_k[base + p];
            if (V) sv[pad32(p)] = in_v[base + p];
        }
    }
    __syncthreads();

    const int p0 = tid * VT;
    K k[VT];
    uint32_t v[VT];
    int w = run_from;
    if (run_from == 1) {
        // Registers: elements past the tile end get a key that nothing comes
        // strictly after, so they stay behind every real element (a swap
        // needs the left key strictly after the right one in the order).
#pragma unroll
        for (int i = 0; i < VT; ++i) {
            const bool real = FULL || p0 + i < count;
            k[i] = real ? sk[padk<K>(p0 + i)] : last_key<K, DESC>();
            if (V) v[i] = real ? sv[pad32(p0 + i)] : 0u;
        }
#pragma unroll
        for (int round = 0; round < VT; ++round) {
#pragma unroll
            for (int i = round & 1; i + 1 < VT; i += 2) {
                if (!a_first<DESC>(k[i], k[i + 1])) {
                    const K tk = k[i];
                    k[i] = k[i + 1];
                    k[i + 1] = tk;
                    if (V) {
                        const uint32_t tv = v[i];
                        v[i] = v[i + 1];
                        v[i + 1] = tv;
                    }
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < VT; ++i) {
            if (FULL || p0 + i < count) {
                sk[padk<K>(p0 + i)] = k[i];
                if (V) sv[pad32(p0 + i)] = v[i];
            }
        }
        __syncthreads();
        w = VT;
    }

    for (; w < run_to; w *= 2) {
        const int cnt = block_merge_step<VT, K, V, DESC, FULL>(sk, sv, p0, count, w, k, v);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < VT; ++i) {
            if (FULL || i < cnt) {
                sk[padk<K>(p0 + i)] = k[i];
                if (V) sv[pad32(p0 + i)] = v[i];
            }
        }
        __syncthreads();
    }

    if (FULL) {
#pragma unroll
        for (int j = 0; j < VT; ++j) {
            const int p = tid + j * NT;
            out_k[base + p] = sk[padk<K>(p)];
            if (V) out_v[base + p] = sv[pad32(p)];
        }
    } else {
        for (int p = tid; p < count; p += NT) {
            out_k[base + p] = sk[padk<K>(p)];
            if (V) out_v[base + p] = sv[pad32(p)];
        }
    }
}

template <typename Cfg, typename K, bool V, bool DESC = false>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MIN_CTAS) block_sort_kernel(const K* in_k, const uint32_t* in_v, K* out_k,
                                                             uint32_t* out_v, int64_t n, int run_from, int run_to) {
    constexpr int TILE = Cfg::TILE;
    constexpr int PADDED_K = block_sort_key_slots<Cfg, K>();
    static_assert(!V || sizeof(K) == 4, "values ride with 4-byte keys");
    extern __shared__ __align__(16) unsigned char bsm_raw[];
    K* sk = reinterpret_cast<K*>(bsm_raw);
    uint32_t* sv = V ? reinterpret_cast<uint32_t*>(sk + PADDED_K) : nullptr;

    const int64_t base = (int64_t)blockIdx.x * TILE;
    const int count = (int)((n - base) < TILE ? (n - base) : TILE);
    if (count == TILE) {
        block_sort_tile<Cfg, K, V, DESC, true>(in_k, in_v, out_k, out_v, base, TILE, run_from, run_to, sk, sv);
    } else {
        block_sort_tile<Cfg, K, V, DESC, false>(in_k, in_v, out_k, out_v, base, count, run_from, run_to, sk, sv);
    }
}

}  // namespace om

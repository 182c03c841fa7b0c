// Internal interface shared by the library's translation units (not part of
// the C ABI): kernel configurations, per-device state, launch counting and
// tracing, argument helpers and the partition + tile-merge launch.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include <cuda_runtime.h>

#include "merge_kernels.cuh"
#include "one_pass_merge.cuh"
#include "ordmerge.h"
#include "sort_kernels.cuh"

namespace om {

// Kernel configurations (consumer threads, outputs per thread, log2 ring,
// log2 chunk; every CTA has two more warps for the producers).
//  merge: 128 consumers x 23 outputs = 2944 outputs per sub-tile; 4096-element
//         rings per side refilled in 1024-element (4 KB) chunks; 45 KB of
//         shared memory, 5 CTAs per SM.  (Measured on GB300 against 1920- and
//         2432-output sub-tiles, 512/2048-element chunks, 8192-element rings
//         and 64- to 256-thread CTAs: per-sub-tile and per-chunk work
//         dominates, so the largest sub-tile and chunk that fit a 4096 ring win.)
using MergeCfg = TileCfg<128, 23, 12, 10>;
//  key+value merge: four rings (keys and values of A and B), so smaller rings
//  keep 5 CTAs per SM: 128 x 11 = 1408 outputs per sub-tile, 2048-element
//  rings, 512-element chunks (best of the shapes measured on GB300).
using PairsCfg = TileCfg<128, 11, 11, 9>;
//  8-byte keys: the same ring bytes as the key+value merge (two 16 KB rings
//  of 2048 keys).  A merge takes half the consumers with about twice the
//  outputs each, so each output pays half a co-rank search: 64 x 23 = 1472
//  outputs per sub-tile and 2 KB chunks for int64 / uint64 (0.705 -> 0.685 ms
//  on 2^28 outputs), 64 x 21 = 1344 and 4 KB chunks for float64, whose every
//  search probe also converts two keys to integers (0.977 -> 0.901 ms).
//  The sort's late passes ran slower with every 64-consumer shape measured
//  (2^26 float64 keys: 5.17 against 5.33-5.74 ms), so sorts keep 128 x 11.
using WideMergeCfg = TileCfg<64, 23, 11, 8>;
using F64MergeCfg = TileCfg<64, 21, 11, 9>;
using WideSortCfg = TileCfg<128, 11, 11, 9>;

// Tile shape of a merge of K keys (with values when V).
template <typename K, bool V>
struct CfgFor {
    using type = MergeCfg;
};
template <typename K>
struct CfgFor<K, true> {
    using type = PairsCfg;
};
template <>
struct CfgFor<int64_t, false> {
    using type = WideMergeCfg;
};
template <>
struct CfgFor<uint64_t, false> {
    using type = WideMergeCfg;
};
template <>
struct CfgFor<double, false> {
    using type = F64MergeCfg;
};

// Tile shape of the sort's late passes.
template <typename K, bool V>
struct SortCfgFor {
    using type = typename std::conditional<sizeof(K) == 8 && !V, WideSortCfg, typename CfgFor<K, V>::type>::type;
};

template <typename Cfg, typename K, bool V>
using SmemOf = TileSmem<Cfg, V, KeyGeom<K>::E>;
template <typename K, bool V>
using SmemFor = SmemOf<typename CfgFor<K, V>::type, K, V>;

// One-pass tile shape of a merge of K keys (with values when V), for merges
// that fit in one wave of it: 128 threads, 8 CTAs per SM (64 registers a
// thread).  4-byte keys alone merge 27 outputs a thread (one wave of 152 x 8
// CTAs covers 4.2 M outputs); keys with values, and 8-byte keys, 15.
template <typename K, bool V>
struct OnePassFor {
    using type = OnePassCfg<128, (sizeof(K) == 4 && !V) ? 27 : 15, 8>;
};

//  sort: one block pass sorts 256 x 16 = 4096-element tiles in shared memory
//        (runs of 16 in registers, then merges of whole pairs of runs per
//        CTA up to 4096); later passes use the tile-merge kernel on each
//        pair of runs.  (8192-element tiles measured even: the extra block
//        level costs what the removed late pass saved.)
using SmallMergeCfg = BlockSortCfg<256, 16>;
constexpr int kEarlyTo = SmallMergeCfg::TILE;  // runs after the block pass

enum KernelKind {
    kKindPartition = 0,
    kKindTileMerge = 1,
    kKindBlockSort = 2,
    kKindCorank = 3,
    kKindBaseline = 4,
    kKindOnePass = 5,
    kNumKinds = 6
};

// ------------------------------------------------------------ device state --

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int resident_merge = 0;  // tile-merge CTAs resident per SM (keys only / with values)
    int resident_merge_v = 0;
    uint32_t* err = nullptr;
    int64_t* corank_slot = nullptr;
    int dev = 0;
    cudaMemPool_t pool = nullptr;  // the library's scratch pool on this device (made by the first sort)
};

// Per-device set-up, once per device (thread-safe): SM count, addresses of
// the library's device words, shared-memory limits and occupancy of the
// merge kernels.  It creates no memory pool and allocates nothing.
om_status device_state(DeviceState** out);

// The library's scratch pool on d's device, created on first use (by the
// first call that needs scratch: a sort).  The pool keeps freed memory
// mapped for the next call (release threshold: unlimited) until
// om_release_scratch() trims it; the caller's default pool is not touched.
om_status scratch_pool(DeviceState* d, cudaMemPool_t* out);

// Stream-ordered scratch from that pool.
inline cudaError_t scratch_alloc(cudaMemPool_t pool, void** p, size_t bytes, cudaStream_t st) {
    return cudaMallocFromPoolAsync(p, bytes, pool, st);
}
inline cudaError_t scratch_free(void* p, cudaStream_t st) { return cudaFreeAsync(p, st); }

// ----------------------------------------------------------------- tracing --

struct TraceRec {
    int kind;
    cudaEvent_t e0, e1;
};

// With tracing on, takes two events and records the first on `stream`.
// Returns whether tracing is on.
bool trace_begin(int kind, cudaStream_t stream, TraceRec* rec);
// Counts one launch and, when `on`, records the second event and files the
// record; returns the launch's error (cudaGetLastError).
cudaError_t trace_end(const TraceRec& rec, bool on, cudaStream_t stream);

// Launches through `launch` (a callable issuing exactly one kernel), counting
// it and, with tracing on, bracketing it with events on `stream`.
template <typename F>
cudaError_t traced(int kind, cudaStream_t stream, F&& launch) {
    TraceRec rec{kind, nullptr, nullptr};
    const bool on = trace_begin(kind, stream, &rec);
    launch();
    return trace_end(rec, on, stream);
}

// ------------------------------------------------------------------ helpers --

inline bool misaligned(const void* p, int bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (uintptr_t)(bytes - 1)) != 0;
}
inline bool misaligned4(const void* p) { return misaligned(p, 4); }

// Whether [a, a + na elements) and [b, b + nb elements) share a byte.
inline bool overlaps(const void* a, int64_t na, const void* b, int64_t nb, int elem = 4) {
    if (na <= 0 || nb <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), a1 = a0 + (uintptr_t)na * (uintptr_t)elem;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b), b1 = b0 + (uintptr_t)nb * (uintptr_t)elem;
    return a0 < b1 && b0 < a1;
}

inline om_status cuda_fail(cudaError_t e) { return e == cudaErrorMemoryAllocation ? OM_ENOMEM : OM_ECUDA; }

// Sub-tiles per CTA output range of a launch over `segs` merges of at most
// `seg_len` outputs, moving bytes_per_output bytes per output, with
// resident_ctas CTAs at a time (see its definition).
int64_t subtiles_per_range(int64_t segs, int64_t seg_len, int64_t T, int64_t bytes_per_output,
                           int64_t resident_ctas);

template <typename K, bool V>
constexpr int64_t bytes_per_output() {
    return 2 * ((int64_t)sizeof(K) + (V ? 4 : 0));
}

// The launches of one merge geometry.  split == nullptr: one tile-merge
// launch whose CTAs find their own range boundaries.  Otherwise split has
// nranges + 1 slots: the partition kernel fills them, then the tile merge
// reads them.
template <typename Cfg, typename K, bool V, bool DESC = false>
cudaError_t launch_merge(const MergeGeom<K>& g, int64_t* split, const DeviceState* d, cudaStream_t st) {
    using Smem = SmemOf<Cfg, K, V>;
    if (split != nullptr) {
        const unsigned pgrid = (unsigned)((g.nranges + 3) / 4);  // one warp per range
        const cudaError_t e =
            traced(kKindPartition, st, [&] { partition_kernel<K, V, DESC><<<pgrid, 128, 0, st>>>(g, split); });
        if (e != cudaSuccess) return e;
    }
    return traced(kKindTileMerge, st, [&] {
        tile_merge_kernel<Cfg, K, V, DESC><<<(unsigned)g.nranges, Cfg::THREADS, Smem::total, st>>>(g, split, d->err);
    });
}

// Outputs one wave of the one-pass kernel covers on the current device (its
// shared-memory limit set and its occupancy queried once per device), or 0
// when the query fails.  The environment variable OM_ONE_PASS_MAX replaces it
// (0: never take the one-pass path); OM_SUBTILES_PER_RANGE or OM_WAVES (the
// tile-merge launch planning) set to a positive value means the ring kernel
// is wanted, so the result is then 0 unless OM_ONE_PASS_MAX says otherwise.
int64_t env_outputs(const char* name, int64_t fallback);

template <typename K, bool V, bool DESC>
int64_t one_pass_capacity(const DeviceState* d) {
    const int64_t forced = env_outputs("OM_ONE_PASS_MAX", -1);
    if (forced >= 0) return forced;
    if (env_outputs("OM_SUBTILES_PER_RANGE", 0) > 0 || env_outputs("OM_WAVES", 0) > 0) return 0;
    using OP = typename OnePassFor<K, V>::type;
    static std::mutex mu;
    static int resident[128];  // CTAs per SM, per device; 0 = not asked yet, -1 = unusable
    std::lock_guard<std::mutex> lk(mu);
    int& r = resident[d->dev & 127];
    if (r == 0) {
        auto* kern = one_pass_merge_kernel<OP, K, V, DESC>;
        int blocks = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)one_pass_smem_bytes<OP, K, V>()) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, OP::NT, one_pass_smem_bytes<OP, K, V>()) !=
                cudaSuccess ||
            blocks < 1) {
            cudaGetLastError();
            r = -1;
        } else {
            r = blocks;
        }
    }
    return r > 0 ? (int64_t)r * d->sm_count * OP::T : 0;
}

// One merge of A[0..m) and B[0..n) into C (values optional); nothing is
// allocated.  A merge that fits in one wave of the one-pass kernel takes it
// (one tile per CTA, merged at once); a larger one takes one tile-merge
// launch whose CTAs stream their output ranges through the rings.  Either
// way each CTA finds its own co-ranks.  `resident_per_sm`: tile-merge CTAs
// of this instantiation resident per SM.
template <typename K, bool V, bool DESC = false>
om_status merge_impl(const K* ak, const uint32_t* av, int64_t m, const K* bk, const uint32_t* bv, int64_t n, K* ck,
                     uint32_t* cv, int resident_per_sm, cudaStream_t st) {
    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return s;
    using Cfg = typename CfgFor<K, V>::type;
    const int64_t total = m + n;
    if (total <= one_pass_capacity<K, V, DESC>(d)) {
        using OP = typename OnePassFor<K, V>::type;
        const int64_t ntiles = (total + OP::T - 1) / OP::T;
        MergeGeom<K> g{ak, av, bk, bv, ck, cv, m, n, 0, OP::T, ntiles, ntiles};
        const cudaError_t e = traced(kKindOnePass, st, [&] {
            one_pass_merge_kernel<OP, K, V, DESC>
                <<<(unsigned)ntiles, OP::NT, one_pass_smem_bytes<OP, K, V>(), st>>>(g, d->err);
        });
        return e == cudaSuccess ? OM_OK : cuda_fail(e);
    }
    const int64_t resident = (int64_t)d->sm_count * (resident_per_sm > 0 ? resident_per_sm : 1);
    const int64_t range_len = subtiles_per_range(1, total, Cfg::T, bytes_per_output<K, V>(), resident) * Cfg::T;
    const int64_t nranges = (total + range_len - 1) / range_len;
    if (nranges > 0x7fffffff) return OM_ERANGE;
    MergeGeom<K> g{ak, av, bk, bv, ck, cv, m, n, 0, range_len, nranges, nranges};
    const cudaError_t e = launch_merge<Cfg, K, V, DESC>(g, nullptr, d, st);
    return e == cudaSuccess ? OM_OK : cuda_fail(e);
}

// Stable merge sort of keys[0..n) in place (values optional), in the
// order DESC.  Pass schedule: one block pass sorts each 4096-element tile in
// shared memory (early stages: many small merges per block); then one
// co-rank-split late pass per doubling of the run length, each one tile-merge
// launch over all pairs of runs.  `resident_per_sm`: tile-merge CTAs of
// this instantiation resident per SM.
template <typename K, bool V, bool DESC = false>
om_status sort_impl(K* keys, uint32_t* vals, int64_t n, int resident_per_sm, cudaStream_t st) {
    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return s;
    {
        // Once per device: the largest shared-memory carveout, so that the
        // block pass runs MIN_CTAS tiles per SM.
        static std::mutex mu;
        static bool carved[128];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return OM_ECUDA;
        std::lock_guard<std::mutex> lk(mu);
        if (!carved[dev]) {
            auto* kern = block_sort_kernel<SmallMergeCfg, K, V, DESC>;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)block_sort_smem_bytes<SmallMergeCfg, K, V>()) != cudaSuccess)
                return OM_ECUDA;
            carved[dev] = true;
        }
    }

    int passes = 0;  // global passes after the block pass
    for (int64_t r = kEarlyTo; r < n; r *= 2) ++passes;
    using Cfg = typename SortCfgFor<K, V>::type;
    const int64_t resident = (int64_t)d->sm_count * (resident_per_sm > 0 ? resident_per_sm : 1);

    K* tk = nullptr;
    uint32_t* tv = nullptr;
    cudaError_t e = cudaSuccess;
    if (passes > 0) {
        cudaMemPool_t pool = nullptr;
        s = scratch_pool(d, &pool);
        if (s != OM_OK) return s;
        e = scratch_alloc(pool, reinterpret_cast<void**>(&tk), (size_t)n * sizeof(K), st);
        if (e == cudaSuccess && V) e = scratch_alloc(pool, reinterpret_cast<void**>(&tv), (size_t)n * 4, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (tk) scratch_free(tk, st);
            if (tv) scratch_free(tv, st);
            return OM_ENOMEM;
        }
    }
    // The block pass writes where the pass count's parity makes the last
    // pass land back in keys / vals.
    K* src_k = (passes % 2 == 0) ? keys : tk;
    uint32_t* src_v = (passes % 2 == 0) ? vals : tv;
    K* dst_k = (passes % 2 == 0) ? tk : keys;
    uint32_t* dst_v = (passes % 2 == 0) ? tv : vals;

    {
        // run sort and early merges in one launch: every CTA sorts 16
        // elements per thread in registers, then merges runs 16 -> ... ->
        // 1024 -> ... -> kEarlyTo in shared memory (whole pairs per CTA)
        const unsigned grid = (unsigned)((n + SmallMergeCfg::TILE - 1) / SmallMergeCfg::TILE);
        e = traced(kKindBlockSort, st, [&] {
            block_sort_kernel<SmallMergeCfg, K, V, DESC>
                <<<grid, SmallMergeCfg::NT, block_sort_smem_bytes<SmallMergeCfg, K, V>(), st>>>(
                    keys, vals, src_k, src_v, n, 1, kEarlyTo);
        });
    }
    for (int64_t r = kEarlyTo; e == cudaSuccess && r < n; r *= 2) {
        // late pass: co-rank split of each pair of runs into output ranges
        // (each CTA finds the boundaries of its own range)
        const int64_t npairs = (n + 2 * r - 1) / (2 * r);
        const int64_t seg = 2 * r < n ? 2 * r : n;
        const int64_t range_len =
            subtiles_per_range(npairs, seg, Cfg::T, bytes_per_output<K, V>(), resident) * Cfg::T;
        const int64_t rps = (2 * r + range_len - 1) / range_len;
        MergeGeom<K> g{src_k, src_v, nullptr, nullptr, dst_k, dst_v, n, 0, r, range_len, rps, npairs * rps};
        if (g.nranges > 0x7fffffff) {
            e = cudaErrorInvalidValue;
            break;
        }
        e = launch_merge<Cfg, K, V, DESC>(g, nullptr, d, st);
        K* t = src_k;
        src_k = dst_k;
        dst_k = t;
        uint32_t* tq = src_v;
        src_v = dst_v;
        dst_v = tq;
    }
    if (passes > 0) {
        scratch_free(tk, st);
        if (V) scratch_free(tv, st);
    }
    return e == cudaSuccess ? OM_OK : cuda_fail(e);
}

}  // namespace om

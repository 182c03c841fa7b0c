// Two merges without shared memory, kept only as comparison rows: what the
// shared-memory ring design of tile_merge_kernel buys on this GPU is
// measured against them.  Neither is a fast path.
//
//  * one_thread_merge_kernel: one device thread merges everything, the
//    sequential baseline on the GPU's own memory system ("merge_path.cu"
//    times such a one-thread device merge).
//  * slice_merge_kernel: the basic parallel merge of "Co-rank Function 實作與
//    Basic Parallel Merge Kernel", §Basic Parallel Merge Kernel: thread t owns
//    the output slice [t * per_thread, (t + 1) * per_thread); it finds the
//    co-ranks of both ends of its slice in global memory, then merges the two
//    input intervals between them straight from global memory.  per_thread is
//    the knob "merge_path.cu" sweeps.
#pragma once

#include <cstdint>

#include "merge_kernels.cuh"

namespace om {

// C[0, la + lb) = stable merge of a[0, la) and b[0, lb) (ties: a first),
// keeping the two current heads in registers: one load per output, and the
// side that runs out first ends the merged part; the other side's rest is
// copied after it.
template <typename K>
__device__ __forceinline__ void merge_intervals(const K* __restrict__ a, int64_t la, const K* __restrict__ b,
                                                int64_t lb, K* __restrict__ c) {
    int64_t ia = 0, ib = 0;
    if (la > 0 && lb > 0) {
        K ha = a[0], hb = b[0];
        for (;;) {
            const bool take_a = a_first<false>(ha, hb);
            c[ia + ib] = take_a ? ha : hb;
            if (take_a) {
                if (++ia == la) break;
                ha = a[ia];
            } else {
                if (++ib == lb) break;
                hb = b[ib];
            }
        }
    }
    for (; ia < la; ++ia) c[ia + ib] = a[ia];
    for (; ib < lb; ++ib) c[ia + ib] = b[ib];
}

// Launch with one block of one thread.
template <typename K>
__global__ void __launch_bounds__(1) one_thread_merge_kernel(const K* __restrict__ A, int64_t m,
                                                             const K* __restrict__ B, int64_t n,
                                                             K* __restrict__ C) {
    if (blockIdx.x == 0 && threadIdx.x == 0) merge_intervals<K>(A, m, B, n, C);
}

// Launch with blocks of 256 threads, enough to cover ceil((m + n) / per_thread).
template <typename K>
__global__ void __launch_bounds__(256) slice_merge_kernel(const K* __restrict__ A, int64_t m,
                                                          const K* __restrict__ B, int64_t n, K* __restrict__ C,
                                                          int64_t per_thread) {
    const int64_t total = m + n;
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t >= (total + per_thread - 1) / per_thread) return;
    const int64_t k_lo = t * per_thread;
    const int64_t k_hi = total - k_lo > per_thread ? k_lo + per_thread : total;
    const int64_t i_lo = corank_global<K>(k_lo, A, m, B, n);
    const int64_t i_hi = corank_global<K>(k_hi, A, m, B, n);
    const int64_t j_lo = k_lo - i_lo, j_hi = k_hi - i_hi;
    merge_intervals<K>(A + i_lo, i_hi - i_lo, B + j_lo, j_hi - j_lo, C + k_lo);
}

}  // namespace om

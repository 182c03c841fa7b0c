// The two unstaged merges that "merge_path.cu" measures against each other,
// re-built here to measure on this GPU what the shared-memory ring design
// buys.  Neither is a fast path.
//
//  * one_thread_merge_kernel: the two-pointer merge run by a single device
//    thread ("merge_path.cu", the one-thread device merge): the sequential
//    baseline on the same memory system.
//  * slice_merge_kernel: one thread per slice of `per_thread` outputs; each
//    thread finds where its slice starts with one co-rank search in global
//    memory and then runs the two-pointer merge for its slice straight from
//    global memory ("merge_path.cu", the per-thread co-rank merge;
//    "Co-rank Function 實作與 Basic Parallel Merge Kernel", §Basic Parallel
//    Merge Kernel).  No shared memory and no barrier.  per_thread is the only
//    knob: small slices mean one search per few outputs; large slices mean
//    each warp's 32 lanes read and write 32 places per_thread elements apart.
#pragma once

#include <cstdint>

#include "merge_kernels.cuh"

namespace om {

// Launch with one block of one thread.
template <typename K>
__global__ void __launch_bounds__(1) one_thread_merge_kernel(const K* __restrict__ A, int64_t m,
                                                             const K* __restrict__ B, int64_t n,
                                                             K* __restrict__ C) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    int64_t i = 0, j = 0;
    for (int64_t k = 0; k < m + n; ++k) {
        const bool take_a = j >= n || (i < m && A[i] <= B[j]);
        C[k] = take_a ? A[i++] : B[j++];
    }
}

// Thread t merges C[t * per_thread, min((t + 1) * per_thread, m + n)).
template <typename K>
__global__ void __launch_bounds__(256) slice_merge_kernel(const K* __restrict__ A, int64_t m,
                                                          const K* __restrict__ B, int64_t n, K* __restrict__ C,
                                                          int64_t per_thread) {
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t total = m + n;
    const int64_t k0 = t * per_thread;
    if (k0 >= total) return;
    const int64_t k1 = k0 + per_thread < total ? k0 + per_thread : total;
    int64_t i = corank_global<K>(k0, A, m, B, n);
    int64_t j = k0 - i;
    for (int64_t k = k0; k < k1; ++k) {
        const bool take_a = j >= n || (i < m && A[i] <= B[j]);
        C[k] = take_a ? A[i++] : B[j++];
    }
}

}  // namespace om

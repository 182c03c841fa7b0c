// om_merge_keys / om_merge_sort_keys: the stable co-rank merge and the
// merge sort on keys of other types and in descending order.  The same
// partition, tile-merge and block-sort kernels as the uint32 / int32 calls,
// instantiated per key type and order: only the element size (4 or 8 bytes)
// and the comparison change.  ("merge_path.cu", CPU reference and GPU
// kernels: the method on float keys.)
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "api_internal.cuh"

namespace om {

// Once per device and instantiation: the shared-memory limit of the
// tile-merge kernel of shape Cfg and how many of its CTAs are resident per SM.
template <typename Cfg, typename K, bool V, bool DESC>
static om_status prepare_typed(int* resident) {
    static std::mutex mu;
    static int cached[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return OM_ECUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        using Smem = SmemOf<Cfg, K, V>;
        auto* kern = tile_merge_kernel<Cfg, K, V, DESC>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem::total) !=
            cudaSuccess)
            return OM_ECUDA;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Cfg::THREADS, Smem::total) != cudaSuccess)
            return OM_ECUDA;
        cached[dev] = occ > 0 ? occ : 1;
    }
    *resident = cached[dev];
    return OM_OK;
}

template <typename K, bool DESC>
static om_status typed_merge(const void* A, int64_t m, const void* B, int64_t n, void* C, cudaStream_t st) {
    int resident = 0;
    const om_status s = prepare_typed<typename CfgFor<K, false>::type, K, false, DESC>(&resident);
    if (s != OM_OK) return s;
    return merge_impl<K, false, DESC>(static_cast<const K*>(A), nullptr, m, static_cast<const K*>(B), nullptr, n,
                                      static_cast<K*>(C), nullptr, resident, st);
}

template <typename K>
static om_status typed_merge_order(int order, const void* A, int64_t m, const void* B, int64_t n, void* C,
                                   cudaStream_t st) {
    return order == OM_DESCENDING ? typed_merge<K, true>(A, m, B, n, C, st)
                                  : typed_merge<K, false>(A, m, B, n, C, st);
}

template <typename K, bool V, bool DESC>
static om_status typed_sort(void* keys, uint32_t* vals, int64_t n, cudaStream_t st) {
    int resident = 0;
    const om_status s = prepare_typed<typename SortCfgFor<K, V>::type, K, V, DESC>(&resident);
    if (s != OM_OK) return s;
    return sort_impl<K, V, DESC>(static_cast<K*>(keys), vals, n, resident, st);
}

template <typename K, bool V>
static om_status typed_sort_order(int order, void* keys, uint32_t* vals, int64_t n, cudaStream_t st) {
    return order == OM_DESCENDING ? typed_sort<K, V, true>(keys, vals, n, st)
                                  : typed_sort<K, V, false>(keys, vals, n, st);
}

// Keys of 4 bytes sort with or without values; 8-byte keys without.
template <typename K>
static om_status typed_sort_vals(int order, void* keys, uint32_t* vals, int64_t n, cudaStream_t st) {
    if constexpr (sizeof(K) == 4) {
        if (vals != nullptr) return typed_sort_order<K, true>(order, keys, vals, n, st);
    }
    return typed_sort_order<K, false>(order, keys, nullptr, n, st);
}

static int key_bytes(int key_type) {
    switch (key_type) {
        case OM_KEY_I32:
        case OM_KEY_U32:
        case OM_KEY_F32: return 4;
        case OM_KEY_I64:
        case OM_KEY_U64:
        case OM_KEY_F64: return 8;
        default: return 0;
    }
}

}  // namespace om

using namespace om;

extern "C" {

om_status om_merge_keys(int key_type, int order, const void* A, int64_t m, const void* B, int64_t n, void* C,
                        void* stream) {
    const int eb = key_bytes(key_type);
    if (eb == 0 || (order != OM_ASCENDING && order != OM_DESCENDING)) return OM_EINVAL;
    if (m < 0 || n < 0) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if ((m > 0 && A == nullptr) || (n > 0 && B == nullptr) || C == nullptr) return OM_EINVAL;
    if (misaligned(A, eb) || misaligned(B, eb) || misaligned(C, eb)) return OM_EINVAL;
    if (overlaps(C, total, A, m, eb) || overlaps(C, total, B, n, eb)) return OM_EINVAL;
    cudaStream_t st = (cudaStream_t)stream;
    switch (key_type) {
        case OM_KEY_I32: return typed_merge_order<int32_t>(order, A, m, B, n, C, st);
        case OM_KEY_U32: return typed_merge_order<uint32_t>(order, A, m, B, n, C, st);
        case OM_KEY_F32: return typed_merge_order<float>(order, A, m, B, n, C, st);
        case OM_KEY_I64: return typed_merge_order<int64_t>(order, A, m, B, n, C, st);
        case OM_KEY_U64: return typed_merge_order<uint64_t>(order, A, m, B, n, C, st);
        default: return typed_merge_order<double>(order, A, m, B, n, C, st);
    }
}

om_status om_merge_sort_keys(int key_type, int order, void* keys, uint32_t* vals, int64_t n, void* stream) {
    const int eb = key_bytes(key_type);
    if (eb == 0 || (order != OM_ASCENDING && order != OM_DESCENDING)) return OM_EINVAL;
    if (n < 0) return OM_EINVAL;
    if (n <= 1) return OM_OK;
    if (keys == nullptr || misaligned(keys, eb) || misaligned(vals, 4)) return OM_EINVAL;
    if (n > (int64_t)1 << 40) return OM_ERANGE;
    if (vals != nullptr) {
        if (eb != 4) return OM_EINVAL;  // values ride with 4-byte keys only
        if ((reinterpret_cast<uintptr_t>(keys) & 15) != (reinterpret_cast<uintptr_t>(vals) & 15)) return OM_EINVAL;
        if (overlaps(keys, n, vals, n)) return OM_EINVAL;
    }
    cudaStream_t st = (cudaStream_t)stream;
    switch (key_type) {
        case OM_KEY_I32: return typed_sort_vals<int32_t>(order, keys, vals, n, st);
        case OM_KEY_U32: return typed_sort_vals<uint32_t>(order, keys, vals, n, st);
        case OM_KEY_F32: return typed_sort_vals<float>(order, keys, vals, n, st);
        case OM_KEY_I64: return typed_sort_vals<int64_t>(order, keys, vals, n, st);
        case OM_KEY_U64: return typed_sort_vals<uint64_t>(order, keys, vals, n, st);
        default: return typed_sort_vals<double>(order, keys, vals, n, st);
    }
}

}  // extern "C"

// om_merge_keys: the stable co-rank merge on keys of other types and in
// descending order.  The same partition and tile-merge kernels as
// om_merge_i32, instantiated per key type and order: only the element size
// (4 or 8 bytes) and the comparison change.  ("merge_path.cu", CPU
// reference and GPU kernels: the method on float keys.)
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "api_internal.cuh"

namespace om {

// Once per device and instantiation: the shared-memory limit of the
// tile-merge kernel and how many of its CTAs are resident per SM.
template <typename K, bool DESC>
static om_status prepare_typed(int* resident) {
    static std::mutex mu;
    static int cached[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return OM_ECUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        using Cfg = typename CfgFor<K, false>::type;
        using Smem = SmemFor<K, false>;
        auto* kern = tile_merge_kernel<Cfg, K, false, DESC>;
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
    const om_status s = prepare_typed<K, DESC>(&resident);
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

}  // extern "C"

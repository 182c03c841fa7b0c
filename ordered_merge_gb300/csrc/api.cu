// C ABI of the stable co-rank merge library (declared in include/ordmerge.h):
// argument checks, stream-ordered scratch, kernel launches, the merge-sort
// pass schedule, tracing and the device error word.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "api_internal.cuh"
#include "baseline_kernels.cuh"

namespace om {

// ------------------------------------------------------------ device state --

static __device__ uint32_t g_error_word;
static __device__ int64_t g_corank_slot;

static std::mutex g_mu;
static DeviceState g_devices[128];
static std::mutex g_corank_mu;
static std::atomic<uint64_t> g_launches{0};

template <typename F>
static cudaError_t set_smem(F* kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

om_status device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return OM_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return OM_ECUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) return OM_ECUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.corank_slot), g_corank_slot) != cudaSuccess)
            return OM_ECUDA;
        cudaError_t e = cudaSuccess;
        e = e ? e : set_smem(tile_merge_kernel<MergeCfg, int32_t, false>, SmemFor<int32_t, false>::total);
        e = e ? e : set_smem(tile_merge_kernel<MergeCfg, uint32_t, false>, SmemFor<uint32_t, false>::total);
        e = e ? e : set_smem(tile_merge_kernel<PairsCfg, uint32_t, true>, SmemFor<uint32_t, true>::total);
        if (e != cudaSuccess) return OM_ECUDA;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.resident_merge,
                                                          tile_merge_kernel<MergeCfg, int32_t, false>,
                                                          MergeCfg::THREADS, SmemFor<int32_t, false>::total);
        e = e ? e : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.resident_merge_v,
                                                                   tile_merge_kernel<PairsCfg, uint32_t, true>,
                                                                   PairsCfg::THREADS, SmemFor<uint32_t, true>::total);
        if (e != cudaSuccess) return OM_ECUDA;
        if (d.resident_merge < 1) d.resident_merge = 1;
        if (d.resident_merge_v < 1) d.resident_merge_v = 1;
        d.dev = dev;
        d.ready = true;
    }
    *out = &d;
    return OM_OK;
}

om_status scratch_pool(DeviceState* d, cudaMemPool_t* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d->pool == nullptr) {
        // Freed scratch stays mapped for the next call, so a sort does not
        // map and unmap its second buffer every time the caller synchronises
        // (which a pool with the default threshold of 0 would do).
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = d->dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return OM_ECUDA;
        }
        uint64_t keep = UINT64_MAX;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaGetLastError();
            cudaMemPoolDestroy(pool);
            return OM_ECUDA;
        }
        d->pool = pool;
    }
    *out = d->pool;
    return OM_OK;
}

// ----------------------------------------------------------------- tracing --

static std::mutex g_trace_mu;
static bool g_trace_on = false;
static std::vector<TraceRec> g_trace_recs;
static std::vector<cudaEvent_t> g_event_pool;
static int64_t g_trace_launches[kNumKinds];
static double g_trace_ms[kNumKinds];

static void trace_collect_locked();

// Launches traced but not yet read are summed (waiting for their events)
// once this many are pending, so tracing left on keeps bounded state.
static constexpr size_t kMaxPendingTraces = 1 << 16;

static cudaEvent_t pool_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

bool trace_begin(int kind, cudaStream_t stream, TraceRec* rec) {
    rec->kind = kind;
    bool on;
    {
        std::lock_guard<std::mutex> lk(g_trace_mu);
        on = g_trace_on;
        if (on) {
            rec->e0 = pool_event();
            rec->e1 = pool_event();
            if (rec->e0 == nullptr || rec->e1 == nullptr) {  // no events to be had: this launch goes untraced
                if (rec->e0) g_event_pool.push_back(rec->e0);
                if (rec->e1) g_event_pool.push_back(rec->e1);
                cudaGetLastError();
                on = false;
            }
        }
    }
    if (on) cudaEventRecord(rec->e0, stream);
    return on;
}

cudaError_t trace_end(const TraceRec& rec, bool on, cudaStream_t stream) {
    cudaError_t e = cudaGetLastError();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (on) {
        cudaEventRecord(rec.e1, stream);
        std::lock_guard<std::mutex> lk(g_trace_mu);
        g_trace_recs.push_back(rec);
        if (g_trace_recs.size() >= kMaxPendingTraces) trace_collect_locked();
    }
    return e;
}

static void trace_collect_locked() {
    for (const TraceRec& r : g_trace_recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.e1) == cudaSuccess && cudaEventElapsedTime(&ms, r.e0, r.e1) == cudaSuccess) {
            g_trace_launches[r.kind] += 1;
            g_trace_ms[r.kind] += ms;
        }
        g_event_pool.push_back(r.e0);
        g_event_pool.push_back(r.e1);
    }
    g_trace_recs.clear();
}

// ------------------------------------------------------------------ helpers --

static int64_t env_int(const char* name, int64_t fallback) {
    const char* s = std::getenv(name);
    if (s == nullptr || *s == 0) return fallback;
    char* end = nullptr;
    const long long v = std::strtoll(s, &end, 10);
    return (end != s && v > 0) ? (int64_t)v : fallback;
}

// An output count from the environment (0 allowed), or fallback when unset
// or not a number.
int64_t env_outputs(const char* name, int64_t fallback) {
    const char* s = std::getenv(name);
    if (s == nullptr || *s == 0) return fallback;
    char* end = nullptr;
    const long long v = std::strtoll(s, &end, 10);
    return (end != s && v >= 0) ? (int64_t)v : fallback;
}

// Sub-tiles per CTA output range for one launch over `segs` independent
// merges of at most `seg_len` outputs each (a merge: one segment; a late
// pass of the sort: one segment per pair of runs).  A range never crosses a
// segment, so each segment splits into ceil(seg_len / L) ranges of
// L = per_range * T outputs, and resident_ctas of them run at a time.
//
// The launch's time is modelled as  waves * (overhead + longest range):
// a partial last wave costs as much as a full one (a few CTAs left over
// after a full wave run alone for a whole range), and every range pays a
// fixed cost, its two co-rank searches in global memory and the latency of
// its first chunks, about what moving kRangeOverheadBytes costs a CTA at
// full rate.  Over 1 to 8 waves the rule takes the range length with the
// least modelled time (ties: fewer waves).  For one segment that is always
// one full wave of equal ranges; for the sort's middle passes, whose pairs
// do not divide evenly into the resident CTAs, it is often two to four
// waves of shorter ranges.  The constant is fitted to the measured late
// passes of a 2^26-key sort, where this rule picked each pass's fastest
// measured range length.  OM_WAVES fixes the wave count;
// OM_SUBTILES_PER_RANGE fixes the result.
static constexpr int64_t kRangeOverheadBytes = 24576;

int64_t subtiles_per_range(int64_t segs, int64_t seg_len, int64_t T, int64_t bytes_per_output,
                           int64_t resident_ctas) {
    const int64_t forced = env_int("OM_SUBTILES_PER_RANGE", 0);
    if (forced > 0) return forced;
    if (segs < 1 || seg_len < 1 || T < 1) return 1;
    const int64_t slots = resident_ctas > 0 ? resident_ctas : 1;
    const int64_t qmax = (seg_len + T - 1) / T;
    const int64_t overhead = kRangeOverheadBytes / (bytes_per_output > 0 ? bytes_per_output : 1);
    const int64_t w_fixed = env_int("OM_WAVES", 0);
    const int64_t w_lo = w_fixed > 0 ? w_fixed : 1, w_hi = w_fixed > 0 ? w_fixed : 8;
    auto ranges = [&](int64_t q) { return segs * ((seg_len + q * T - 1) / (q * T)); };
    int64_t best_q = qmax, best_cost = -1;
    for (int64_t w = w_lo; w <= w_hi; ++w) {
        // the shortest ranges that keep the count within w waves
        int64_t lo = 1, hi = qmax;
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (ranges(mid) <= w * slots) hi = mid;
            else lo = mid + 1;
        }
        const int64_t len = lo * T < seg_len ? lo * T : seg_len;
        const int64_t waves = (ranges(lo) + slots - 1) / slots;
        const int64_t cost = waves * (overhead + len);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_q = lo;
        }
    }
    return best_q;
}

}  // namespace om

using namespace om;

extern "C" {

int64_t om_corank_i32(int64_t k, const int32_t* A, int64_t m, const int32_t* B, int64_t n) {
    if (m < 0 || n < 0 || (m > 0 && A == nullptr) || (n > 0 && B == nullptr) || misaligned4(A) || misaligned4(B))
        return -(int64_t)OM_EINVAL;
    if (m > INT64_MAX - n || k < 0 || k > m + n) return -(int64_t)OM_ERANGE;
    if (m == 0 || n == 0) return k < m ? k : m;  // the split is forced
    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return -(int64_t)s;
    std::lock_guard<std::mutex> lk(g_corank_mu);
    cudaError_t e = traced(kKindCorank, (cudaStream_t)0,
                           [&] { corank_one_kernel<int32_t><<<1, 32, 0, 0>>>(k, A, m, B, n, d->corank_slot); });
    if (e != cudaSuccess) return -(int64_t)OM_ECUDA;
    int64_t i = -1;
    if (cudaMemcpy(&i, d->corank_slot, sizeof(i), cudaMemcpyDeviceToHost) != cudaSuccess)
        return -(int64_t)OM_ECUDA;
    return i;
}

om_status om_corank_i32_batch(const int64_t* ks, int64_t count, const int32_t* A, int64_t m, const int32_t* B,
                              int64_t n, int64_t* i_out, void* stream) {
    if (count < 0 || m < 0 || n < 0) return OM_EINVAL;
    if (count == 0) return OM_OK;
    if (ks == nullptr || i_out == nullptr || (m > 0 && A == nullptr) || (n > 0 && B == nullptr) ||
        misaligned4(A) || misaligned4(B))
        return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    const unsigned grid = (unsigned)((count + 127) / 128);
    cudaError_t e = traced(kKindCorank, st,
                           [&] { corank_batch_kernel<int32_t><<<grid, 128, 0, st>>>(ks, count, A, m, B, n, i_out); });
    return e == cudaSuccess ? OM_OK : OM_ECUDA;
}

om_status om_partition_i32(const int32_t* A, int64_t m, const int32_t* B, int64_t n, int64_t tile, int64_t count,
                           int64_t* split, void* stream) {
    if (m < 0 || n < 0 || count < 0 || tile < 1) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    if (count == 0) return OM_OK;
    if (split == nullptr || misaligned(split, 8) || (m > 0 && A == nullptr) || (n > 0 && B == nullptr) ||
        misaligned4(A) || misaligned4(B))
        return OM_EINVAL;
    // split counted in 4-byte units (2 per int64), like A and B
    if (overlaps(split, 2 * count, A, m) || overlaps(split, 2 * count, B, n)) return OM_EINVAL;
    if ((count + 3) / 4 > 0x7fffffff) return OM_ERANGE;
    DeviceState* d = nullptr;
    const om_status s = device_state(&d);
    if (s != OM_OK) return s;
    const int64_t total = m + n;
    // tile boundaries t * tile for t < count, each clamped to m + n in the
    // kernel; ranges_per_seg = count keeps every boundary in the one merge
    const int64_t range_len = tile < total ? tile : (total > 0 ? total : 1);
    MergeGeom<int32_t> g{A, nullptr, B, nullptr, nullptr, nullptr, m, n, 0, range_len, count, count};
    cudaStream_t st = (cudaStream_t)stream;
    const unsigned pgrid = (unsigned)((count + 3) / 4);  // one warp per boundary
    const cudaError_t e =
        traced(kKindPartition, st, [&] { partition_kernel<int32_t, false><<<pgrid, 128, 0, st>>>(g, split); });
    return e == cudaSuccess ? OM_OK : OM_ECUDA;
}

om_status om_merge_i32(const int32_t* A, int64_t m, const int32_t* B, int64_t n, int32_t* C, void* stream) {
    if (m < 0 || n < 0) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if ((m > 0 && A == nullptr) || (n > 0 && B == nullptr) || C == nullptr) return OM_EINVAL;
    if (misaligned4(A) || misaligned4(B) || misaligned4(C)) return OM_EINVAL;
    if (overlaps(C, total, A, m) || overlaps(C, total, B, n)) return OM_EINVAL;
    DeviceState* d = nullptr;
    const om_status s = device_state(&d);
    if (s != OM_OK) return s;
    return merge_impl<int32_t, false>(A, nullptr, m, B, nullptr, n, C, nullptr, d->resident_merge,
                                      (cudaStream_t)stream);
}

om_status om_merge_pairs_u32(const uint32_t* keysA, const uint32_t* valsA, int64_t m, const uint32_t* keysB,
                             const uint32_t* valsB, int64_t n, uint32_t* keysC, uint32_t* valsC, void* stream) {
    if (m < 0 || n < 0) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if ((m > 0 && (keysA == nullptr || valsA == nullptr)) || (n > 0 && (keysB == nullptr || valsB == nullptr)) ||
        keysC == nullptr || valsC == nullptr)
        return OM_EINVAL;
    const void* ptrs[6] = {keysA, valsA, keysB, valsB, keysC, valsC};
    for (const void* p : ptrs)
        if (misaligned4(p)) return OM_EINVAL;
    auto phase = [](const void* p) { return reinterpret_cast<uintptr_t>(p) & 15; };
    if ((m > 0 && phase(keysA) != phase(valsA)) || (n > 0 && phase(keysB) != phase(valsB)) ||
        phase(keysC) != phase(valsC))
        return OM_EINVAL;
    if (overlaps(keysC, total, valsC, total)) return OM_EINVAL;
    for (const void* out : {(const void*)keysC, (const void*)valsC})
        if (overlaps(out, total, keysA, m) || overlaps(out, total, valsA, m) || overlaps(out, total, keysB, n) ||
            overlaps(out, total, valsB, n))
            return OM_EINVAL;
    DeviceState* d = nullptr;
    const om_status s = device_state(&d);
    if (s != OM_OK) return s;
    return merge_impl<uint32_t, true>(keysA, valsA, m, keysB, valsB, n, keysC, valsC, d->resident_merge_v,
                                      (cudaStream_t)stream);
}

om_status om_merge_sort_u32(uint32_t* keys, uint32_t* vals, int64_t n, void* stream) {
    if (n < 0) return OM_EINVAL;
    if (n <= 1) return OM_OK;
    if (keys == nullptr || misaligned4(keys) || misaligned4(vals)) return OM_EINVAL;
    if (n > (int64_t)1 << 40) return OM_ERANGE;
    if (vals != nullptr) {
        if ((reinterpret_cast<uintptr_t>(keys) & 15) != (reinterpret_cast<uintptr_t>(vals) & 15)) return OM_EINVAL;
        if (overlaps(keys, n, vals, n)) return OM_EINVAL;
        DeviceState* d = nullptr;
        const om_status s = device_state(&d);
        if (s != OM_OK) return s;
        return sort_impl<uint32_t, true>(keys, vals, n, d->resident_merge_v, (cudaStream_t)stream);
    }
    DeviceState* d = nullptr;
    const om_status s = device_state(&d);
    if (s != OM_OK) return s;
    return sort_impl<uint32_t, false>(keys, nullptr, n, d->resident_merge, (cudaStream_t)stream);
}

om_status om_merge_i32_one_thread(const int32_t* A, int64_t m, const int32_t* B, int64_t n, int32_t* C,
                                  void* stream) {
    if (m < 0 || n < 0) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if ((m > 0 && A == nullptr) || (n > 0 && B == nullptr) || C == nullptr) return OM_EINVAL;
    if (misaligned4(A) || misaligned4(B) || misaligned4(C)) return OM_EINVAL;
    if (overlaps(C, total, A, m) || overlaps(C, total, B, n)) return OM_EINVAL;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e =
        traced(kKindBaseline, st, [&] { one_thread_merge_kernel<int32_t><<<1, 1, 0, st>>>(A, m, B, n, C); });
    return e == cudaSuccess ? OM_OK : OM_ECUDA;
}

om_status om_merge_i32_slices(const int32_t* A, int64_t m, const int32_t* B, int64_t n, int32_t* C,
                              int64_t per_thread, void* stream) {
    if (m < 0 || n < 0 || per_thread < 1) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if ((m > 0 && A == nullptr) || (n > 0 && B == nullptr) || C == nullptr) return OM_EINVAL;
    if (misaligned4(A) || misaligned4(B) || misaligned4(C)) return OM_EINVAL;
    if (overlaps(C, total, A, m) || overlaps(C, total, B, n)) return OM_EINVAL;
    const int64_t threads = (total + per_thread - 1) / per_thread;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffff) return OM_ERANGE;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = traced(kKindBaseline, st, [&] {
        slice_merge_kernel<int32_t><<<(unsigned)blocks, 256, 0, st>>>(A, m, B, n, C, per_thread);
    });
    return e == cudaSuccess ? OM_OK : OM_ECUDA;
}

const char* om_status_string(int status) {
    switch (status) {
        case OM_OK: return "OM_OK";
        case OM_EINVAL: return "OM_EINVAL: invalid argument (null, negative length, misaligned or overlapping)";
        case OM_ERANGE: return "OM_ERANGE: k or a length out of range";
        case OM_ENOMEM: return "OM_ENOMEM: scratch allocation failed";
        case OM_ECUDA: return "OM_ECUDA: CUDA runtime or launch error";
        case OM_EDEVICE: return "OM_EDEVICE: a kernel reported an error";
        default: return "unknown status";
    }
}

om_status om_device_error(void* stream, uint32_t* detail) {
    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return s;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return OM_ECUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, d->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return OM_ECUDA;
    if (w != 0 && cudaMemset(d->err, 0, sizeof(w)) != cudaSuccess) return OM_ECUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return OM_ECUDA;
    if (detail) *detail = w;
    return w ? OM_EDEVICE : OM_OK;
}

om_status om_trace_enable(int on) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace_on = on != 0;
    return OM_OK;
}

om_status om_trace_reset(void) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    trace_collect_locked();
    for (int k = 0; k < kNumKinds; ++k) {
        g_trace_launches[k] = 0;
        g_trace_ms[k] = 0.0;
    }
    return OM_OK;
}

om_status om_trace_read(int kind, int64_t* launches, double* total_ms) {
    if (kind < 0 || kind >= kNumKinds) return OM_EINVAL;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    trace_collect_locked();
    if (launches) *launches = g_trace_launches[kind];
    if (total_ms) *total_ms = g_trace_ms[kind];
    return OM_OK;
}

uint64_t om_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int64_t om_subtiles_per_range(int64_t segs, int64_t seg_len, int64_t subtile, int64_t bytes_per_output,
                              int64_t resident_ctas) {
    if (segs < 1 || seg_len < 1 || subtile < 1 || bytes_per_output < 1 || resident_ctas < 1) return 0;
    return subtiles_per_range(segs, seg_len, subtile, bytes_per_output, resident_ctas);
}

om_status om_release_scratch(void) {
    DeviceState* d = nullptr;
    const om_status s = device_state(&d);
    if (s != OM_OK) return s;
    if (cudaDeviceSynchronize() != cudaSuccess) return OM_ECUDA;
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        pool = d->pool;
    }
    if (pool == nullptr) return OM_OK;  // no sort has run on this device: nothing is held
    return cudaMemPoolTrimTo(pool, 0) == cudaSuccess ? OM_OK : OM_ECUDA;
}

// ------------------------------------------------- merge without allocating --
//
// om_merge_i32_noalloc: the merge in its two-kernel form -- the partition
// kernel writes one co-rank splitter per output range into the fixed array
// below and the tile-merge kernel reads them (om_merge_i32 instead lets each
// tile-merge CTA find its own range boundaries).  It exists for callers that must
// not allocate device memory on the call path: a process whose device memory
// is already reserved in full by another allocator (a framework's caching
// allocator, a fixed arena), where a stream-ordered allocation could fail for
// lack of memory that is in fact idle; and code with hard latency bounds that
// must not enter an allocator (pool growth, allocator locks) per call.
//
// The array is a file-scope __device__ object: every GPU that loads this
// library holds its 64 KiB until the process exits, and all calls on a device
// share it.  The splitters a call needs are all written by its own partition
// kernel before its tile-merge kernel reads them, so nothing has to be
// cleared between calls; but two calls whose kernels overlap on the GPU (for
// example on two streams) race on the array and may produce wrong output.
constexpr int64_t kNoAllocSplits = 8192;  // int64 slots: 64 KiB
// The documented limit on m + n (2^30).  It is a fixed bound of the API, not
// a kernel limit: output ranges are lengthened as needed so that a merge of
// any length needs at most kNoAllocSplits - 1 of them (at the limit a range
// is 45 sub-tiles long).
constexpr int64_t kNoAllocMaxOutputs = (int64_t)1 << 30;

static __device__ __align__(256) int64_t g_noalloc_splits[kNoAllocSplits];

static std::mutex g_noalloc_mu;
static int64_t* g_noalloc_addr[128];  // device address of g_noalloc_splits, per device

// Once per device, with that device current: the device address of the
// array.  (In host code the array's name is only a host-side stand-in.)
static om_status noalloc_scratch(int64_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return OM_ECUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        int64_t* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_splits) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return OM_ECUDA;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return OM_OK;
}

om_status om_merge_i32_noalloc(const int32_t* A, int64_t m, const int32_t* B, int64_t n, int32_t* C,
                               void* stream) {
    if (m < 0 || n < 0) return OM_EINVAL;
    if (m > INT64_MAX - n) return OM_ERANGE;
    const int64_t total = m + n;
    if (total == 0) return OM_OK;
    if (total > kNoAllocMaxOutputs) return OM_ERANGE;  // beyond the fixed splitter array
    if ((m > 0 && A == nullptr) || (n > 0 && B == nullptr) || C == nullptr) return OM_EINVAL;
    if (misaligned4(A) || misaligned4(B) || misaligned4(C)) return OM_EINVAL;
    if (overlaps(C, total, A, m) || overlaps(C, total, B, n)) return OM_EINVAL;

    DeviceState* d = nullptr;
    om_status s = device_state(&d);
    if (s != OM_OK) return s;
    int64_t* split = nullptr;
    s = noalloc_scratch(&split);
    if (s != OM_OK) return s;

    const int64_t subtiles = (total + MergeCfg::T - 1) / MergeCfg::T;
    int64_t per_range = subtiles_per_range(1, total, MergeCfg::T, 8, (int64_t)d->sm_count * d->resident_merge);
    const int64_t fit = (subtiles + kNoAllocSplits - 2) / (kNoAllocSplits - 1);  // ranges must fit the array
    if (per_range < fit) per_range = fit;
    const int64_t range_len = per_range * MergeCfg::T;
    const int64_t nranges = (total + range_len - 1) / range_len;
    if (nranges + 1 > kNoAllocSplits) return OM_ERANGE;
    MergeGeom<int32_t> g{A, nullptr, B, nullptr, C, nullptr, m, n, 0, range_len, nranges, nranges};
    const cudaError_t e = launch_merge<MergeCfg, int32_t, false>(g, split, d, (cudaStream_t)stream);
    return e == cudaSuccess ? OM_OK : cuda_fail(e);
}

}  // extern "C"

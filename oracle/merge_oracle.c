/*
 * CPU oracle for the stable co-rank merge.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline and
 * reference legs may load or call this file.  The GPU library never links,
 * includes or calls it, and it includes nothing from the GPU library.
 *
 * Every routine is a plain, single-threaded, obviously-correct restatement of
 * the definition it cites.  No blocking, no vectorisation, no reordering.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "Co-rank Function 實作與 Basic Parallel Merge Kernel"
 *   [P2] "Tiled 與 Circular Buffer Merge Kernel (Memory Coalescing)"
 *   [P3] "排序 (Sorting) 練習題 (Practice - Sorting Foundations and
 *         Parallel Radix Sort)"
 *   [P4] "merge_path.cu"
 *
 * Contents
 *   O1  oracle_merge_i32 / _u32 / _f32 / oracle_merge_pairs_u32 /
 *       oracle_merge_keys (six key types, either order): the two-pointer
 *       stable merge.  Equal keys take A first.  ([P1] §Overview, acceptance row;
 *       [P4] mergeCpu, "CPU reference".)
 *   O2  oracle_corank_pages_i32: the co-rank bisection in the order and
 *       notation of [P1] §Binary-Search Implementation (i, j, i_low, j_low,
 *       delta = ceil half-step), with an optional per-iteration trace.
 *   O3  oracle_corank_count_i32: the co-rank by its definition: run the
 *       stable merge for k outputs and count how many came from A
 *       ([P1] §Co-rank Function 定義與不變式; [P4] coRank comment:
 *       "a[0..i) and b[0..j) are exactly the k smallest elements").
 *   O4  oracle_merge_sort_pairs_u32 / oracle_merge_sort_keys: bottom-up
 *       stable merge sort built only from O1 (runs of one, doubling), as in
 *       [P3] (merge-sort stages).
 *   O5  oracle_merge_at_i32: one output element C[k] from O2's split and one
 *       two-pointer step; used for sampled checks at sizes where a full merge
 *       is not wanted.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against the pages' worked example and trace, hand-derived tie cases,
 * closed forms, brute-force stable sorting of the concatenation and
 * library stable sorts.  The unsigned variant of O2 is pinned by brute force
 * over keys on both sides of the sign bit and by random heavy-tie inputs,
 * against the co-rank counted from Python's stable sort
 * (check_corank_pages_u32).  None is "parity unpinned".
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ O1 -- */

/*
 * C = stable merge of sorted A[0..m) and sorted B[0..n).  While both inputs
 * have elements, the smaller head goes out; on a tie A's head goes out (the
 * "<=" side of the acceptance test).  When one input is exhausted the rest of
 * the other is copied.  C must hold m + n elements.
 */
void oracle_merge_i32(const int32_t *A, int64_t m, const int32_t *B,
                      int64_t n, int32_t *C)
{
    int64_t i = 0, j = 0, k = 0;
    while (i < m && j < n) {
        if (B[j] < A[i]) {
            C[k++] = B[j++];
        } else {
            C[k++] = A[i++]; /* A[i] <= B[j]: A first, also on a tie */
        }
    }
    while (i < m) C[k++] = A[i++];
    while (j < n) C[k++] = B[j++];
}

/* O1 on uint32 keys (unsigned order). */
void oracle_merge_u32(const uint32_t *A, int64_t m, const uint32_t *B,
                      int64_t n, uint32_t *C)
{
    int64_t i = 0, j = 0, k = 0;
    while (i < m && j < n) {
        if (B[j] < A[i]) {
            C[k++] = B[j++];
        } else {
            C[k++] = A[i++];
        }
    }
    while (i < m) C[k++] = A[i++];
    while (j < n) C[k++] = B[j++];
}

/* O1 on float keys with the float order of merge_path.cu's mergeCpu: B goes
 * first only when B[j] < A[i] as floats, so keys that compare equal (for
 * example -0.0 and +0.0) keep A first.  Inputs must not hold NaN. */
void oracle_merge_f32(const float *A, int64_t m, const float *B, int64_t n,
                      float *C)
{
    int64_t i = 0, j = 0, k = 0;
    while (i < m && j < n) {
        if (B[j] < A[i]) {
            C[k++] = B[j++];
        } else {
            C[k++] = A[i++];
        }
    }
    while (i < m) C[k++] = A[i++];
    while (j < n) C[k++] = B[j++];
}

/*
 * O1 for keys of other types and for descending order.  `type` is one of the
 * ORACLE_KEY_* codes below; desc = 0 merges nondecreasing inputs, desc = 1
 * nonincreasing ones.  B's head goes out first only when it comes strictly
 * before A's head in the order (ascending: B[j] < A[i]; descending:
 * B[j] > A[i]), so equal keys keep A first in both orders.  Floats compare
 * as IEEE values (-0.0 == +0.0); inputs must not hold NaN.  Returns 0, or
 * -1 for an unknown type.
 */
enum {
    ORACLE_KEY_I32 = 0,
    ORACLE_KEY_U32 = 1,
    ORACLE_KEY_F32 = 2,
    ORACLE_KEY_I64 = 3,
    ORACLE_KEY_U64 = 4,
    ORACLE_KEY_F64 = 5
};

static size_t oracle_key_size(int type)
{
    switch (type) {
    case ORACLE_KEY_I32: case ORACLE_KEY_U32: case ORACLE_KEY_F32: return 4;
    case ORACLE_KEY_I64: case ORACLE_KEY_U64: case ORACLE_KEY_F64: return 8;
    default: return 0;
    }
}

/* 1 when B[j] comes strictly before A[i] in the merge order. */
static int oracle_b_before_a(int type, int desc, const void *A, int64_t i,
                             const void *B, int64_t j)
{
    switch (type) {
    case ORACLE_KEY_I32: {
        int32_t x = ((const int32_t *)A)[i], y = ((const int32_t *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    case ORACLE_KEY_U32: {
        uint32_t x = ((const uint32_t *)A)[i], y = ((const uint32_t *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    case ORACLE_KEY_F32: {
        float x = ((const float *)A)[i], y = ((const float *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    case ORACLE_KEY_I64: {
        int64_t x = ((const int64_t *)A)[i], y = ((const int64_t *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    case ORACLE_KEY_U64: {
        uint64_t x = ((const uint64_t *)A)[i], y = ((const uint64_t *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    default: {
        double x = ((const double *)A)[i], y = ((const double *)B)[j];
        return desc ? (y > x) : (y < x);
    }
    }
}

/* The merge above with optional uint32 values that travel with their keys
 * (va, vb, vc all NULL for keys only). */
static int oracle_merge_keys_vals(int type, int desc, const void *A,
                                  const uint32_t *va, int64_t m, const void *B,
                                  const uint32_t *vb, int64_t n, void *C,
                                  uint32_t *vc)
{
    const size_t e = oracle_key_size(type);
    const unsigned char *a = (const unsigned char *)A;
    const unsigned char *b = (const unsigned char *)B;
    unsigned char *c = (unsigned char *)C;
    int64_t i = 0, j = 0, k = 0;
    if (e == 0) return -1;
    while (i < m && j < n) {
        if (oracle_b_before_a(type, desc, A, i, B, j)) {
            memcpy(c + (size_t)k * e, b + (size_t)j * e, e);
            if (vc != NULL) vc[k] = vb[j];
            ++j;
        } else {
            memcpy(c + (size_t)k * e, a + (size_t)i * e, e);
            if (vc != NULL) vc[k] = va[i];
            ++i;
        }
        ++k;
    }
    for (; i < m; ++i, ++k) {
        memcpy(c + (size_t)k * e, a + (size_t)i * e, e);
        if (vc != NULL) vc[k] = va[i];
    }
    for (; j < n; ++j, ++k) {
        memcpy(c + (size_t)k * e, b + (size_t)j * e, e);
        if (vc != NULL) vc[k] = vb[j];
    }
    return 0;
}

int oracle_merge_keys(int type, int desc, const void *A, int64_t m,
                      const void *B, int64_t n, void *C)
{
    return oracle_merge_keys_vals(type, desc, A, NULL, m, B, NULL, n, C, NULL);
}

/* Same rule on unsigned keys; each value travels with its key. */
void oracle_merge_pairs_u32(const uint32_t *keysA, const uint32_t *valsA,
                            int64_t m, const uint32_t *keysB,
                            const uint32_t *valsB, int64_t n,
                            uint32_t *keysC, uint32_t *valsC)
{
    int64_t i = 0, j = 0, k = 0;
    while (i < m && j < n) {
        if (keysB[j] < keysA[i]) {
            keysC[k] = keysB[j];
            valsC[k] = valsB[j];
            ++j;
        } else {
            keysC[k] = keysA[i];
            valsC[k] = valsA[i];
            ++i;
        }
        ++k;
    }
    for (; i < m; ++i, ++k) { keysC[k] = keysA[i]; valsC[k] = valsA[i]; }
    for (; j < n; ++j, ++k) { keysC[k] = keysB[j]; valsC[k] = valsB[j]; }
}

/* ------------------------------------------------------------------ O2 -- */

/* One row of the [P1] §Trace table: state at the top of an iteration. */
typedef struct {
    int64_t i_low, i, j, j_low;
    int32_t verdict; /* 1: i too big, 2: j too big, 0: accepted */
    int64_t delta;   /* step taken (0 when accepted) */
} oracle_trace_row;

/*
 * co_rank(k, A, m, B, n) following [P1] §Binary-Search Implementation:
 *   start at the upper end i = min(k, m), j = k - i, with lower bounds
 *   i_low = max(0, k - n) and j_low = max(0, k - m);
 *   if A[i-1] > B[j]  (i too big): delta = ceil((i - i_low) / 2),
 *                                  j_low = j, i -= delta, j += delta;
 *   else if B[j-1] >= A[i] (j too big): delta = ceil((j - j_low) / 2),
 *                                  i_low = i, i += delta, j -= delta;
 *   else accept (A[i-1] <= B[j] and B[j-1] < A[i]) and return i.
 * The ceiling step is what makes the loop finish on sorted input ([P1]
 * §Binary-Search Implementation, tip on delta).  On unsorted input the pages'
 * loop may never finish; this oracle stops after 200 iterations and returns
 * -1 so a bad test input cannot hang the test run.  With trace != NULL, up to
 * max_rows rows are written and *rows_out receives the iteration count.
 */
int64_t oracle_corank_pages_i32(int64_t k, const int32_t *A, int64_t m,
                                const int32_t *B, int64_t n,
                                oracle_trace_row *trace, int64_t max_rows,
                                int64_t *rows_out)
{
    int64_t i = (k < m) ? k : m;
    int64_t j = k - i;
    int64_t i_low = (k - n > 0) ? k - n : 0;
    int64_t j_low = (k - m > 0) ? k - m : 0;
    int64_t iter;
    for (iter = 0; iter < 200; ++iter) {
        int32_t verdict;
        int64_t delta = 0;
        if (i > 0 && j < n && A[i - 1] > B[j]) {
            verdict = 1;
        } else if (j > 0 && i < m && B[j - 1] >= A[i]) {
            verdict = 2;
        } else {
            verdict = 0;
        }
        if (trace != NULL && iter < max_rows) {
            trace[iter].i_low = i_low;
            trace[iter].i = i;
            trace[iter].j = j;
            trace[iter].j_low = j_low;
            trace[iter].verdict = verdict;
        }
        if (verdict == 1) {
            delta = (i - i_low + 1) >> 1;
            j_low = j;
            i -= delta;
            j += delta;
        } else if (verdict == 2) {
            delta = (j - j_low + 1) >> 1;
            i_low = i;
            i += delta;
            j -= delta;
        }
        if (trace != NULL && iter < max_rows) trace[iter].delta = delta;
        if (verdict == 0) {
            if (rows_out != NULL) *rows_out = iter + 1;
            return i;
        }
    }
    if (rows_out != NULL) *rows_out = iter;
    return -1;
}

/* Unsigned-key variant of O2 (same steps, unsigned compares). */
int64_t oracle_corank_pages_u32(int64_t k, const uint32_t *A, int64_t m,
                                const uint32_t *B, int64_t n)
{
    int64_t i = (k < m) ? k : m;
    int64_t j = k - i;
    int64_t i_low = (k - n > 0) ? k - n : 0;
    int64_t j_low = (k - m > 0) ? k - m : 0;
    for (int iter = 0; iter < 200; ++iter) {
        if (i > 0 && j < n && A[i - 1] > B[j]) {
            int64_t delta = (i - i_low + 1) >> 1;
            j_low = j;
            i -= delta;
            j += delta;
        } else if (j > 0 && i < m && B[j - 1] >= A[i]) {
            int64_t delta = (j - j_low + 1) >> 1;
            i_low = i;
            i += delta;
            j -= delta;
        } else {
            return i;
        }
    }
    return -1;
}

/* ------------------------------------------------------------------ O3 -- */

/*
 * co_rank by definition: the number of the first k outputs of the stable
 * merge that came from A.  Walks the merge for k steps without writing it.
 */
int64_t oracle_corank_count_i32(int64_t k, const int32_t *A, int64_t m,
                                const int32_t *B, int64_t n)
{
    int64_t i = 0, j = 0;
    if (k < 0 || k > m + n) return -1;
    for (int64_t step = 0; step < k; ++step) {
        if (i < m && (j >= n || A[i] <= B[j])) {
            ++i;
        } else {
            ++j;
        }
    }
    return i;
}

/* ------------------------------------------------------------------ O5 -- */

/*
 * C[k] of the stable merge, from the split (i, k - i) given by O2 and one
 * step of the two-pointer rule: the next output is A[i] unless A is
 * exhausted or B[j] < A[i].  Requires 0 <= k < m + n.  *from_a receives 1
 * when the element came from A.
 */
int32_t oracle_merge_at_i32(int64_t k, const int32_t *A, int64_t m,
                            const int32_t *B, int64_t n, int32_t *from_a)
{
    int64_t i = oracle_corank_pages_i32(k, A, m, B, n, NULL, 0, NULL);
    int64_t j = k - i;
    int take_a = (i < m) && (j >= n || A[i] <= B[j]);
    if (from_a != NULL) *from_a = take_a;
    return take_a ? A[i] : B[j];
}

/* ------------------------------------------------------------------ O4 -- */

/*
 * Stable bottom-up merge sort of (key, value) pairs, built only from O1:
 * runs of one element are merged pairwise into runs of 2, 4, 8, ... until a
 * single run remains.  In every merge the earlier run is A, so equal keys
 * keep their input order ([P3], stable sort; merge-sort stages).  Returns 0,
 * or -1 if the scratch buffers cannot be allocated.
 */
int oracle_merge_sort_pairs_u32(uint32_t *keys, uint32_t *vals, int64_t n)
{
    if (n <= 1) return 0;
    uint32_t *tk = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    uint32_t *tv = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    if (tk == NULL || tv == NULL) {
        free(tk);
        free(tv);
        return -1;
    }
    uint32_t *src_k = keys, *src_v = vals, *dst_k = tk, *dst_v = tv;
    for (int64_t width = 1; width < n; width *= 2) {
        for (int64_t lo = 0; lo < n; lo += 2 * width) {
            int64_t mid = (lo + width < n) ? lo + width : n;
            int64_t hi = (lo + 2 * width < n) ? lo + 2 * width : n;
            oracle_merge_pairs_u32(src_k + lo, src_v + lo, mid - lo,
                                   src_k + mid, src_v + mid, hi - mid,
                                   dst_k + lo, dst_v + lo);
        }
        uint32_t *t;
        t = src_k; src_k = dst_k; dst_k = t;
        t = src_v; src_v = dst_v; dst_v = t;
    }
    if (src_k != keys) {
        memcpy(keys, src_k, (size_t)n * sizeof(uint32_t));
        memcpy(vals, src_v, (size_t)n * sizeof(uint32_t));
    }
    free(tk);
    free(tv);
    return 0;
}

/*
 * O4 for the key types of oracle_merge_keys, either order: the same
 * bottom-up stable merge sort (runs of one, doubling; the earlier run is A),
 * each merge being O1 on typed keys.  vals (uint32, may be NULL) travel with
 * their keys.  Returns 0, -1 for an unknown type, -2 if scratch cannot be
 * allocated.
 */
int oracle_merge_sort_keys(int type, int desc, void *keys, uint32_t *vals,
                           int64_t n)
{
    const size_t e = oracle_key_size(type);
    if (e == 0) return -1;
    if (n <= 1) return 0;
    unsigned char *tk = (unsigned char *)malloc((size_t)n * e);
    uint32_t *tv = vals != NULL ? (uint32_t *)malloc((size_t)n * sizeof(uint32_t)) : NULL;
    if (tk == NULL || (vals != NULL && tv == NULL)) {
        free(tk);
        free(tv);
        return -2;
    }
    unsigned char *src_k = (unsigned char *)keys, *dst_k = tk;
    uint32_t *src_v = vals, *dst_v = tv;
    for (int64_t width = 1; width < n; width *= 2) {
        for (int64_t lo = 0; lo < n; lo += 2 * width) {
            int64_t mid = (lo + width < n) ? lo + width : n;
            int64_t hi = (lo + 2 * width < n) ? lo + 2 * width : n;
            oracle_merge_keys_vals(type, desc,
                                   src_k + (size_t)lo * e, src_v ? src_v + lo : NULL, mid - lo,
                                   src_k + (size_t)mid * e, src_v ? src_v + mid : NULL, hi - mid,
                                   dst_k + (size_t)lo * e, dst_v ? dst_v + lo : NULL);
        }
        unsigned char *t = src_k; src_k = dst_k; dst_k = t;
        uint32_t *tq = src_v; src_v = dst_v; dst_v = tq;
    }
    if (src_k != (unsigned char *)keys) {
        memcpy(keys, src_k, (size_t)n * e);
        if (vals != NULL) memcpy(vals, src_v, (size_t)n * sizeof(uint32_t));
    }
    free(tk);
    free(tv);
    return 0;
}

"""GPU parity of om_merge_i32 and om_corank_i32 against the CPU oracle:
element-by-element, bit-exact, with guard bands around every output.

Sizes span one sub-tile, many sub-tiles, many output ranges and ragged
tails; edge cases cover empty sides, one-element sides, all-equal keys,
disjoint value ranges in both orders, extreme int32 values and pointers that
are not 16-byte aligned.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_i32, guarded_empty, guards_intact, host, shifted

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("merge_path")]


def run_merge(om, A_np, B_np, offs=(0, 0, 0)):
    A = shifted(dev_i32(A_np), offs[0])
    B = shifted(dev_i32(B_np), offs[1])
    total = A_np.size + B_np.size
    buf, C = guarded_empty(total, offs[2])
    om.merge_i32(A, B, C)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    assert guards_intact(buf, total, offs[2]), "merge wrote outside C"
    return host(C)


def check(om, A_np, B_np, offs=(0, 0, 0)):
    got = run_merge(om, A_np, B_np, offs)
    want = oracle.merge_i32(A_np, B_np)
    if not np.array_equal(got, want):
        bad = int(np.flatnonzero(got != want)[0])
        raise AssertionError(f"first mismatch at {bad}: got {got[bad]}, want {want[bad]} "
                             f"(m={A_np.size}, n={B_np.size}, offs={offs})")


def sorted_rand(rng, size, lo, hi):
    return np.sort(rng.integers(lo, hi, size, dtype=np.int64)).astype(np.int32)


def test_pages_worked_example(gpu):
    A = np.array([1, 7, 8, 9, 10], dtype=np.int32)
    B = np.array([7, 10, 10, 12], dtype=np.int32)
    check(gpu, A, B)
    dA, dB = dev_i32(A), dev_i32(B)
    assert [gpu.corank_i32(k, dA, dB) for k in (0, 3, 6, 9)] == [0, 2, 5, 5]


def test_tie_case(gpu):
    check(gpu, np.array([1, 1, 2, 3], np.int32), np.array([1, 2, 2, 4], np.int32))


@pytest.mark.parametrize("m,n", [(0, 0), (0, 1), (1, 0), (0, 5000), (5000, 0), (1, 1), (3, 1), (1, 3),
                                 (1919, 1), (960, 960), (961, 960), (1920, 1920), (7, 100000),
                                 (100000, 7), (12345, 54321), (250001, 249999)])
def test_shapes(gpu, m, n):
    rng = np.random.default_rng(m * 7919 + n)
    check(gpu, sorted_rand(rng, m, -1000, 1000), sorted_rand(rng, n, -1000, 1000))


@pytest.mark.parametrize("span", [1, 2, 16, 1 << 31])
def test_value_spans(gpu, span):
    rng = np.random.default_rng(span)
    lo, hi = (-span, span) if span > 1 else (5, 6)
    check(gpu, sorted_rand(rng, 300007, lo, hi), sorted_rand(rng, 299993, lo, hi))


def test_all_equal_keys(gpu):
    check(gpu, np.full(100003, 42, np.int32), np.full(77777, 42, np.int32))


def test_disjoint_both_orders(gpu):
    A = np.arange(0, 200000, dtype=np.int32)
    B = np.arange(200000, 350001, dtype=np.int32)
    check(gpu, A, B)
    check(gpu, B, A)


def test_int32_extremes(gpu):
    lo, hi = np.iinfo(np.int32).min, np.iinfo(np.int32).max
    A = np.array([lo, lo, -1, 0, hi, hi], np.int32)
    B = np.array([lo, 0, 0, 1, hi], np.int32)
    check(gpu, A, B)
    rng = np.random.default_rng(4)
    A = np.sort(np.concatenate([np.full(5000, lo), rng.integers(lo, hi, 5000), np.full(5000, hi)])).astype(np.int32)
    B = np.sort(np.concatenate([np.full(3000, hi), np.full(3000, lo)])).astype(np.int32)
    check(gpu, A, B)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 3, 0), (0, 0, 2), (1, 2, 3), (3, 3, 1)])
def test_misaligned_pointers(gpu, offs):
    rng = np.random.default_rng(sum(offs))
    check(gpu, sorted_rand(rng, 54321, -500, 500), sorted_rand(rng, 43210, -500, 500), offs)
    check(gpu, sorted_rand(rng, 13, -5, 5), sorted_rand(rng, 1, -5, 5), offs)


@pytest.mark.parametrize("workload", ["evens_odds", "skewed", "uniform"])
def test_workloads_scaled(gpu, workload):
    d = synth.make_host(workload, scale_log2=6)
    check(gpu, d["A"], d["B"])


def test_evens_odds_full_size(gpu):
    d = synth.make_host("evens_odds")
    check(gpu, d["A"], d["B"])


def test_corank_against_oracle(gpu):
    rng = np.random.default_rng(8)
    for span in [3, 1 << 20, 1 << 31]:
        A = sorted_rand(rng, 70001, -span, span)
        B = sorted_rand(rng, 50003, -span, span)
        dA, dB = dev_i32(A), dev_i32(B)
        ks = np.concatenate([[0, 1, A.size, B.size, A.size + B.size - 1, A.size + B.size],
                             rng.integers(0, A.size + B.size + 1, 200)]).astype(np.int64)
        got = host(gpu.corank_i32_batch(torch.from_numpy(ks).cuda(), dA, dB))
        want = np.array([oracle.corank_pages(int(k), A, B) for k in ks])
        assert np.array_equal(got, want)
        for k in ks[:20]:
            assert gpu.corank_i32(int(k), dA, dB) == oracle.corank_count(int(k), A, B)


@pytest.mark.parametrize("m,n,layout", [(65, 3_000_001, "mixed"), (3_000_001, 65, "mixed"),
                                        (1_500_000, 1_500_000, "a_below"), (1_500_000, 1_500_000, "b_below"),
                                        (2_000_003, 999, "a_below"), (999, 2_000_003, "b_below"),
                                        (70, 70, "a_below"), (70, 70, "b_below")])
def test_corank_far_from_proportional_estimate(gpu, m, n, layout):
    """The warp range search opens with probes around e = k m / (m + n),
    computed in single precision; it stays exact where the co-rank lies far
    from e (one input wholly before the other) and at extreme size ratios,
    through om_corank_i32 and through the merge's own range searches."""
    rng = np.random.default_rng(m * 31 + n + len(layout))
    if layout == "mixed":
        A = sorted_rand(rng, m, -2**31, 2**31)
        B = sorted_rand(rng, n, -2**31, 2**31)
    else:
        low = (-2**31, -1)
        high = (0, 2**31 - 1)
        A = sorted_rand(rng, m, *(low if layout == "a_below" else high))
        B = sorted_rand(rng, n, *(high if layout == "a_below" else low))
    dA, dB = dev_i32(A), dev_i32(B)
    total = m + n
    ks = np.unique(np.concatenate([[0, 1, 64, 65, min(m, n), max(m, n), total // 2, total - 1, total],
                                   rng.integers(0, total + 1, 40)]))
    for k in ks:
        assert gpu.corank_i32(int(k), dA, dB) == oracle.corank_pages(int(k), A, B), int(k)
    check(gpu, A, B)


def test_merge_on_side_stream(gpu):
    rng = np.random.default_rng(12)
    A, B = sorted_rand(rng, 100000, 0, 1000), sorted_rand(rng, 90000, 0, 1000)
    s = torch.cuda.Stream()
    dA, dB = dev_i32(A), dev_i32(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = gpu.merge_i32(dA, dB)
    s.synchronize()
    assert np.array_equal(host(C), oracle.merge_i32(A, B))


def test_device_error_word_clear(gpu):
    assert gpu.device_error() == 0


def _bursty(rng, nblocks, ties):
    """Labels of a merged sequence: balanced stretches (A and B interleaved)
    broken by long one-sided runs, so consecutive sub-tiles of one range use
    each side very unevenly; values nondecreasing (with ties if asked)."""
    labels = []
    for q in range(nblocks):
        kind = q % 7
        if kind == 3:
            labels += [0] * int(rng.integers(3000, 9000))      # A only
        elif kind == 5:
            labels += [1] * int(rng.integers(3000, 9000))      # B only
        else:
            labels += list(rng.integers(0, 2, int(rng.integers(2000, 6000))))
    labels = np.array(labels)
    vals = np.arange(labels.size, dtype=np.int64)
    if ties:
        vals //= 3
    vals = (vals - labels.size // 2).astype(np.int32)
    return vals[labels == 0], vals[labels == 1]


@pytest.mark.parametrize("per_range", [8, 40])
@pytest.mark.parametrize("ties", [False, True])
def test_long_ranges_uneven_consumption(gpu, monkeypatch, per_range, ties):
    """Many sub-tiles per output range with abrupt changes in how much each
    sub-tile takes from A and B: exercises windows published before all of
    their data was requested, and sub-tiles merged again with whole windows."""
    monkeypatch.setenv("OM_SUBTILES_PER_RANGE", str(per_range))
    rng = np.random.default_rng(per_range + 7 * ties)
    A, B = _bursty(rng, 400, ties)
    check(gpu, A, B)
    check(gpu, B, A)


@pytest.mark.parametrize("m,n", [(100003, 99991), (5000, 300007), (1, 50000)])
def test_unsorted_input_terminates_in_bounds(gpu, m, n):
    """Sortedness is a precondition the library does not check.  On unsorted
    input the output is unspecified, but every kernel must still end (its
    searches and waits are bounded) and write nothing outside C; the device
    error word may report a dropped range, never a timed-out wait."""
    rng = np.random.default_rng(m + n)
    A = rng.integers(-1000, 1000, m).astype(np.int32)
    B = rng.integers(-1000, 1000, n).astype(np.int32)
    total = m + n
    buf, C = guarded_empty(total)
    gpu.merge_i32(dev_i32(A), dev_i32(B), C)
    torch.cuda.synchronize()
    assert gpu.device_error() in (0, 2), "a kernel wait timed out on unsorted input"
    assert guards_intact(buf, total), "merge wrote outside C"


def test_one_pass_path_taken_and_matches_oracle(gpu, monkeypatch):
    """A merge that fits in one wave takes the one-pass kernel (traced as its
    own kind) and a larger one the tile-merge kernel; both give the oracle's
    result, at tile boundaries of the one-pass shape (3456 outputs a CTA for
    int32) and around them."""
    monkeypatch.delenv("OM_ONE_PASS_MAX", raising=False)
    rng = np.random.default_rng(21)
    for total in [1, 3455, 3456, 3457, 2 * 3456, 3456 * 40 + 17, 1 << 20]:
        m = total // 3
        A = np.sort(rng.integers(-1000, 1000, m)).astype(np.int32)
        B = np.sort(rng.integers(-1000, 1000, total - m)).astype(np.int32)
        gpu.om_trace_reset()
        gpu.om_trace_enable(True)
        C = gpu.merge_i32(dev_i32(A), dev_i32(B))
        torch.cuda.synchronize()
        gpu.om_trace_enable(False)
        one_pass, _ = gpu.om_trace_read(gpu.KIND_ONE_PASS)
        tile, _ = gpu.om_trace_read(gpu.KIND_TILE_MERGE)
        assert (one_pass, tile) == (1, 0), (total, one_pass, tile)
        assert np.array_equal(host(C), oracle.merge_i32(A, B)), total
    # forced off: the same merge through the tile-merge kernel
    monkeypatch.setenv("OM_ONE_PASS_MAX", "0")
    gpu.om_trace_reset()
    gpu.om_trace_enable(True)
    C = gpu.merge_i32(dev_i32(A), dev_i32(B))
    torch.cuda.synchronize()
    gpu.om_trace_enable(False)
    assert gpu.om_trace_read(gpu.KIND_ONE_PASS)[0] == 0 and gpu.om_trace_read(gpu.KIND_TILE_MERGE)[0] == 1
    assert np.array_equal(host(C), oracle.merge_i32(A, B))


@pytest.mark.parametrize("total", [1919, 1920, 1921, 2 * 1920, 1920 * 7 + 3])
def test_one_pass_pairs_and_wide_keys_at_tile_edges(gpu, monkeypatch, total):
    """Key+value merges and 8-byte keys take the one-pass kernel with 1920
    outputs a CTA: outputs around that tile edge match the oracle (values
    travel with their keys; float64 descending with -0.0 / +0.0 ties)."""
    monkeypatch.delenv("OM_ONE_PASS_MAX", raising=False)
    rng = np.random.default_rng(total)
    m = total // 2 + 7
    n = total - m
    ka = np.sort(rng.integers(0, 9, m)).astype(np.uint32)
    kb = np.sort(rng.integers(0, 9, n)).astype(np.uint32)
    va = np.arange(m, dtype=np.uint32)
    vb = (np.arange(n) | (1 << 31)).astype(np.uint32)
    d = lambda x: torch.from_numpy(x.view(np.int32)).cuda()
    gpu.om_trace_reset()
    gpu.om_trace_enable(True)
    kc, vc = gpu.merge_pairs_u32(d(ka), d(va), d(kb), d(vb))
    torch.cuda.synchronize()
    gpu.om_trace_enable(False)
    assert gpu.om_trace_read(gpu.KIND_ONE_PASS)[0] == 1
    wk, wv = oracle.merge_pairs_u32(ka, va, kb, vb)
    assert np.array_equal(host(kc).view(np.uint32), wk)
    assert np.array_equal(host(vc).view(np.uint32), wv)
    fa = np.sort(rng.choice(np.array([-2.0, -0.0, 0.0, 1.5]), m))[::-1].copy()
    fb = np.sort(rng.choice(np.array([-2.0, 0.0, -0.0, 3.0]), n))[::-1].copy()
    fc = gpu.merge_keys(torch.from_numpy(fa).cuda(), torch.from_numpy(fb).cuda(), descending=True)
    want = oracle.merge_keys(fa, fb, descending=True)
    assert np.array_equal(host(fc).view(np.uint64), want.view(np.uint64))

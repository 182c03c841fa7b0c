"""The five workloads at their full sizes, through the same C-ABI calls and
launch configuration the benchmark times.

Merges are compared with the CPU oracle element by element over the whole
output, plus sampled single outputs through the oracle's co-rank lookup.  The
2^26-key sort is compared with the oracle's merge sort over the whole output
(keys and values), after checks of the properties that fix the stable sort
uniquely: keys nondecreasing, values a permutation of 0..n-1, keys[p] equal
to the input key at position vals[p], and ascending values inside every run
of equal keys.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import host

pytestmark = pytest.mark.gpu


def _sampled_lookup(A, B, C, count=400, seed=0):
    rng = np.random.default_rng(seed)
    total = A.size + B.size
    ks = np.concatenate([[0, total - 1], rng.integers(0, total, count)])
    for k in ks:
        v, _ = oracle.merge_at_i32(int(k), A, B)
        assert C[k] == v, f"C[{k}] = {C[k]}, oracle lookup gives {v}"


@pytest.mark.parametrize("workload", ["evens_odds", "skewed", "uniform"])
def test_merge_i32_full(gpu, workload):
    d = synth.make_device(workload, "cuda")
    A, B = d["A"], d["B"]
    C = gpu.merge_i32(A, B)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    hA, hB, hC = host(A), host(B), host(C)
    del C, d, A, B
    torch.cuda.empty_cache()
    _sampled_lookup(hA, hB, hC)
    want = oracle.merge_i32(hA, hB)
    assert np.array_equal(hC, want), f"first mismatch at {int(np.flatnonzero(hC != want)[0])}"


def test_merge_pairs_full(gpu):
    d = synth.make_device("pairs_ties", "cuda")
    kc, vc = gpu.merge_pairs_u32(d["keysA"], d["valsA"], d["keysB"], d["valsB"])
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    u = lambda t: host(t).view(np.uint32)
    wk, wv = oracle.merge_pairs_u32(u(d["keysA"]), u(d["valsA"]), u(d["keysB"]), u(d["valsB"]))
    assert np.array_equal(u(kc), wk)
    assert np.array_equal(u(vc), wv)


def test_merge_sort_full(gpu):
    d = synth.make_device("sort", "cuda")
    keys0 = host(d["keys"]).view(np.uint32).copy()
    gpu.merge_sort_u32(d["keys"], d["vals"])
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    k = host(d["keys"]).view(np.uint32)
    v = host(d["vals"]).view(np.uint32)
    n = keys0.size
    assert np.all(k[1:] >= k[:-1]), "keys not nondecreasing"
    assert np.array_equal(np.sort(v), np.arange(n, dtype=np.uint32)), "values not a permutation"
    assert np.array_equal(keys0[v], k), "a value does not travel with its key"
    same = k[1:] == k[:-1]
    assert np.all(v[1:][same] > v[:-1][same]), "equal keys out of input order (unstable)"
    # and the oracle's merge sort of the whole 2^26-key input, keys and values
    wk, wv = oracle.merge_sort_pairs_u32(keys0, np.arange(n, dtype=np.uint32))
    assert np.array_equal(k, wk), f"keys: first mismatch at {int(np.flatnonzero(k != wk)[0])}"
    assert np.array_equal(v, wv), f"values: first mismatch at {int(np.flatnonzero(v != wv)[0])}"


@pytest.mark.parametrize("workload", ["f64", "i64_desc"])
def test_merge_keys_full(gpu, workload):
    """2^28 outputs of 8-byte keys (the benchmark's typed merges), compared
    with the oracle over the whole output, bit for bit."""
    d = synth.make_device(workload, "cuda")
    desc = synth.TYPED[workload][1]
    C = gpu.merge_keys(d["A"], d["B"], descending=desc)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    hA, hB, hC = host(d["A"]), host(d["B"]), host(C)
    del C, d
    torch.cuda.empty_cache()
    want = oracle.merge_keys(hA, hB, descending=desc)
    assert np.array_equal(hC.view(np.uint64), want.view(np.uint64)), (
        f"first mismatch at {int(np.flatnonzero(hC.view(np.uint64) != want.view(np.uint64))[0])}")


@pytest.mark.parametrize("workload", ["sort_f32_desc", "sort_f64"])
def test_merge_sort_keys_full(gpu, workload):
    """2^26 float keys through the benchmark's typed sorts: ordered, a
    permutation of the input, and (with the index payload) stable."""
    d = synth.make_device(workload, "cuda")
    desc = synth.TYPED[workload][1]
    keys0 = host(d["keys"]).copy()
    vals = d.get("vals")
    gpu.merge_sort_keys(d["keys"], vals, descending=desc)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    k = host(d["keys"])
    order = k[:-1] >= k[1:] if desc else k[:-1] <= k[1:]
    assert np.all(order), "keys out of order"
    if vals is None:
        assert np.array_equal(np.sort(k), np.sort(keys0)), "keys not a permutation of the input"
    else:
        v = host(vals).view(np.uint32)
        assert np.array_equal(np.sort(v), np.arange(k.size, dtype=np.uint32)), "values not a permutation"
        assert np.array_equal(keys0[v].view(np.uint32), k.view(np.uint32)), "a value does not travel with its key"
        same = k[1:] == k[:-1]
        assert np.all(v[1:][same] > v[:-1][same]), "equal keys out of input order (unstable)"

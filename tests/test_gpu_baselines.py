"""GPU parity of the two unstaged comparison merges (om_merge_i32_one_thread,
om_merge_i32_slices at every slice size of the sweep) against the CPU
oracle, bit-exact, with guard bands: the comparison rows are only meaningful
if every row computes the same merge."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_i32, guarded_empty, guards_intact, host

pytestmark = pytest.mark.gpu

SLICES = [1, 4, 16, 64, 256]


def sorted_rand(rng, size, lo, hi):
    return np.sort(rng.integers(lo, hi, size, dtype=np.int64)).astype(np.int32)


def run(om, fn, A_np, B_np, **kw):
    total = A_np.size + B_np.size
    buf, C = guarded_empty(total)
    fn(dev_i32(A_np), dev_i32(B_np), C, **kw)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    assert guards_intact(buf, total), "wrote outside C"
    return host(C)


@pytest.mark.parametrize("per_thread", SLICES + [3, 1000])
@pytest.mark.parametrize("m,n", [(0, 0), (0, 9), (9, 0), (1, 1), (255, 2), (12345, 54321), (300007, 299993)])
def test_slices(gpu, per_thread, m, n):
    rng = np.random.default_rng(m + 17 * n + per_thread)
    for span in (4, 1 << 31):
        A, B = sorted_rand(rng, m, -span, span), sorted_rand(rng, n, -span, span)
        got = run(gpu, gpu.merge_i32_slices, A, B, per_thread=per_thread)
        assert np.array_equal(got, oracle.merge_i32(A, B))


@pytest.mark.parametrize("m,n", [(0, 5), (5, 0), (1, 1), (1000, 999), (65537, 30001)])
def test_one_thread(gpu, m, n):
    rng = np.random.default_rng(m * 3 + n)
    A, B = sorted_rand(rng, m, -50, 50), sorted_rand(rng, n, -50, 50)
    got = run(gpu, gpu.merge_i32_one_thread, A, B)
    assert np.array_equal(got, oracle.merge_i32(A, B))


def test_evens_odds_full_size_every_row(gpu):
    """The comparison workload itself: every row gives the oracle's merge."""
    d = synth.make_host("evens_odds")
    want = oracle.merge_i32(d["A"], d["B"])
    assert np.array_equal(run(gpu, gpu.merge_i32_one_thread, d["A"], d["B"]), want)
    for s in SLICES:
        assert np.array_equal(run(gpu, gpu.merge_i32_slices, d["A"], d["B"], per_thread=s), want)

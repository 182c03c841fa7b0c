"""The grid-level partition kernel (om_partition_i32) against the oracle.

Every splitter the kernel writes is compared with the oracle's co-rank of
the same output rank: the pages' bisection (O2) at every boundary, and the
co-rank by counting merge steps (O3) at a sample of them.  Inputs cover
distinct keys, heavy ties across the two sides, wholly one-sided inputs in
both directions, a narrow B inside a long A, empty sides, and tile lengths
from 1 output to more than the whole merge, so boundaries fall on ties, at
the ends and past the end.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_i32, host

pytestmark = pytest.mark.gpu


def _case(name, seed):
    rng = np.random.default_rng(seed)
    if name == "distinct":
        A = np.arange(0, 2 * 5003, 2, dtype=np.int32)
        B = np.arange(1, 2 * 4001, 2, dtype=np.int32)
    elif name == "heavy_ties":
        A = np.sort(rng.integers(0, 4, 7000)).astype(np.int32)
        B = np.sort(rng.integers(0, 4, 6500)).astype(np.int32)
    elif name == "all_A_first":
        A = np.sort(rng.integers(-1000, 0, 6000)).astype(np.int32)
        B = np.sort(rng.integers(0, 1000, 5000)).astype(np.int32)
    elif name == "all_B_first":
        A = np.sort(rng.integers(1, 1000, 5000)).astype(np.int32)
        B = np.sort(rng.integers(-1000, 1, 6000)).astype(np.int32)
    elif name == "narrow_B":
        A = np.sort(rng.integers(-2**31, 2**31, 20000)).astype(np.int32)
        B = np.sort(rng.integers(-2**20, 2**20 + 1, 300)).astype(np.int32)
    elif name == "extremes":
        A = np.sort(rng.choice(np.array([-2**31, -1, 0, 2**31 - 1], dtype=np.int64), 3000)).astype(np.int32)
        B = np.sort(rng.choice(np.array([-2**31, 0, 2**31 - 1], dtype=np.int64), 2000)).astype(np.int32)
    elif name == "empty_B":
        A = np.sort(rng.integers(-50, 50, 3001)).astype(np.int32)
        B = np.zeros(0, dtype=np.int32)
    elif name == "empty_A":
        A = np.zeros(0, dtype=np.int32)
        B = np.sort(rng.integers(-50, 50, 2999)).astype(np.int32)
    else:
        raise ValueError(name)
    return A, B


CASES = ["distinct", "heavy_ties", "all_A_first", "all_B_first", "narrow_B", "extremes", "empty_B", "empty_A"]


@pytest.mark.parametrize("tile", [1, 7, 256, 2944, 3 * 2944, 1 << 20])
@pytest.mark.parametrize("case", CASES)
def test_partition_matches_oracle(gpu, case, tile):
    A, B = _case(case, seed=CASES.index(case))
    total = A.size + B.size
    count = (total + tile - 1) // tile + 2  # one boundary past the end as well: clamped to m + n
    if tile == 1:
        count = min(count, 2500)  # a prefix of the boundaries keeps the oracle loop short
    split = gpu.partition_i32(dev_i32(A), dev_i32(B), tile, count)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    got = host(split)
    rng = np.random.default_rng(tile)
    sample = set(rng.integers(0, count, 12).tolist()) | {0, count - 1}
    for t in range(count):
        k = min(t * tile, total)
        want = oracle.corank_pages(k, A, B)
        assert got[t] == want, f"{case}: split[{t}] (k={k}) = {got[t]}, oracle co-rank {want}"
        if t in sample:
            assert oracle.corank_count(k, A, B) == want


def test_partition_large_merge_samples(gpu):
    """2^25 outputs of uniform keys: every 2944th rank through the kernel;
    a sample checked with the pages' bisection."""
    rng = np.random.default_rng(11)
    A = np.sort(rng.integers(-2**31, 2**31, 1 << 24)).astype(np.int32)
    B = np.sort(rng.integers(-2**31, 2**31, 1 << 24)).astype(np.int32)
    tile = 2944
    split = host(gpu.partition_i32(dev_i32(A), dev_i32(B), tile))
    total = A.size + B.size
    assert split.size == (total + tile - 1) // tile + 1
    for t in np.concatenate([[0, 1, split.size - 2, split.size - 1], rng.integers(0, split.size, 300)]):
        k = min(int(t) * tile, total)
        assert split[t] == oracle.corank_pages(k, A, B), f"split[{t}]"

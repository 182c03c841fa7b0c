"""GPU parity of om_merge_pairs_u32 and om_merge_sort_u32 against the CPU
oracle, bit-exact on keys and values (values make stability visible)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_i32, guarded_empty, guards_intact, host, shifted

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("merge_path")]


def run_pairs(om, ka, va, kb, vb, offs=(0, 0, 0)):
    total = ka.size + kb.size
    dka, dva = shifted(dev_i32(ka), offs[0]), shifted(dev_i32(va), offs[0])
    dkb, dvb = shifted(dev_i32(kb), offs[1]), shifted(dev_i32(vb), offs[1])
    bk, kc = guarded_empty(total, offs[2])
    bv, vc = guarded_empty(total, offs[2])
    om.merge_pairs_u32(dka, dva, dkb, dvb, kc, vc)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    assert guards_intact(bk, total, offs[2]) and guards_intact(bv, total, offs[2])
    return host(kc).view(np.uint32), host(vc).view(np.uint32)


def check_pairs(om, ka, va, kb, vb, offs=(0, 0, 0)):
    gk, gv = run_pairs(om, ka, va, kb, vb, offs)
    wk, wv = oracle.merge_pairs_u32(ka, va, kb, vb)
    assert np.array_equal(gk, wk), f"keys differ first at {int(np.flatnonzero(gk != wk)[0])}"
    assert np.array_equal(gv, wv), f"values differ first at {int(np.flatnonzero(gv != wv)[0])}"


def tagged(m, n):
    return np.arange(m, dtype=np.uint32), np.arange(n, dtype=np.uint32) | np.uint32(1 << 31)


def test_pairs_tie_case(gpu):
    ka = np.array([1, 1, 2, 3], np.uint32)
    kb = np.array([1, 2, 2, 4], np.uint32)
    va, vb = tagged(4, 4)
    check_pairs(gpu, ka, va, kb, vb)


@pytest.mark.parametrize("m,n,hi", [(0, 10, 4), (10, 0, 4), (1, 1, 2), (1920, 1920, 3), (30001, 29999, 16),
                                    (100000, 3, 2), (3, 100000, 2), (77777, 66666, 1 << 32)])
def test_pairs_shapes(gpu, m, n, hi):
    rng = np.random.default_rng(m + 3 * n)
    ka = np.sort(rng.integers(0, hi, m, dtype=np.uint64)).astype(np.uint32)
    kb = np.sort(rng.integers(0, hi, n, dtype=np.uint64)).astype(np.uint32)
    va, vb = tagged(m, n)
    check_pairs(gpu, ka, va, kb, vb)


def test_pairs_unsigned_order(gpu):
    """Keys with the top bit set sort after small keys (unsigned compare)."""
    ka = np.array([1, 5, 0x80000000, 0xFFFFFFFF], np.uint32)
    kb = np.array([0, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF], np.uint32)
    va, vb = tagged(4, 4)
    check_pairs(gpu, ka, va, kb, vb)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 2, 3), (3, 1, 2)])
def test_pairs_misaligned(gpu, offs):
    rng = np.random.default_rng(99)
    ka = np.sort(rng.integers(0, 16, 20011)).astype(np.uint32)
    kb = np.sort(rng.integers(0, 16, 19997)).astype(np.uint32)
    va, vb = tagged(ka.size, kb.size)
    check_pairs(gpu, ka, va, kb, vb, offs)


@pytest.mark.parametrize("offs", [(0, 0, 0), (1, 0, 0), (0, 2, 3), (3, 1, 2), (2, 2, 1)])
def test_pairs_one_sided_ranges(gpu, offs):
    """Key+value output ranges that take every element from one side, at
    every 16-byte phase of A, B and C."""
    rng = np.random.default_rng(sum(offs) + 17)
    lo = np.sort(rng.integers(0, 1 << 20, 250007)).astype(np.uint32)
    hi = np.sort(rng.integers(1 << 20, 1 << 21, 180001)).astype(np.uint32)
    for ka, kb in ((lo, hi), (hi, lo)):
        va, vb = tagged(ka.size, kb.size)
        check_pairs(gpu, ka, va, kb, vb, offs)
    blocks = (np.arange(60 * 7000).reshape(60, 7000) // 5).astype(np.uint32)
    ka, kb = np.sort(blocks[0::2].ravel()), np.sort(blocks[1::2].ravel())
    va, vb = tagged(ka.size, kb.size)
    check_pairs(gpu, ka, va, kb, vb, offs)


def test_pairs_ties_workload_scaled(gpu):
    d = synth.make_host("pairs_ties", scale_log2=4)
    check_pairs(gpu, d["keysA"], d["valsA"], d["keysB"], d["valsB"])


# ------------------------------------------------------------------- sort --

def run_sort(om, keys, vals):
    dk = dev_i32(keys)
    dv = dev_i32(vals) if vals is not None else None
    om.merge_sort_u32(dk, dv)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    return host(dk).view(np.uint32), (host(dv).view(np.uint32) if dv is not None else None)


def check_sort(om, keys, with_vals=True):
    vals = np.arange(keys.size, dtype=np.uint32) if with_vals else None
    gk, gv = run_sort(om, keys, vals)
    wk, wv = oracle.merge_sort_pairs_u32(keys, np.arange(keys.size, dtype=np.uint32))
    assert np.array_equal(gk, wk), f"keys differ first at {int(np.flatnonzero(gk != wk)[0])}"
    if with_vals:
        assert np.array_equal(gv, wv), f"values differ first at {int(np.flatnonzero(gv != wv)[0])}"


@pytest.mark.parametrize("n", [0, 1, 2, 3, 16, 17, 18, 34, 35, 1023, 1024, 1025, 2048, 4095, 4097, 4351, 4352, 4353,
                               8192, 8703, 8704, 8705, 10000, 13057, 65536,
                               100003, 1 << 18, (1 << 18) + 12345])
def test_sort_sizes(gpu, n):
    rng = np.random.default_rng(n)
    check_sort(gpu, rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32))


@pytest.mark.parametrize("hi", [1, 2, 16, 1000])
def test_sort_heavy_ties(gpu, hi):
    rng = np.random.default_rng(hi)
    check_sort(gpu, rng.integers(0, hi, 300007, dtype=np.uint64).astype(np.uint32))


def test_sort_presorted_and_reversed(gpu):
    check_sort(gpu, np.arange(200000, dtype=np.uint32))
    check_sort(gpu, np.arange(200000, dtype=np.uint32)[::-1].copy())


def test_sort_keys_only(gpu):
    rng = np.random.default_rng(5)
    for n in [5, 5000, 123457]:
        check_sort(gpu, rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32), with_vals=False)


def test_sort_workload_scaled(gpu):
    d = synth.make_host("sort", scale_log2=6)
    check_sort(gpu, d["keys"])


@pytest.mark.parametrize("per_range", [1, 3])
@pytest.mark.parametrize("n", [200001, (1 << 18) + 4097])
def test_sort_pairs_split_into_ranges(gpu, monkeypatch, per_range, n):
    """Late passes whose pairs of runs split into several output ranges (as
    at full size), with a ragged last pair: short ranges forced."""
    monkeypatch.setenv("OM_SUBTILES_PER_RANGE", str(per_range))
    rng = np.random.default_rng(per_range * 7 + n)
    check_sort(gpu, rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32))
    check_sort(gpu, rng.integers(0, 50, n, dtype=np.uint64).astype(np.uint32))


@pytest.mark.parametrize("waves", [2, 5])
def test_merge_and_sort_forced_waves(gpu, monkeypatch, waves):
    """The range rule held to a fixed wave count: several waves of shorter
    ranges give the same merge and sort."""
    monkeypatch.setenv("OM_WAVES", str(waves))
    rng = np.random.default_rng(waves)
    ka = np.sort(rng.integers(0, 1000, 300007, dtype=np.uint64).astype(np.uint32))
    kb = np.sort(rng.integers(0, 1000, 200003, dtype=np.uint64).astype(np.uint32))
    va, vb = tagged(ka.size, kb.size)
    check_pairs(gpu, ka, va, kb, vb)
    check_sort(gpu, rng.integers(0, 1 << 32, 300007, dtype=np.uint64).astype(np.uint32))


@pytest.mark.parametrize("per_range", [8, 40])
def test_pairs_long_ranges_uneven_consumption(gpu, monkeypatch, per_range):
    """Key+value merge with many sub-tiles per range and bursty consumption."""
    monkeypatch.setenv("OM_SUBTILES_PER_RANGE", str(per_range))
    rng = np.random.default_rng(per_range)
    labels = []
    for q in range(300):
        if q % 5 == 2:
            labels += [q % 2] * int(rng.integers(2000, 6000))
        else:
            labels += list(rng.integers(0, 2, int(rng.integers(1000, 4000))))
    labels = np.array(labels)
    keys = (np.arange(labels.size) // 4).astype(np.uint32)
    ka, kb = keys[labels == 0], keys[labels == 1]
    va, vb = tagged(ka.size, kb.size)
    check_pairs(gpu, ka, va, kb, vb)


def test_scratch_pool_reuse_and_release(gpu):
    """Sorts reuse the library's scratch pool across synchronising calls;
    om_release_scratch hands the cached scratch back (device free memory
    grows by at least the sort's second buffer) and later sorts still work."""
    rng = np.random.default_rng(77)
    n = 1 << 22
    keys = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    check_sort(gpu, keys)
    check_sort(gpu, keys)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    gpu.release_scratch()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after - free_before >= 2 * n * 4 - (2 << 20)
    check_sort(gpu, keys)

"""The seeded input generator: the C draw equals the numpy reference draw, the
SplitMix64 stream matches its published first outputs, and every workload has
the shape, ordering and value range it is defined with."""
import numpy as np

import synth


def test_splitmix64_known_values():
    # First outputs of splitmix64 seeded with 0 (Vigna's splitmix64.c).
    assert list(synth.splitmix64(0, 3)) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # counter-based: a window of the stream equals the same draws from the start
    assert list(synth.splitmix64(0, 2, start=1)) == list(synth.splitmix64(0, 3)[1:])


def test_c_generator_matches_numpy():
    for seed in [0, 1, 1025, (1 << 63) + 5]:
        assert np.array_equal(synth.uniform_u32(seed, 5000), synth.np_top32(seed, 5000))
        for bound in [1, 16, (1 << 21) + 1, 1 << 32]:
            assert np.array_equal(synth.uniform_below(seed, 3000, bound), synth.np_below(seed, 3000, bound))


def test_workload_shapes():
    d = synth.make_host("evens_odds")
    assert d["A"].size == (1 << 21) + 611 and d["B"].size == 1 << 21
    assert (d["A"].size + d["B"].size) % 2 == 1
    d = synth.make_host("skewed", 12)
    assert d["B"].min() >= -(1 << 20) and d["B"].max() <= (1 << 20)
    assert np.all(np.diff(d["A"].astype(np.int64)) >= 0)
    d = synth.make_host("pairs_ties", 12)
    assert d["keysA"].max() < 16 and np.all(np.diff(d["keysB"].astype(np.int64)) >= 0)
    assert np.all(d["valsB"] >> np.uint32(31) == 1) and np.all(d["valsA"] >> np.uint32(31) == 0)
    d = synth.make_host("sort", 14)
    assert d["keys"].size == 1 << 12 and np.array_equal(d["vals"], np.arange(1 << 12, dtype=np.uint32))
    u = synth.make_host("uniform", 16)
    assert u["A"].size == 1 << 12 and not np.array_equal(u["A"], u["B"])

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


def test_typed_workloads_host_equals_device_on_cpu():
    """The typed workloads: host arrays sorted in their order, and the device
    path (here torch on the CPU) gives the same bits."""
    import torch

    for wl, (kt, desc) in synth.TYPED.items():
        h = synth.make_host(wl, 12)
        d = synth.make_device(wl, torch.device("cpu"), 12)
        for key in h:
            hv = h[key]
            dv = d[key].numpy()
            assert hv.dtype.itemsize == dv.dtype.itemsize
            assert np.array_equal(hv.view(np.uint8), np.ascontiguousarray(dv).view(np.uint8)), (wl, key)
        if "A" in h:
            for arr in (h["A"], h["B"]):
                diffs = np.diff(arr.astype(np.float64)) if arr.dtype.kind == "f" else np.diff(arr.astype(object))
                assert all(x <= 0 for x in diffs) if desc else all(x >= 0 for x in diffs)
        assert synth.sizes(wl, 12)[0] == h["A" if "A" in h else "keys"].size

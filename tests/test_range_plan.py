"""Host-side launch planning: how many sub-tiles each CTA output range gets
(om_subtiles_per_range).  Pure host code, so these run without a GPU.

The rule: a launch over `segs` merges of at most `seg_len` outputs, cut into
ranges of q sub-tiles that never cross a merge, runs `resident` CTAs at a
time; its time is modelled as waves * (fixed cost per range + longest range)
and q minimises that over one to eight waves."""
import pytest

import ordered_merge_gb300 as om

SLOTS = 152 * 5  # SMs x resident tile-merge CTAs per SM
OVERHEAD_BYTES = 24576  # fixed cost of one range, as bytes moved at full rate


@pytest.fixture(autouse=True)
def no_overrides(monkeypatch):
    monkeypatch.delenv("OM_WAVES", raising=False)
    monkeypatch.delenv("OM_SUBTILES_PER_RANGE", raising=False)


def ceil_div(a, b):
    return -(-a // b)


def ranges(segs, seg_len, T, q):
    return segs * ceil_div(seg_len, q * T)


def modelled_cost(segs, seg_len, T, bpo, slots, q):
    return ceil_div(ranges(segs, seg_len, T, q), slots) * (OVERHEAD_BYTES // bpo + min(q * T, seg_len))


def test_bad_arguments_return_zero():
    assert om.om_subtiles_per_range(0, 100, 10, 8, SLOTS) == 0
    assert om.om_subtiles_per_range(1, 0, 10, 8, SLOTS) == 0
    assert om.om_subtiles_per_range(1, 100, 0, 8, SLOTS) == 0
    assert om.om_subtiles_per_range(1, 100, 10, 0, SLOTS) == 0
    assert om.om_subtiles_per_range(1, 100, 10, 8, -1) == 0


@pytest.mark.parametrize("total", [1, 2944, 2945, 4_194_915, 33_554_432, 268_436_480, 1 << 29, (1 << 29) + 7])
def test_one_merge_is_one_full_wave(total):
    """A single merge: equal ranges, as short as one wave allows."""
    T = 2944
    q = om.om_subtiles_per_range(1, total, T, 8, SLOTS)
    assert q == max(1, ceil_div(ceil_div(total, T), SLOTS))
    assert ranges(1, total, T, q) <= SLOTS


def test_sort_passes_of_2e26_pairs():
    """Late passes of a 2^26-key sort with values (4096-key runs, 1408-output
    sub-tiles, 16 bytes per output).  Pairs that do not divide evenly into the
    760 resident CTAs get shorter ranges over two to four waves; the last
    passes keep one full wave (no pass ends on a few leftover CTAs)."""
    n, T, bpo = 1 << 26, 1408, 16
    got = []
    r = 4096
    while r < n:
        npairs = ceil_div(n, 2 * r)
        got.append(om.om_subtiles_per_range(npairs, min(2 * r, n), T, bpo, SLOTS))
        r *= 2
    assert got == [6, 12, 24, 24, 24, 17, 22, 33, 65, 64, 63, 63, 63, 63]
    r = 4096
    for q in got:
        npairs = ceil_div(n, 2 * r)
        nr = ranges(npairs, 2 * r, T, q)
        if q * T < 2 * r:  # pairs split into several ranges: the last wave is at least half full
            assert nr <= SLOTS or nr % SLOTS == 0 or nr % SLOTS > SLOTS // 2, (r, q, nr)
        r *= 2


@pytest.mark.parametrize(
    "segs,seg_len,T,bpo",
    [(1, 1 << 29, 2944, 8), (512, 131072, 1408, 16), (100, 1_000_003, 1408, 16), (7, 12345, 2944, 8),
     (3000, 8192, 1408, 16), (256, 262144, 2944, 8), (33, 5_000_000, 1408, 16)],
)
def test_choice_minimises_the_model(segs, seg_len, T, bpo):
    """The choice is the cheapest of every range length within eight waves."""
    q = om.om_subtiles_per_range(segs, seg_len, T, bpo, SLOTS)
    qmax = ceil_div(seg_len, T)
    assert 1 <= q <= qmax
    feasible = [x for x in range(1, qmax + 1) if ceil_div(ranges(segs, seg_len, T, x), SLOTS) <= 8] or [qmax]
    best = min(modelled_cost(segs, seg_len, T, bpo, SLOTS, x) for x in feasible)
    assert modelled_cost(segs, seg_len, T, bpo, SLOTS, q) == best


def test_environment_overrides(monkeypatch):
    monkeypatch.setenv("OM_SUBTILES_PER_RANGE", "7")
    assert om.om_subtiles_per_range(1, 1 << 29, 2944, 8, SLOTS) == 7
    monkeypatch.delenv("OM_SUBTILES_PER_RANGE")
    monkeypatch.setenv("OM_WAVES", "2")
    q = om.om_subtiles_per_range(1, 1 << 29, 2944, 8, SLOTS)
    assert q == ceil_div(ceil_div(1 << 29, 2944), 2 * SLOTS)

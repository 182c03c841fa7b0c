"""GPU parity of om_merge_keys and om_merge_sort_keys (six key types,
ascending and descending) against the CPU oracle: element by element, bit
for bit, with guard bands around every merge output; values (index tags)
make the sort's stability visible.

Sizes span one sub-tile, many sub-tiles and output ranges, and ragged
tails; edge cases cover empty and one-element sides, heavy ties, -0.0 and
+0.0 (equal keys with different bits, so the tie rule is visible), the
types' extreme values, infinities and subnormals, and pointers that are not
16-byte aligned.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("merge_path")]

TYPES = ["i32", "u32", "f32", "i64", "u64", "f64"]
NP = {"i32": np.int32, "u32": np.uint32, "f32": np.float32, "i64": np.int64, "u64": np.uint64, "f64": np.float64}
GUARD = 36


def _carrier(name):
    """The signed integer numpy/torch types that carry a key type's bits."""
    return (np.int32, torch.int32) if np.dtype(NP[name]).itemsize == 4 else (np.int64, torch.int64)


def to_dev(x, name, offset=0):
    """Device copy of x whose first element sits `offset` elements past a
    16-byte boundary."""
    npc, tc = _carrier(name)
    h = torch.from_numpy(np.ascontiguousarray(x, dtype=NP[name]).view(npc))
    buf = torch.empty(h.numel() + 4, dtype=tc, device="cuda")
    view = buf[offset: offset + h.numel()]
    view.copy_(h)
    return view


def run(om, name, A, B, desc=False, offs=(0, 0, 0)):
    npc, tc = _carrier(name)
    total = A.size + B.size
    dA, dB = to_dev(A, name, offs[0]), to_dev(B, name, offs[1])
    sentinel = -0x5A5A5A5B
    buf = torch.full((total + 2 * GUARD + 4,), sentinel, dtype=tc, device="cuda")
    C = buf[GUARD + offs[2]: GUARD + offs[2] + total]
    om.merge_keys(dA, dB, C, key_type=name, descending=desc)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    h = buf.cpu().numpy()
    assert np.all(h[: GUARD + offs[2]] == sentinel) and np.all(h[GUARD + offs[2] + total:] == sentinel), \
        "merge wrote outside C"
    return C.cpu().numpy().view(NP[name])


def check(om, name, A, B, desc=False, offs=(0, 0, 0)):
    A = np.ascontiguousarray(A, dtype=NP[name])
    B = np.ascontiguousarray(B, dtype=NP[name])
    got = run(om, name, A, B, desc, offs)
    want = oracle.merge_keys(A, B, descending=desc)
    npc, _ = _carrier(name)
    g, w = got.view(npc), want.view(npc)
    if not np.array_equal(g, w):
        bad = int(np.flatnonzero(g != w)[0])
        raise AssertionError(f"{name} desc={desc}: first mismatch at {bad}: got {got[bad]!r}, want {want[bad]!r} "
                             f"(m={A.size}, n={B.size}, offs={offs})")


def sorted_keys(rng, name, size, span, desc):
    """`size` sorted keys of type `name` drawn from about `span` distinct
    values (heavy ties for a small span); floats include signed zeros."""
    dt = NP[name]
    if np.issubdtype(dt, np.floating):
        base = rng.integers(-span, span, size).astype(np.float64) / 4.0
        base[rng.random(size) < 0.05] = 0.0
        x = base.astype(dt)
        x[(x == 0) & (rng.random(size) < 0.5)] = -0.0
    elif np.issubdtype(dt, np.unsignedinteger):
        info = np.iinfo(dt)
        if span >= 1 << 20:
            x = rng.integers(0, info.max, size, dtype=dt, endpoint=True)
        else:
            x = (rng.integers(0, span, size, dtype=np.int64).astype(dt) * dt(info.max // max(span, 1)))
    else:
        info = np.iinfo(dt)
        if span >= 1 << 20:
            x = rng.integers(info.min, info.max, size, dtype=dt, endpoint=True)
        else:
            x = rng.integers(-span, span, size, dtype=np.int64).astype(dt)
    x = np.sort(x, kind="stable")
    return x[::-1].copy() if desc else x


@pytest.mark.parametrize("desc", [False, True], ids=["asc", "desc"])
@pytest.mark.parametrize("name", TYPES)
@pytest.mark.parametrize("m,n", [(0, 0), (0, 7), (7, 0), (1, 1), (1343, 1), (1344, 1344), (1407, 1), (1408, 1408),
                                 (1471, 1), (1472, 1472), (2944, 1), (4037, 2945), (12345, 54321),
                                 (250001, 249999)])
def test_shapes(gpu, name, desc, m, n):
    rng = np.random.default_rng(m * 31 + n + 7 * TYPES.index(name) + desc)
    for span in (8, 1 << 30):
        check(gpu, name, sorted_keys(rng, name, m, span, desc), sorted_keys(rng, name, n, span, desc), desc)


@pytest.mark.parametrize("desc", [False, True], ids=["asc", "desc"])
@pytest.mark.parametrize("name", TYPES)
def test_extremes(gpu, name, desc):
    dt = NP[name]
    if np.issubdtype(dt, np.floating):
        vals = [-np.inf, -np.finfo(dt).max, -1.0, -np.finfo(dt).tiny, -0.0, 0.0, np.finfo(dt).smallest_subnormal,
                1.0, np.finfo(dt).max, np.inf]
    else:
        info = np.iinfo(dt)
        vals = sorted({int(info.min), int(info.min) + 1, -1 if info.min < 0 else 1, 0, 1 << 7,
                       int(info.max) // 2, int(info.max) // 2 + 1, int(info.max) - 1, int(info.max)})
    rng = np.random.default_rng(TYPES.index(name) * 2 + desc)
    src = np.array(vals, dtype=dt)
    for m, n in [(len(vals), len(vals)), (30011, 20011)]:
        A = np.sort(src[rng.integers(0, src.size, m)], kind="stable")
        B = np.sort(src[rng.integers(0, src.size, n)], kind="stable")
        if desc:
            A, B = A[::-1].copy(), B[::-1].copy()
        check(gpu, name, A, B, desc)


@pytest.mark.parametrize("name", ["f32", "f64"])
def test_signed_zero_ties(gpu, name):
    """All keys zero: A holds -0.0 and B +0.0 (then the reverse); the output
    must be all of A's zeros, then all of B's, in either order."""
    dt = NP[name]
    for desc in (False, True):
        for za, zb in ((-0.0, 0.0), (0.0, -0.0)):
            check(gpu, name, np.full(40007, za, dt), np.full(30011, zb, dt), desc)


@pytest.mark.parametrize("name", TYPES)
@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 1, 1), (1, 1, 0), (3, 2, 1)])
def test_misaligned_pointers(gpu, name, offs):
    if np.dtype(NP[name]).itemsize == 8:
        offs = tuple(o & 1 for o in offs)  # one 8-byte element = half a 16-byte group
    rng = np.random.default_rng(sum(offs) + TYPES.index(name))
    for desc in (False, True):
        check(gpu, name, sorted_keys(rng, name, 54321, 500, desc), sorted_keys(rng, name, 43210, 500, desc),
              desc, offs)
        check(gpu, name, sorted_keys(rng, name, 13, 5, desc), sorted_keys(rng, name, 1, 5, desc), desc, offs)


@pytest.mark.parametrize("name,desc", [("i64", False), ("f64", True), ("u32", True), ("f32", False)])
@pytest.mark.parametrize("per_range", [8, 40])
def test_long_ranges_uneven_consumption(gpu, monkeypatch, name, desc, per_range):
    """Many sub-tiles per output range, with stretches where one side supplies
    every output: windows cut to landed data, and sub-tiles merged again with
    whole windows."""
    monkeypatch.setenv("OM_SUBTILES_PER_RANGE", str(per_range))
    rng = np.random.default_rng(per_range + TYPES.index(name))
    labels = []
    for q in range(300):
        if q % 6 == 2:
            labels += [q % 2] * int(rng.integers(2000, 7000))
        else:
            labels += list(rng.integers(0, 2, int(rng.integers(1000, 5000))))
    labels = np.array(labels)
    keys = (np.arange(labels.size, dtype=np.int64) // 3 - labels.size // 6)
    if NP[name] in (np.uint32, np.uint64):
        keys = keys - keys.min()
    keys = keys.astype(NP[name])
    if desc:
        keys = keys[::-1].copy()
        labels = labels[::-1].copy()
    A, B = keys[labels == 0], keys[labels == 1]
    check(gpu, name, A, B, desc)
    check(gpu, name, B, A, desc)


@pytest.mark.parametrize("name", ["i32", "f32"])
def test_i32_ascending_matches_merge_i32(gpu, name):
    """The typed call with i32 ascending keys gives om_merge_i32's output."""
    rng = np.random.default_rng(3)
    A = sorted_keys(rng, "i32", 100003, 1000, False)
    B = sorted_keys(rng, "i32", 99997, 1000, False)
    dA, dB = to_dev(A, "i32"), to_dev(B, "i32")
    c1 = gpu.merge_i32(dA, dB)
    c2 = gpu.merge_keys(dA, dB, key_type="i32")
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("name", ["i64", "f64", "u64"])
def test_wide_keys_large(gpu, name):
    """2^24 outputs of 8-byte keys: many ranges per CTA wave; checked in full."""
    rng = np.random.default_rng(11)
    for desc in (False, True):
        check(gpu, name, sorted_keys(rng, name, (1 << 23) + 3, 1 << 30, desc),
              sorted_keys(rng, name, (1 << 23) - 3, 1 << 30, desc), desc)


# ------------------------------------------------------------------- sort --

def run_sort(om, name, keys, with_vals, desc):
    dk = to_dev(keys, name)
    dv = torch.from_numpy(np.arange(keys.size, dtype=np.int32)).cuda() if with_vals else None
    om.merge_sort_keys(dk, dv, key_type=name, descending=desc)
    torch.cuda.synchronize()
    assert om.device_error() == 0
    return dk.cpu().numpy().view(NP[name]), (dv.cpu().numpy().view(np.uint32) if with_vals else None)


def check_sort(om, name, keys, desc, with_vals=None):
    keys = np.ascontiguousarray(keys, dtype=NP[name])
    if with_vals is None:
        with_vals = np.dtype(NP[name]).itemsize == 4
    gk, gv = run_sort(om, name, keys, with_vals, desc)
    wk, wv = oracle.merge_sort_keys(keys, np.arange(keys.size, dtype=np.uint32), descending=desc)
    npc, _ = _carrier(name)
    if not np.array_equal(gk.view(npc), wk.view(npc)):
        bad = int(np.flatnonzero(gk.view(npc) != wk.view(npc))[0])
        raise AssertionError(f"{name} desc={desc} n={keys.size}: keys differ first at {bad}: "
                             f"got {gk[bad]!r}, want {wk[bad]!r}")
    if with_vals:
        assert np.array_equal(gv, wv), f"values differ first at {int(np.flatnonzero(gv != wv)[0])}"


def unsorted_keys(rng, name, size, span):
    x = sorted_keys(rng, name, size, span, False)
    return x[rng.permutation(size)]


@pytest.mark.parametrize("desc", [False, True], ids=["asc", "desc"])
@pytest.mark.parametrize("name", TYPES)
@pytest.mark.parametrize("n", [0, 1, 2, 17, 18, 4095, 4096, 4351, 4352, 4353, 8705, 10000, 100003,
                               (1 << 18) + 12345])
def test_sort_sizes(gpu, name, desc, n):
    rng = np.random.default_rng(n + 13 * TYPES.index(name) + desc)
    check_sort(gpu, name, unsorted_keys(rng, name, n, 1 << 30), desc)


@pytest.mark.parametrize("desc", [False, True], ids=["asc", "desc"])
@pytest.mark.parametrize("name", TYPES)
def test_sort_heavy_ties_and_extremes(gpu, name, desc):
    rng = np.random.default_rng(5 + TYPES.index(name) + 100 * desc)
    check_sort(gpu, name, unsorted_keys(rng, name, 300007, 4), desc)
    dt = NP[name]
    if np.issubdtype(dt, np.floating):
        vals = np.array([-np.inf, -1.0, -0.0, 0.0, np.finfo(dt).smallest_subnormal, np.inf], dt)
    else:
        info = np.iinfo(dt)
        vals = np.array([info.min, info.min + 1, 0, 1, info.max - 1, info.max], dt)
    check_sort(gpu, name, vals[rng.integers(0, vals.size, 200003)], desc)


@pytest.mark.parametrize("name", TYPES)
def test_sort_presorted_reversed_keys_only(gpu, name):
    rng = np.random.default_rng(TYPES.index(name))
    x = sorted_keys(rng, name, 150001, 1 << 30, False)
    for desc in (False, True):
        check_sort(gpu, name, x, desc)
        check_sort(gpu, name, x[::-1].copy(), desc)
        check_sort(gpu, name, unsorted_keys(rng, name, 70001, 100), desc, with_vals=False)


def test_sort_u32_typed_matches_merge_sort_u32(gpu):
    """The typed call on uint32 keys ascending gives om_merge_sort_u32's output."""
    rng = np.random.default_rng(2)
    keys = rng.integers(0, 1 << 32, 300001, dtype=np.uint64).astype(np.uint32)
    vals = np.arange(keys.size, dtype=np.uint32)
    k1, v1 = to_dev(keys, "u32"), torch.from_numpy(vals.view(np.int32)).cuda()
    k2, v2 = k1.clone(), v1.clone()
    gpu.merge_sort_u32(k1, v1)
    gpu.merge_sort_keys(k2, v2, key_type="u32")
    torch.cuda.synchronize()
    assert torch.equal(k1, k2) and torch.equal(v1, v2)


@pytest.mark.parametrize("name", ["f32", "f64", "i64"])
def test_unsorted_or_nan_input_terminates_in_bounds(gpu, name):
    """NaN keys (no place in the order) and unsorted keys break the merge's
    precondition: the output is unspecified, but every kernel ends, writes
    nothing outside its output, and the error word reports at most a dropped
    range, never a timed-out wait.  The same holds for the in-place sort of
    keys holding NaN (a NaN makes the order intransitive, so neighbouring
    co-rank searches may disagree and the result need not be a permutation);
    without NaN the sort of the same unsorted keys is checked exactly."""
    npc, tc = _carrier(name)
    dt = NP[name]
    rng = np.random.default_rng(TYPES.index(name))
    for m, n in [(70001, 50003), (5000, 3)]:
        A = rng.integers(-1000, 1000, m).astype(dt)
        B = rng.integers(-1000, 1000, n).astype(dt)
        if np.issubdtype(dt, np.floating):
            A[rng.integers(0, m, m // 10)] = np.nan
            B = np.sort(B)
            B[n // 2] = np.nan
        total = m + n
        sentinel = -0x5A5A5A5B
        buf = torch.full((total + 2 * GUARD + 4,), sentinel, dtype=tc, device="cuda")
        C = buf[GUARD: GUARD + total]
        for desc in (False, True):
            gpu.merge_keys(to_dev(A, name), to_dev(B, name), C, key_type=name, descending=desc)
            torch.cuda.synchronize()
            assert gpu.device_error() in (0, 2), "a kernel wait timed out"
            h = buf.cpu().numpy()
            assert np.all(h[:GUARD] == sentinel) and np.all(h[GUARD + total:] == sentinel), "merge wrote outside C"
        # in-place sort of the same keys inside guard bands
        keys = np.concatenate([A, B])
        sbuf = torch.full((total + 2 * GUARD + 4,), sentinel, dtype=tc, device="cuda")
        K = sbuf[GUARD: GUARD + total]
        K.copy_(torch.from_numpy(keys.view(npc)))
        gpu.merge_sort_keys(K, key_type=name)
        torch.cuda.synchronize()
        assert gpu.device_error() in (0, 2), "a sort wait timed out"
        h = sbuf.cpu().numpy()
        assert np.all(h[:GUARD] == sentinel) and np.all(h[GUARD + total:] == sentinel), "sort wrote outside its keys"
        if not np.issubdtype(dt, np.floating):
            # no NaN: an ordinary sort of unsorted keys, fully defined
            assert np.array_equal(K.cpu().numpy().view(dt), np.sort(keys)), "int64 sort differs"


@pytest.mark.parametrize("name", TYPES)
@pytest.mark.parametrize("offs", [(0, 0, 0), (1, 0, 0), (0, 1, 3), (3, 2, 1), (2, 3, 0), (1, 1, 1)])
def test_one_sided_ranges(gpu, name, offs):
    """Output ranges that take every element from one side: A wholly before
    B (and B wholly before A), runs that alternate in long blocks, every
    16-byte phase of A, B and C, both orders."""
    if np.dtype(NP[name]).itemsize == 8:
        offs = tuple(o & 1 for o in offs)
    rng = np.random.default_rng(sum(offs) * 7 + TYPES.index(name))
    for desc in (False, True):
        lo = np.sort(rng.integers(0, 1 << 20, 300001)).astype(NP[name])
        hi = np.sort(rng.integers(1 << 20, 1 << 21, 200003)).astype(NP[name])
        A, B = (lo, hi) if not desc else (hi[::-1].copy(), lo[::-1].copy())
        check(gpu, name, A, B, desc, offs)
        check(gpu, name, B, A, desc, offs)
        # long alternating blocks: most ranges one-sided, a few straddle a block edge
        blocks = np.arange(2 * 40 * 9000).reshape(80, 9000)
        keys = (blocks // 3).astype(NP[name]) if not np.issubdtype(NP[name], np.floating) \
            else (blocks / 3.0).astype(NP[name])
        A2 = np.sort(keys[0::2].ravel())
        B2 = np.sort(keys[1::2].ravel())
        if desc:
            A2, B2 = A2[::-1].copy(), B2[::-1].copy()
        check(gpu, name, A2, B2, desc, offs)

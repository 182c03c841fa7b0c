"""Randomised GPU parity: many merges and sorts of random shapes, value
spans, tie densities, pointer alignments, key types and orders, each checked
bit for bit against the CPU oracle.  Seeds are fixed, so a failure names the
case and reproduces."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("merge_path")]

NP = {"i32": np.int32, "u32": np.uint32, "f32": np.float32, "i64": np.int64, "u64": np.uint64, "f64": np.float64}


def _carrier(dt):
    return (np.int32, torch.int32) if np.dtype(dt).itemsize == 4 else (np.int64, torch.int64)


def _dev(x, offset):
    npc, tc = _carrier(x.dtype)
    h = torch.from_numpy(np.ascontiguousarray(x).view(npc))
    buf = torch.empty(h.numel() + 4, dtype=tc, device="cuda")
    view = buf[offset: offset + h.numel()]
    view.copy_(h)
    return view


def _keys(rng, dt, size, span):
    if np.issubdtype(dt, np.floating):
        return (rng.integers(-span, span + 1, size).astype(np.float64) * 0.5).astype(dt)
    if np.issubdtype(dt, np.unsignedinteger):
        return rng.integers(0, min(span, np.iinfo(dt).max), size, dtype=np.uint64, endpoint=True).astype(dt)
    return rng.integers(-span, span + 1, size, dtype=np.int64).astype(dt)


@pytest.mark.parametrize("seed", range(150))
def test_random_merge(gpu, seed):
    rng = np.random.default_rng(1000 + seed)
    name = ["i32", "i32", "u32", "f32", "i64", "u64", "f64"][seed % 7]
    dt = NP[name]
    desc = bool(seed % 3 == 0) and name != "i32"
    size_pick = rng.integers(0, 4)
    m = int(rng.integers(0, [50, 5000, 200000, 900000][size_pick] + 1))
    n = int(rng.integers(0, [50, 5000, 200000, 900000][int(rng.integers(0, 4))] + 1))
    span = int(rng.choice([1, 3, 100, 1 << 20, 1 << 30]))
    A = np.sort(_keys(rng, dt, m, span), kind="stable")
    B = np.sort(_keys(rng, dt, n, span), kind="stable")
    if desc:
        A, B = A[::-1].copy(), B[::-1].copy()
    g = 16 // np.dtype(dt).itemsize
    offs = [int(rng.integers(0, g)) for _ in range(3)]
    npc, tc = _carrier(dt)
    sentinel = -0x5A5A5A5B
    buf = torch.full((m + n + 80,), sentinel, dtype=tc, device="cuda")
    C = buf[36 + offs[2]: 36 + offs[2] + m + n]
    if name == "i32" and not desc:
        gpu.merge_i32(_dev(A, offs[0]), _dev(B, offs[1]), C)
    else:
        gpu.merge_keys(_dev(A, offs[0]), _dev(B, offs[1]), C, key_type=name, descending=desc)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    h = buf.cpu().numpy()
    assert np.all(h[: 36 + offs[2]] == sentinel) and np.all(h[36 + offs[2] + m + n:] == sentinel)
    want = oracle.merge_keys(A, B, descending=desc)
    got = C.cpu().numpy()
    assert np.array_equal(got, want.view(npc)), (name, desc, m, n, span, offs)


@pytest.mark.parametrize("seed", range(40))
def test_random_sort(gpu, seed):
    rng = np.random.default_rng(5000 + seed)
    name = ["u32", "i32", "f32", "i64", "f64"][seed % 5]
    dt = NP[name]
    desc = bool(seed % 2)
    n = int(rng.integers(0, [100, 10000, 300000, 2000000][int(rng.integers(0, 4))] + 1))
    keys = _keys(rng, dt, n, int(rng.choice([2, 50, 1 << 30])))
    with_vals = np.dtype(dt).itemsize == 4 and bool(seed % 3)
    npc, tc = _carrier(dt)
    dk = torch.from_numpy(keys.view(npc).copy()).cuda()
    dv = torch.arange(n, dtype=torch.int32, device="cuda") if with_vals else None
    if name == "u32" and not desc:
        gpu.merge_sort_u32(dk, dv)
    else:
        gpu.merge_sort_keys(dk, dv, key_type=name, descending=desc)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    wk, wv = oracle.merge_sort_keys(keys, np.arange(n, dtype=np.uint32), descending=desc)
    assert np.array_equal(dk.cpu().numpy(), wk.view(npc)), (name, desc, n)
    if with_vals:
        assert np.array_equal(dv.cpu().numpy().view(np.uint32), wv), (name, desc, n)

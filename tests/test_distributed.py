"""Multi-rank merge split by co-rank and multi-rank sample sort
(ordered_merge_gb300.distributed) on CPU ranks with the gloo backend.

Each case generates the whole A and B from a seed in every rank, deals each
rank a contiguous piece of each (uneven pieces, some empty), and runs the
distributed merge with the oracle's merge as the per-rank merge.  Every rank
checks that its global co-ranks equal the oracle's co-rank (the pages'
bisection) at k_r = floor(r (m + n) / P), that its output slice is the
oracle's merge of the whole inputs over [k_r, k_{r+1}), and that the slices
are balanced.  The sample sort deals uint32 keys with their global
positions as values; every rank's bucket must equal the oracle's stable sort
of all keys over that bucket's place in the sequence.  A GPU test runs both
with the library's CUDA merge, pair merge and sort as the per-rank steps.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def make_case(name, seed):
    rng = np.random.default_rng(seed)
    if name == "distinct":
        A = np.arange(0, 2 * 3001, 2, dtype=np.int32)
        B = np.arange(1, 2 * 2500, 2, dtype=np.int32)
    elif name == "heavy_ties":
        A = np.sort(rng.integers(0, 3, 4000)).astype(np.int32)
        B = np.sort(rng.integers(0, 3, 3500)).astype(np.int32)
    elif name == "all_A_first":
        A = np.sort(rng.integers(-500, 0, 2000)).astype(np.int32)
        B = np.sort(rng.integers(0, 500, 2600)).astype(np.int32)
    elif name == "all_B_first":
        A = np.sort(rng.integers(1, 500, 2600)).astype(np.int32)
        B = np.sort(rng.integers(-500, 1, 2000)).astype(np.int32)
    elif name == "uniform":
        A = np.sort(rng.integers(-2**31, 2**31, 9000)).astype(np.int32)
        B = np.sort(rng.integers(-2**31, 2**31, 7000)).astype(np.int32)
    elif name == "empty_A":
        A = np.zeros(0, dtype=np.int32)
        B = np.sort(rng.integers(-9, 9, 777)).astype(np.int32)
    elif name == "tiny":
        A = np.array([1, 7, 8, 9, 10], dtype=np.int32)  # the co-rank page's worked example
        B = np.array([7, 10, 10, 12], dtype=np.int32)
    else:
        raise ValueError(name)
    return A, B


def make_sort_case(name, seed):
    """uint32 keys and their global input positions as values (so the
    stable sort is unique)."""
    rng = np.random.default_rng(seed)
    if name == "uniform":
        keys = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    elif name == "heavy_ties":
        keys = rng.integers(0, 5, 15000, dtype=np.uint64).astype(np.uint32)
    elif name == "sign_bit":  # unsigned order across the sign bit
        keys = rng.choice(np.array([0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF], dtype=np.uint32), 9000)
    elif name == "presorted":
        keys = np.arange(12000, dtype=np.uint32)
    elif name == "tiny":
        keys = np.array([5, 3, 5, 1], dtype=np.uint32)
    else:
        raise ValueError(name)
    return keys, np.arange(keys.size, dtype=np.uint32)


def deal(x, world, rng):
    """Contiguous pieces of x, one per rank, of random (possibly zero) lengths."""
    cuts = np.sort(rng.integers(0, x.size + 1, world - 1)) if x.size else np.zeros(world - 1, dtype=np.int64)
    bounds = [0] + [int(c) for c in cuts] + [x.size]
    return [x[bounds[r]:bounds[r + 1]] for r in range(world)]


def _worker(rank, world, port, cases, device, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        import oracle
        from ordered_merge_gb300 import distributed as D

        dist.init_process_group("gloo", rank=rank, world_size=world)
        if device == "cuda":
            torch.cuda.set_device(0)
            local_merge = None  # the library's CUDA merge
        else:
            def local_merge(a, b):
                return torch.from_numpy(oracle.merge_i32(a.numpy(), b.numpy()))
        for name, seed in cases:
            A, B = make_case(name, seed)
            rng = np.random.default_rng(seed + 1000 * world)
            pa = deal(A, world, rng)[rank]
            pb = deal(B, world, rng)[rank]
            ta = torch.from_numpy(pa.copy()).to(device)
            tb = torch.from_numpy(pb.copy()).to(device)
            a_offs = D.piece_offsets(ta.numel())
            b_offs = D.piece_offsets(tb.numel())
            ks = D.split_ranks(A.size + B.size, world)
            inner, _ = D.global_coranks(ks[1:-1], ta, a_offs, tb, b_offs)
            for k, i in zip(ks[1:-1], inner):
                assert i == oracle.corank_pages(k, A, B), (name, k, i)
            C, k_lo, k_hi = D.merge_i32(ta, tb, local_merge=local_merge)
            want = oracle.merge_i32(A, B)
            assert (k_lo, k_hi) == (ks[rank], ks[rank + 1])
            assert C.numel() == k_hi - k_lo
            assert np.array_equal(C.cpu().numpy(), want[k_lo:k_hi]), (name, rank)
            assert abs((k_hi - k_lo) - (A.size + B.size) / world) <= 1
        for name, seed in SORT_CASES:
            keys, vals = make_sort_case(name, seed)
            rng = np.random.default_rng(seed + 77 * world)
            pk = deal(keys, world, rng)
            rng = np.random.default_rng(seed + 77 * world)
            pv = deal(vals, world, rng)
            tk = torch.from_numpy(pk[rank].view(np.int32).copy()).to(device)
            tv = torch.from_numpy(pv[rank].view(np.int32).copy()).to(device)
            if device == "cuda":
                bk, bv = D.sample_sort_u32(tk, tv)
            else:
                def lsort(k, v):
                    a, b = oracle.merge_sort_pairs_u32(k.numpy().view(np.uint32), v.numpy().view(np.uint32))
                    return torch.from_numpy(a.view(np.int32)), torch.from_numpy(b.view(np.int32))

                def lmerge(ka, va, kb, vb):
                    kc, vc = oracle.merge_pairs_u32(ka.numpy().view(np.uint32), va.numpy().view(np.uint32),
                                                    kb.numpy().view(np.uint32), vb.numpy().view(np.uint32))
                    return torch.from_numpy(kc.view(np.int32)), torch.from_numpy(vc.view(np.int32))

                bk, bv = D.sample_sort_u32(tk, tv, local_sort=lsort, local_merge=lmerge)
            offs = D.piece_offsets(bk.numel())
            wk, wv = oracle.merge_sort_pairs_u32(keys, vals)
            assert offs[-1] == keys.size
            lo, hi = offs[rank], offs[rank + 1]
            assert np.array_equal(bk.cpu().numpy().view(np.uint32), wk[lo:hi]), (name, rank)
            assert np.array_equal(bv.cpu().numpy().view(np.uint32), wv[lo:hi]), (name, rank)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent, which fails the test
        import traceback

        q.put((rank, traceback.format_exc()))


def _run(world, cases, device="cpu"):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cases, device, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        r, msg = q.get(timeout=300)
        results[r] = msg
    for p in procs:
        p.join(timeout=60)
    bad = {r: m for r, m in results.items() if m != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{m}" for r, m in bad.items())


CASES = [(n, s) for s, n in enumerate(["distinct", "heavy_ties", "all_A_first", "all_B_first", "uniform",
                                        "empty_A", "tiny"])]
SORT_CASES = [(n, 50 + s) for s, n in enumerate(["uniform", "heavy_ties", "sign_bit", "presorted", "tiny"])]


@pytest.mark.parametrize("world", [2, 3, 4])
def test_distributed_merge_matches_oracle(world):
    _run(world, CASES)


def test_global_corank_rounds_are_few():
    """The 33-way search needs about log33(range) + 1 rounds, not log2."""
    import torch.distributed as dist  # noqa: F401  (single process: no group needed below)
    from ordered_merge_gb300 import distributed as D

    # the update rule alone, on one process: simulate the owners with full arrays
    rng = np.random.default_rng(3)
    A = np.sort(rng.integers(-2**31, 2**31, 1 << 20)).astype(np.int32)
    B = np.sort(rng.integers(-2**31, 2**31, 1 << 20)).astype(np.int32)
    port = _free_port()
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        ta, tb = torch.from_numpy(A), torch.from_numpy(B)
        ks = [1 << 19, 1 << 20, 3 << 19]
        got, rounds = D.global_coranks(ks, ta, [0, A.size], tb, [0, B.size])
        import oracle

        assert got == [oracle.corank_pages(k, A, B) for k in ks]
        assert rounds <= 6, rounds  # log33(2^20) + 1 = 5
    finally:
        dist.destroy_process_group()


@pytest.mark.gpu
def test_distributed_merge_cuda_local_merge():
    """Two ranks on one GPU exchanging through gloo (host staging); each
    rank's window merge runs in the library's CUDA kernel.  No kernel waits
    on another rank: ranks meet only in host collectives between launches."""
    _run(2, CASES, device="cuda")

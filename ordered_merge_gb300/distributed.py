"""Stable merge across several GPUs, split by the co-rank function.

One process per GPU.  A and B are each block-distributed over the ranks of a
``torch.distributed`` process group: rank r holds one contiguous piece of A
and one of B, in rank order (piece lengths may differ and may be zero).  The
merged C is block-distributed too: rank r receives C[k_r, k_{r+1}) with
k_r = floor(r * (m + n) / P), so every rank gets the same number of outputs
(up to one).

The split follows the co-rank function ("Co-rank Function 實作與 Basic
Parallel Merge Kernel", §Co-rank Function 定義與不變式: A[0..i) and B[0..j)
with i + j = k are exactly the first k outputs; "Tiled 與 Circular Buffer
Merge Kernel", §Block-Level Co-Rank: one co-rank per output block, here one
per GPU):

1. the P - 1 interior co-ranks i_r = co_rank(k_r) are found by one search run
   in lockstep on every rank.  Each round probes up to 32 candidates per
   splitter (the higher-radix search of the pages' overview); the probed
   elements A[c - 1] and B[k - c] live on whichever ranks own them, so every
   rank writes the probes it owns into a buffer of zeros and one all-reduce
   (sum) hands all of them to every rank.  About log33(m) + 1 rounds.
2. rank r needs A[i_r, i_{r+1}) and B[j_r, j_{r+1}) (j = k - i).  Those
   windows tile A and B in rank order, so every rank's piece splits into
   consecutive parts, one per destination, and one all-to-all moves them
   (no packing).
3. rank r merges its two windows on its own GPU (om_merge_i32).  Its output
   is exactly C[k_r, k_{r+1}).

Only step 3 computes the merge; steps 1-2 are control (comparisons of
gathered scalars on the host) and data movement through the process
group's collectives.  With the NCCL backend the pieces move GPU to GPU;
with gloo they are staged through host memory.  ``local_merge`` replaces
step 3 (for example a CPU reference in tests); the default is the library's
CUDA merge, which refuses CPU tensors: there is no CPU fallback.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist

RADIX = 32  # probes per splitter per round


def _coll_device(group) -> torch.device:
    """Device of the tensors handed to the group's collectives."""
    backend = dist.get_backend(group)
    if backend == "nccl":
        return torch.device("cuda", torch.cuda.current_device())
    return torch.device("cpu")


def piece_offsets(local_len: int, group=None) -> List[int]:
    """Global start offsets of every rank's piece (plus the total at the end),
    from the local piece lengths (one all-gather)."""
    world = dist.get_world_size(group)
    dev = _coll_device(group)
    mine = torch.tensor([int(local_len)], dtype=torch.int64, device=dev)
    lens = [torch.zeros(1, dtype=torch.int64, device=dev) for _ in range(world)]
    dist.all_gather(lens, mine, group=group)
    offs = [0]
    for t in lens:
        offs.append(offs[-1] + int(t.item()))
    return offs


def split_ranks(total: int, world: int) -> List[int]:
    """k_r = floor(r * total / world) for r = 0 .. world (balanced output blocks)."""
    return [(r * total) // world for r in range(world + 1)]


def _owned_values(local: torch.Tensor, offs: Sequence[int], rank: int, idx: Sequence[int]) -> List[int]:
    """Values at the global indices idx that this rank owns, 0 at the others."""
    lo, hi = offs[rank], offs[rank + 1]
    pos = [x - lo for x in idx if lo <= x < hi]
    vals = local[torch.tensor(pos, dtype=torch.int64, device=local.device)].tolist() if pos else []
    out, it = [], iter(vals)
    for x in idx:
        out.append(int(next(it)) if lo <= x < hi else 0)
    return out


def global_coranks(ks: Sequence[int], A_local: torch.Tensor, a_offs: Sequence[int], B_local: torch.Tensor,
                   b_offs: Sequence[int], group=None, radix: int = RADIX) -> Tuple[List[int], int]:
    """co_rank(k) of the block-distributed A and B for every k in ks, found in
    lockstep on all ranks of the group; returns (the co-ranks, rounds used).

    co_rank(k) is the largest i in [max(0, k - n), min(k, m)] with i at the
    lower bound or A[i - 1] <= B[k - i]: on sorted input the pages' i, on any
    input a value in that interval (each round shrinks every interval, so
    the search always ends)."""
    rank = dist.get_rank(group)
    dev = _coll_device(group)
    m, n = a_offs[-1], b_offs[-1]
    lo = [max(0, k - n) for k in ks]
    hi = [min(k, m) for k in ks]
    rounds = 0
    while any(h > l for l, h in zip(lo, hi)):
        rounds += 1
        cands = []  # (splitter, candidate)
        for s, (l, h) in enumerate(zip(lo, hi)):
            span = h - l
            if span <= 0:
                continue
            if span > radix:
                cands += [(s, l + (span * (t + 1)) // (radix + 1)) for t in range(radix)]  # l < c < h
            else:
                cands += [(s, l + 1 + t) for t in range(span)]
        a_idx = [c - 1 for _, c in cands]
        b_idx = [ks[s] - c for s, c in cands]
        buf = torch.tensor(_owned_values(A_local, a_offs, rank, a_idx) + _owned_values(B_local, b_offs, rank, b_idx),
                           dtype=torch.int64, device=dev)
        dist.all_reduce(buf, op=dist.ReduceOp.SUM, group=group)  # exactly one owner per probe
        vals = buf.tolist()
        na = len(cands)
        passed = {}
        for q, (s, _) in enumerate(cands):
            passed.setdefault(s, []).append(vals[q] <= vals[na + q])  # A first on ties
        for s, ps in passed.items():
            l, h = lo[s], hi[s]
            span = h - l
            t = sum(ps)
            if span > radix:
                lo[s] = l if t == 0 else l + (span * t) // (radix + 1)
                hi[s] = h if t == radix else l + (span * (t + 1)) // (radix + 1) - 1
            else:
                lo[s] = hi[s] = l + t
    return lo, rounds


def _overlaps(offs: Sequence[int], wins: Sequence[int], who: int, by_src: bool) -> List[int]:
    """Lengths of the overlaps of one piece with every window (by_src False:
    piece `who` against each window) or of one window with every piece
    (by_src True: window `who` against each piece)."""
    out = []
    P = len(offs) - 1
    for x in range(P):
        p, w = (x, who) if by_src else (who, x)
        a0, a1 = offs[p], offs[p + 1]
        w0, w1 = wins[w], wins[w + 1]
        out.append(max(0, min(a1, w1) - max(a0, w0)))
    return out


def _exchange(local: torch.Tensor, offs: Sequence[int], wins: Sequence[int], group) -> torch.Tensor:
    """All-to-all of a block-distributed array into the windows wins
    (window r = [wins[r], wins[r+1]) goes to rank r); returns this rank's window."""
    rank = dist.get_rank(group)
    send = _overlaps(offs, wins, rank, by_src=False)
    recv = _overlaps(offs, wins, rank, by_src=True)
    dev = _coll_device(group)
    src = local.to(dev) if local.device != dev else local
    out = torch.empty(sum(recv), dtype=local.dtype, device=dev)
    dist.all_to_all_single(out, src.contiguous(), recv, send, group=group)
    return out.to(local.device) if out.device != local.device else out


def merge_i32(A_local: torch.Tensor, B_local: torch.Tensor, group=None,
              local_merge: Optional[Callable[[torch.Tensor, torch.Tensor], torch.Tensor]] = None):
    """Stable merge of int32 A and B block-distributed over the group (ties
    take A first).  Returns (C_local, k_lo, k_hi): this rank's C[k_lo, k_hi).

    local_merge(A_window, B_window) -> C_window does step 3; default: the
    library's CUDA merge (the windows stay on A_local's device)."""
    if local_merge is None:
        from . import merge_i32 as local_merge  # the CUDA kernel; raises on CPU tensors
    if A_local.dtype != torch.int32 or B_local.dtype != torch.int32:
        raise ValueError("A and B must be int32")
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    a_offs = piece_offsets(A_local.numel(), group)
    b_offs = piece_offsets(B_local.numel(), group)
    m, n = a_offs[-1], b_offs[-1]
    ks = split_ranks(m + n, world)
    inner, _ = global_coranks(ks[1:-1], A_local, a_offs, B_local, b_offs, group)
    i_split = [0] + inner + [m]
    j_split = [k - i for k, i in zip(ks, i_split)]
    A_win = _exchange(A_local, a_offs, i_split, group)
    B_win = _exchange(B_local, b_offs, j_split, group)
    C = local_merge(A_win, B_win)
    return C, ks[rank], ks[rank + 1]


# ----------------------------------------------------------------- sample sort


def _local_bounds(keys: torch.Tensor, probes: Sequence[Tuple[int, bool]], radix: int = RADIX) -> List[int]:
    """For sorted uint32 keys (carried in an int32 tensor) and probes (v, upper):
    the number of keys < v (upper False) or <= v (upper True), by a search run
    on the host over values gathered from the device, radix + 1 ways a round."""
    n = keys.numel()
    lo = [0] * len(probes)   # answer in [lo, hi]
    hi = [n] * len(probes)
    while any(h > l for l, h in zip(lo, hi)):
        cands = []
        for s, (l, h) in enumerate(zip(lo, hi)):
            span = h - l
            if span <= 0:
                continue
            if span > radix:
                cands += [(s, l + (span * (t + 1)) // (radix + 1)) for t in range(radix)]
            else:
                cands += [(s, l + 1 + t) for t in range(span)]
        idx = torch.tensor([c - 1 for _, c in cands], dtype=torch.int64, device=keys.device)
        vals = [x & 0xFFFFFFFF for x in keys[idx].tolist()]
        passed = {}
        for (s, _), x in zip(cands, vals):
            v, upper = probes[s]
            passed.setdefault(s, []).append(x <= v if upper else x < v)  # key[c-1] still counts
        for s, ps in passed.items():
            l, h = lo[s], hi[s]
            span = h - l
            t = sum(ps)
            if span > radix:
                lo[s] = l if t == 0 else l + (span * t) // (radix + 1)
                hi[s] = h if t == radix else l + (span * (t + 1)) // (radix + 1) - 1
            else:
                lo[s] = hi[s] = l + t
    return lo


def sample_sort_u32(keys_local: torch.Tensor, vals_local: torch.Tensor, group=None, oversample: int = 8,
                    local_sort: Optional[Callable] = None, local_merge: Optional[Callable] = None):
    """Stable sort of uint32 keys (unsigned order, carried in int32 or uint32
    tensors) with uint32 values, block-distributed over the group; equal keys
    keep their global input order (rank order, then position).  Returns
    (keys, vals) of this rank's bucket; the buckets in rank order are the
    sorted sequence.

    The sample sort of "排序 (Sorting) 練習題" (§sample sort): every rank
    sorts its piece (om_merge_sort_u32), takes `oversample` * P regular
    samples, all ranks agree on P - 1 splitters from the gathered samples,
    every piece is cut at the splitters and one all-to-all deals the parts
    to their buckets, and each rank merges the P sorted parts it received
    (om_merge_pairs_u32, earlier rank first on ties).  Splitters are
    (key, rank, position) triples, so equal keys are cut consistently and
    stability holds across ranks.  Bucket sizes follow the samples (they are
    balanced only approximately, as in any sample sort).

    local_sort(keys, vals) -> (keys, vals) and local_merge(ka, va, kb, vb)
    -> (kc, vc) replace the library's CUDA sort and pair merge (tests)."""
    if local_sort is None:
        from . import merge_sort_u32

        def local_sort(k, v):
            k, v = k.clone(), v.clone()
            merge_sort_u32(k, v)
            return k, v
    if local_merge is None:
        from . import merge_pairs_u32 as local_merge
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = _coll_device(group)
    keys, vals = local_sort(keys_local, vals_local)
    n = keys.numel()
    # regular samples (key, rank, position) of the sorted piece
    s = max(1, oversample) * world
    pos = sorted({(j * n) // (s + 1) for j in range(1, s + 1)} if n else set())
    pos = [p for p in pos if p < n]
    sk = [x & 0xFFFFFFFF for x in keys[torch.tensor(pos, dtype=torch.int64, device=keys.device)].tolist()] if pos else []
    rows = [[k, rank, p] for p, k in zip(pos, sk)] + [[-1, -1, -1]] * (s - len(pos))  # -1 rows: no sample
    mine = torch.tensor(rows, dtype=torch.int64, device=dev)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine, group=group)
    samples = sorted(tuple(int(x) for x in row) for g in gathered for row in g.cpu().tolist() if row[0] >= 0)
    if samples:
        splitters = [samples[((r + 1) * len(samples)) // world - 1] for r in range(world - 1)]
    else:
        splitters = []
    # cut this rank's sorted piece at every splitter: elements before the
    # triple (key, rank, position) in the order key, then rank, then position
    probes = []
    for (kv, rr, pp) in splitters:
        probes.append((kv, rank < rr))  # earlier rank: all equal keys precede; later: none
    bounds = _local_bounds(keys, probes) if probes else []
    cut = []
    for (kv, rr, pp), b in zip(splitters, bounds):
        cut.append(pp if rr == rank else b)
    cut = [0] + [max(0, min(n, c)) for c in cut] + [n]
    for t in range(1, len(cut)):  # monotone (splitters are sorted)
        cut[t] = max(cut[t], cut[t - 1])
    send = [cut[t + 1] - cut[t] for t in range(world)]
    send_t = torch.tensor(send, dtype=torch.int64, device=dev)
    all_send = [torch.empty_like(send_t) for _ in range(world)]
    dist.all_gather(all_send, send_t, group=group)
    recv = [int(all_send[q][rank].item()) for q in range(world)]

    def move(x):
        src = x.to(dev) if x.device != dev else x
        out = torch.empty(sum(recv), dtype=x.dtype, device=dev)
        dist.all_to_all_single(out, src.contiguous(), recv, send, group=group)
        return out.to(x.device) if out.device != x.device else out

    rk, rv = move(keys), move(vals)
    # the received parts are sorted runs in source-rank order: merge them
    # pairwise, earlier runs as A, so ties keep rank order
    offs = [0]
    for c in recv:
        offs.append(offs[-1] + c)
    runs = [(rk[offs[q]:offs[q + 1]], rv[offs[q]:offs[q + 1]]) for q in range(world)]
    while len(runs) > 1:
        nxt = []
        for t in range(0, len(runs) - 1, 2):
            (ka, va), (kb, vb) = runs[t], runs[t + 1]
            if ka.numel() == 0:
                nxt.append((kb, vb))
            elif kb.numel() == 0:
                nxt.append((ka, va))
            else:
                nxt.append(local_merge(ka.contiguous(), va.contiguous(), kb.contiguous(), vb.contiguous()))
        if len(runs) % 2:
            nxt.append(runs[-1])
        runs = nxt
    return runs[0]

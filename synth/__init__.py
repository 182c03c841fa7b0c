"""Seeded synthetic inputs for the stable merge workloads.

This module only *generates* inputs; it holds none of the merge's arithmetic
(no co-rank, no merge, no merge sort), so both the GPU path's tests/bench and
the CPU oracle can draw from it.  Sorting a generated array so that it can be
a merge input uses a library sort (``numpy.sort`` on the host, ``torch.sort``
on the device): the sorted multiset is unique, so both give the same array.

Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are the
ones Vigna published for ``splitmix64.c``), used counter-style:
``x_i = mix(seed + (i + 1) * 0x9E3779B97F4A7C15)``.  Mappings from a 64-bit
draw ``x``:

* full-range int32: the top 32 bits reinterpreted as two's-complement int32
* full-range uint32: the top 32 bits
* uniform integer in ``[0, bound)``: ``((x >> 32) * bound) >> 32``
  (Lemire's multiply-shift range reduction)

Workloads (lengths in elements):

1. ``evens_odds``: A = 0, 2, 4, ... (2^21 + 611 elements), B = 1, 3, 5, ...
   (2^21 elements); int32; no randomness.
2. ``pairs_ties``: m = n = 2^24 uint32 keys uniform in [0, 16), each side
   sorted; values = (side << 31) | position in that side's sorted array.
3. ``skewed``: A = 2^28 sorted full-range int32, B = 2^10 sorted int32 uniform
   in [-2^20, 2^20].
4. ``uniform``: A, B = 2^28 sorted full-range int32 each.
5. ``sort``: 2^26 full-range uint32 keys (unsorted), values = 0 .. n-1.

Other key types and descending order (same bytes per merge as ``uniform``):

6. ``f64``: A, B = 2^27 sorted float64 each, value = a full-range int32 draw
   times 2^-20 (exact; negatives, both signs).
7. ``i64_desc``: A, B = 2^27 int64 each, sorted nonincreasing, value =
   (top 32 bits of one draw) << 32 | (top 32 bits of a second stream's draw).
8. ``sort_f32_desc``: 2^26 float32 keys (a full-range int32 draw times 2^-8,
   rounded to float32), values = 0 .. n-1, to be sorted nonincreasing.
9. ``sort_f64``: 2^26 float64 keys (int32 draw times 2^-20), keys only.

Every length can be scaled down for tests (``scale_log2``), keeping the
value distribution and structure.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

SEEDS = {"evens_odds": 1, "pairs_ties": 2, "skewed": 3, "uniform": 4, "sort": 5,
         "f64": 6, "i64_desc": 7, "sort_f32_desc": 8, "sort_f64": 9}

WORKLOADS = ("evens_odds", "pairs_ties", "skewed", "uniform", "sort", "f64", "i64_desc", "sort_f32_desc",
             "sort_f64")


def side_seed(workload: str, side: int) -> int:
    """Seed of one input array: workload seed in the high bits, side (0=A, 1=B) low."""
    return (SEEDS[workload] << 8) | side


def splitmix64(seed: int, count: int, start: int = 0, chunk: int = 1 << 24) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the counter-based SplitMix64 stream."""
    out = np.empty(count, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    tmp = np.empty(min(chunk, max(count, 1)), dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, count, chunk):
            hi = min(count, lo + chunk)
            z = out[lo:hi]
            t = tmp[: hi - lo]
            z[:] = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            np.multiply(z, GOLDEN_GAMMA, out=z)
            np.add(z, s, out=z)
            np.right_shift(z, np.uint64(30), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M1, out=z)
            np.right_shift(z, np.uint64(27), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M2, out=z)
            np.right_shift(z, np.uint64(31), out=t)
            np.bitwise_xor(z, t, out=z)
    return out


def np_top32(seed: int, count: int) -> np.ndarray:
    """Top 32 bits of each draw (numpy reference implementation)."""
    return (splitmix64(seed, count) >> np.uint64(32)).astype(np.uint32)


def np_below(seed: int, count: int, bound: int) -> np.ndarray:
    """Uniform integers in ``[0, bound)`` (numpy reference implementation)."""
    hi = splitmix64(seed, count)
    np.right_shift(hi, np.uint64(32), out=hi)
    np.multiply(hi, np.uint64(bound), out=hi)
    np.right_shift(hi, np.uint64(32), out=hi)
    return hi.astype(np.uint32)


# The same two draws in plain C (synth/gen.c), about 50x faster; built with gcc
# on first use.  tests/test_synth.py checks it against the numpy version.
_HERE = os.path.dirname(os.path.abspath(__file__))
_GEN_SRC = os.path.join(_HERE, "gen.c")
_GEN_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_gen = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_GEN_LIB) and os.path.getmtime(_GEN_LIB) >= os.path.getmtime(_GEN_SRC):
        return _GEN_LIB
    os.makedirs(os.path.dirname(_GEN_LIB), exist_ok=True)
    tmp = _GEN_LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _GEN_SRC])
    os.replace(tmp, _GEN_LIB)
    return _GEN_LIB


def _lib():
    global _gen
    if _gen is None:
        lib = ctypes.CDLL(build())
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_top32.argtypes = [u64, i64, i64, p]
        lib.synth_top32.restype = None
        lib.synth_below.argtypes = [u64, i64, i64, u64, p]
        lib.synth_below.restype = None
        _gen = lib
    return _gen


def uniform_u32(seed: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint32)
    _lib().synth_top32(seed & 0xFFFFFFFFFFFFFFFF, 0, count, out.ctypes.data_as(ctypes.c_void_p))
    return out


def uniform_i32(seed: int, count: int) -> np.ndarray:
    return uniform_u32(seed, count).view(np.int32)


def uniform_below(seed: int, count: int, bound: int) -> np.ndarray:
    """Uniform integers in ``[0, bound)`` (bound <= 2^32), as uint32."""
    assert 0 < bound <= (1 << 32)
    out = np.empty(count, dtype=np.uint32)
    _lib().synth_below(seed & 0xFFFFFFFFFFFFFFFF, 0, count, bound, out.ctypes.data_as(ctypes.c_void_p))
    return out


# ------------------------------------------------------------------ sizes --

def sizes(workload: str, scale_log2: int = 0) -> tuple[int, int]:
    """(m, n) of a workload; ``scale_log2`` shrinks the power-of-two parts."""
    s = scale_log2
    if workload == "evens_odds":
        return (1 << (21 - s)) + 611, 1 << (21 - s)
    if workload == "pairs_ties":
        return 1 << (24 - s), 1 << (24 - s)
    if workload == "skewed":
        return 1 << (28 - s), 1 << max(0, 10 - s)
    if workload == "uniform":
        return 1 << (28 - s), 1 << (28 - s)
    if workload in ("sort", "sort_f32_desc", "sort_f64"):
        return 1 << (26 - s), 0
    if workload in ("f64", "i64_desc"):
        return 1 << (27 - s), 1 << (27 - s)
    raise ValueError(workload)


# ---------------------------------------------------------- raw generators --

def evens_odds(m: int, n: int):
    """A = 0, 2, 4, ... (m values), B = 1, 3, 5, ... (n values), int32."""
    A = (2 * np.arange(m, dtype=np.int64)).astype(np.int32)
    B = (2 * np.arange(n, dtype=np.int64) + 1).astype(np.int32)
    return A, B


def raw_i32_full(seed: int, count: int) -> np.ndarray:
    return uniform_i32(seed, count)


def raw_i32_window(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Uniform int32 in the closed interval [lo, hi]."""
    v = uniform_below(seed, count, hi - lo + 1).astype(np.int64) + lo
    return v.astype(np.int32)


def raw_u32_below(seed: int, count: int, bound: int) -> np.ndarray:
    return uniform_below(seed, count, bound).astype(np.uint32)


def host_sorted(x: np.ndarray) -> np.ndarray:
    return np.sort(x, kind="stable")


def raw_f64_scaled(seed: int, count: int, shift: int = 20) -> np.ndarray:
    """Full-range int32 draws times 2^-shift, as float64 (exact)."""
    return np.ldexp(uniform_i32(seed, count).astype(np.float64), -shift)


def raw_f32_scaled(seed: int, count: int, shift: int = 8) -> np.ndarray:
    """Full-range int32 draws times 2^-shift, rounded to float32."""
    return np.ldexp(uniform_i32(seed, count).astype(np.float64), -shift).astype(np.float32)


def raw_i64_full(seed: int, count: int) -> np.ndarray:
    """Full-range int64: top 32 bits of one stream, low 32 of a second."""
    hi = uniform_u32(seed, count).astype(np.uint64) << np.uint64(32)
    lo = uniform_u32(seed ^ (1 << 12), count).astype(np.uint64)
    return (hi | lo).view(np.int64)


def _typed_raw(workload: str, sa: int, sb: int, m: int, n: int):
    """Unsorted raw arrays of the typed workloads (None for B of a sort)."""
    if workload == "f64":
        return raw_f64_scaled(sa, m), raw_f64_scaled(sb, n)
    if workload == "i64_desc":
        return raw_i64_full(sa, m), raw_i64_full(sb, n)
    if workload == "sort_f32_desc":
        return raw_f32_scaled(sa, m), None
    if workload == "sort_f64":
        return raw_f64_scaled(sa, m), None
    raise ValueError(workload)


# key type and order of the typed workloads
TYPED = {"f64": ("f64", False), "i64_desc": ("i64", True), "sort_f32_desc": ("f32", True),
         "sort_f64": ("f64", False)}


# ------------------------------------------------------------- workloads --

def make_host(workload: str, scale_log2: int = 0, seed_offset: int = 0) -> dict:
    """Host (numpy) arrays of one workload, inputs already sorted where the
    workload says so.  Keys: 'A', 'B' (int32 merges); 'keysA', 'valsA',
    'keysB', 'valsB' (pairs); 'keys', 'vals' (sort)."""
    m, n = sizes(workload, scale_log2)
    sa = side_seed(workload, 0) + (seed_offset << 16)
    sb = side_seed(workload, 1) + (seed_offset << 16)
    if workload == "evens_odds":
        A, B = evens_odds(m, n)
        return {"A": A, "B": B}
    if workload == "uniform":
        return {"A": host_sorted(raw_i32_full(sa, m)), "B": host_sorted(raw_i32_full(sb, n))}
    if workload == "skewed":
        return {
            "A": host_sorted(raw_i32_full(sa, m)),
            "B": host_sorted(raw_i32_window(sb, n, -(1 << 20), 1 << 20)),
        }
    if workload == "pairs_ties":
        ka = host_sorted(raw_u32_below(sa, m, 16))
        kb = host_sorted(raw_u32_below(sb, n, 16))
        va = np.arange(m, dtype=np.uint32)
        vb = (np.arange(n, dtype=np.uint32) | np.uint32(1 << 31)).astype(np.uint32)
        return {"keysA": ka, "valsA": va, "keysB": kb, "valsB": vb}
    if workload == "sort":
        return {"keys": uniform_u32(sa, m), "vals": np.arange(m, dtype=np.uint32)}
    if workload in TYPED:
        ra, rb = _typed_raw(workload, sa, sb, m, n)
        desc = TYPED[workload][1]
        if rb is None:
            out = {"keys": ra}
            if workload == "sort_f32_desc":
                out["vals"] = np.arange(m, dtype=np.uint32)
            return out
        A, B = host_sorted(ra), host_sorted(rb)
        if desc:
            A, B = A[::-1].copy(), B[::-1].copy()
        return {"A": A, "B": B}
    raise ValueError(workload)


def make_device(workload: str, device, scale_log2: int = 0, seed_offset: int = 0) -> dict:
    """The same arrays as :func:`make_host`, resident on ``device`` (torch).

    The raw draws are made on the host and sorted on the device with
    ``torch.sort`` (values only), which yields the identical sorted arrays.
    All tensors are int32 (uint32 data is carried bit-for-bit in int32).
    """
    import torch

    m, n = sizes(workload, scale_log2)
    sa = side_seed(workload, 0) + (seed_offset << 16)
    sb = side_seed(workload, 1) + (seed_offset << 16)

    def dev_sorted(raw: np.ndarray):
        t = torch.from_numpy(raw.view(np.int32)).to(device)
        return torch.sort(t).values

    def dev(raw: np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(raw).view(np.int32)).to(device)

    if workload == "evens_odds":
        A, B = evens_odds(m, n)
        return {"A": dev(A), "B": dev(B)}
    if workload == "uniform":
        return {"A": dev_sorted(raw_i32_full(sa, m)), "B": dev_sorted(raw_i32_full(sb, n))}
    if workload == "skewed":
        return {
            "A": dev_sorted(raw_i32_full(sa, m)),
            "B": dev_sorted(raw_i32_window(sb, n, -(1 << 20), 1 << 20)),
        }
    if workload == "pairs_ties":
        # keys < 16, so int32 order equals uint32 order
        ka = dev_sorted(raw_u32_below(sa, m, 16))
        kb = dev_sorted(raw_u32_below(sb, n, 16))
        va = torch.arange(m, dtype=torch.int32, device=device)
        vb = torch.arange(n, dtype=torch.int32, device=device) | torch.tensor(
            np.array([1 << 31], dtype=np.uint32).view(np.int32)[0], device=device)
        return {"keysA": ka, "valsA": va, "keysB": kb, "valsB": vb}
    if workload == "sort":
        return {"keys": dev(uniform_u32(sa, m)), "vals": torch.arange(m, dtype=torch.int32, device=device)}
    if workload in TYPED:
        # typed tensors (float64 / int64 / float32); sorted with torch.sort,
        # whose values equal numpy's for these (no NaN; the only equal keys
        # with different bits, -0.0 and +0.0, cannot occur: zero draws give +0.0)
        ra, rb = _typed_raw(workload, sa, sb, m, n)
        desc = TYPED[workload][1]
        if rb is None:
            out = {"keys": torch.from_numpy(ra).to(device)}
            if workload == "sort_f32_desc":
                out["vals"] = torch.arange(m, dtype=torch.int32, device=device)
            return out
        A = torch.sort(torch.from_numpy(ra).to(device), descending=desc).values
        B = torch.sort(torch.from_numpy(rb).to(device), descending=desc).values
        return {"A": A, "B": B}
    raise ValueError(workload)

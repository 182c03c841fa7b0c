"""CPU oracle for the stable co-rank merge -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
GPU library (``ordered_merge_gb300``) never imports it and shares no code with
it: the arithmetic lives in ``merge_oracle.c`` (plain C, single thread), built
here with gcc and called through ctypes on numpy arrays.

Functions (see ``merge_oracle.c`` for the definition each one restates):

* :func:`merge_i32`, :func:`merge_u32`, :func:`merge_f32`, :func:`merge_keys`,
  :func:`merge_pairs_u32` -- two-pointer stable merge (O1)
* :func:`corank_pages` -- the pages' co-rank bisection, with trace (O2)
* :func:`corank_count` -- co-rank by counting merge steps (O3)
* :func:`merge_sort_pairs_u32`, :func:`merge_sort_keys` -- bottom-up stable
  merge sort from O1 (O4)
* :func:`merge_at_i32` -- one output element C[k] via O2 (O5)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "merge_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile ``merge_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC]
    )
    os.replace(tmp, _LIB)
    return _LIB


class TraceRow(ctypes.Structure):
    _fields_ = [
        ("i_low", ctypes.c_int64),
        ("i", ctypes.c_int64),
        ("j", ctypes.c_int64),
        ("j_low", ctypes.c_int64),
        ("verdict", ctypes.c_int32),
        ("delta", ctypes.c_int64),
    ]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` overrides."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    lib.oracle_merge_i32.argtypes = [_P, _I64, _P, _I64, _P]
    lib.oracle_merge_i32.restype = None
    lib.oracle_merge_u32.argtypes = [_P, _I64, _P, _I64, _P]
    lib.oracle_merge_u32.restype = None
    lib.oracle_merge_f32.argtypes = [_P, _I64, _P, _I64, _P]
    lib.oracle_merge_f32.restype = None
    lib.oracle_merge_keys.argtypes = [ctypes.c_int, ctypes.c_int, _P, _I64, _P, _I64, _P]
    lib.oracle_merge_keys.restype = ctypes.c_int
    lib.oracle_merge_sort_keys.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P, _I64]
    lib.oracle_merge_sort_keys.restype = ctypes.c_int
    lib.oracle_merge_pairs_u32.argtypes = [_P, _P, _I64, _P, _P, _I64, _P, _P]
    lib.oracle_merge_pairs_u32.restype = None
    lib.oracle_corank_pages_i32.argtypes = [_I64, _P, _I64, _P, _I64, _P, _I64, _P]
    lib.oracle_corank_pages_i32.restype = _I64
    lib.oracle_corank_pages_u32.argtypes = [_I64, _P, _I64, _P, _I64]
    lib.oracle_corank_pages_u32.restype = _I64
    lib.oracle_corank_count_i32.argtypes = [_I64, _P, _I64, _P, _I64]
    lib.oracle_corank_count_i32.restype = _I64
    lib.oracle_merge_at_i32.argtypes = [_I64, _P, _I64, _P, _I64, _P]
    lib.oracle_merge_at_i32.restype = ctypes.c_int32
    lib.oracle_merge_sort_pairs_u32.argtypes = [_P, _P, _I64]
    lib.oracle_merge_sort_pairs_u32.restype = ctypes.c_int
    return lib


def _arr(x, dtype):
    a = np.ascontiguousarray(x, dtype=dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def merge_i32(A, B, lib=None) -> np.ndarray:
    """O1: stable merge of sorted int32 arrays (ties take A first)."""
    lib = lib or load()
    A = _arr(A, np.int32)
    B = _arr(B, np.int32)
    C = np.empty(A.size + B.size, dtype=np.int32)
    lib.oracle_merge_i32(_ptr(A), A.size, _ptr(B), B.size, _ptr(C))
    return C


def merge_u32(A, B, lib=None) -> np.ndarray:
    """O1 on uint32 keys (unsigned order)."""
    lib = lib or load()
    A = _arr(A, np.uint32)
    B = _arr(B, np.uint32)
    C = np.empty(A.size + B.size, dtype=np.uint32)
    lib.oracle_merge_u32(_ptr(A), A.size, _ptr(B), B.size, _ptr(C))
    return C


def merge_f32(A, B, lib=None) -> np.ndarray:
    """O1 on float32 keys (float order; keys comparing equal keep A first)."""
    lib = lib or load()
    A = _arr(A, np.float32)
    B = _arr(B, np.float32)
    C = np.empty(A.size + B.size, dtype=np.float32)
    lib.oracle_merge_f32(_ptr(A), A.size, _ptr(B), B.size, _ptr(C))
    return C


# the oracle's key-type codes, by numpy dtype
KEY_CODES = {np.dtype(np.int32): 0, np.dtype(np.uint32): 1, np.dtype(np.float32): 2,
             np.dtype(np.int64): 3, np.dtype(np.uint64): 4, np.dtype(np.float64): 5}


def merge_keys(A, B, descending=False, lib=None) -> np.ndarray:
    """O1 for any of the six key types (taken from A's dtype), either order."""
    lib = lib or load()
    A = np.ascontiguousarray(A)
    dt = A.dtype
    if dt not in KEY_CODES:
        raise ValueError(f"no oracle key type for {dt}")
    B = _arr(B, dt)
    C = np.empty(A.size + B.size, dtype=dt)
    rc = lib.oracle_merge_keys(KEY_CODES[dt], 1 if descending else 0, _ptr(A), A.size, _ptr(B), B.size, _ptr(C))
    if rc != 0:
        raise ValueError("oracle_merge_keys rejected the key type")
    return C


def merge_pairs_u32(keysA, valsA, keysB, valsB, lib=None):
    """O1 on (uint32 key, uint32 value) pairs; compares keys only."""
    lib = lib or load()
    ka, va = _arr(keysA, np.uint32), _arr(valsA, np.uint32)
    kb, vb = _arr(keysB, np.uint32), _arr(valsB, np.uint32)
    assert ka.size == va.size and kb.size == vb.size
    kc = np.empty(ka.size + kb.size, dtype=np.uint32)
    vc = np.empty_like(kc)
    lib.oracle_merge_pairs_u32(_ptr(ka), _ptr(va), ka.size, _ptr(kb), _ptr(vb), kb.size,
                               _ptr(kc), _ptr(vc))
    return kc, vc


def corank_pages(k: int, A, B, trace: bool = False, lib=None):
    """O2: the pages' co-rank loop.  Returns ``i`` (or ``(i, rows)`` with trace).

    ``rows`` is a list of dicts with keys i_low, i, j, j_low, verdict
    ('i too big' / 'j too big' / 'accept') and delta.
    """
    lib = lib or load()
    A = _arr(A, np.int32)
    B = _arr(B, np.int32)
    if not trace:
        return int(lib.oracle_corank_pages_i32(k, _ptr(A), A.size, _ptr(B), B.size, None, 0, None))
    rows = (TraceRow * 200)()
    nrows = ctypes.c_int64(0)
    i = lib.oracle_corank_pages_i32(k, _ptr(A), A.size, _ptr(B), B.size, rows, 200,
                                    ctypes.byref(nrows))
    names = {0: "accept", 1: "i too big", 2: "j too big"}
    out = [
        dict(i_low=r.i_low, i=r.i, j=r.j, j_low=r.j_low, verdict=names[r.verdict], delta=r.delta)
        for r in rows[: nrows.value]
    ]
    return int(i), out


def corank_pages_u32(k: int, A, B, lib=None) -> int:
    """O2 with unsigned compares."""
    lib = lib or load()
    A = _arr(A, np.uint32)
    B = _arr(B, np.uint32)
    return int(lib.oracle_corank_pages_u32(k, _ptr(A), A.size, _ptr(B), B.size))


def corank_count(k: int, A, B, lib=None) -> int:
    """O3: co-rank as the number of A elements among the first k merge outputs."""
    lib = lib or load()
    A = _arr(A, np.int32)
    B = _arr(B, np.int32)
    return int(lib.oracle_corank_count_i32(k, _ptr(A), A.size, _ptr(B), B.size))


def merge_at_i32(k: int, A, B, lib=None):
    """O5: ``(C[k], came_from_A)`` from the co-rank split and one merge step."""
    lib = lib or load()
    A = _arr(A, np.int32)
    B = _arr(B, np.int32)
    flag = ctypes.c_int32(0)
    v = lib.oracle_merge_at_i32(k, _ptr(A), A.size, _ptr(B), B.size, ctypes.byref(flag))
    return int(v), bool(flag.value)


def merge_sort_pairs_u32(keys, vals, lib=None):
    """O4: stable bottom-up merge sort of (key, value) pairs; returns copies."""
    lib = lib or load()
    k = np.array(keys, dtype=np.uint32, copy=True)
    v = np.array(vals, dtype=np.uint32, copy=True)
    assert k.size == v.size
    rc = lib.oracle_merge_sort_pairs_u32(_ptr(k), _ptr(v), k.size)
    if rc != 0:
        raise MemoryError("oracle merge sort could not allocate its scratch")
    return k, v


def merge_sort_keys(keys, vals=None, descending=False, lib=None):
    """O4 for any of the six key types (from keys' dtype), either order;
    optional uint32 values.  Returns sorted copies (keys, vals or None)."""
    lib = lib or load()
    k = np.array(keys, copy=True)
    if k.dtype not in KEY_CODES:
        raise ValueError(f"no oracle key type for {k.dtype}")
    v = None if vals is None else np.array(vals, dtype=np.uint32, copy=True)
    assert v is None or v.size == k.size
    rc = lib.oracle_merge_sort_keys(KEY_CODES[k.dtype], 1 if descending else 0, _ptr(k),
                                    None if v is None else _ptr(v), k.size)
    if rc == -2:
        raise MemoryError("oracle merge sort could not allocate its scratch")
    if rc != 0:
        raise ValueError("oracle_merge_sort_keys rejected the key type")
    return k, v

"""Python binding of libordmerge.so, the GB300 stable co-rank merge library.

Argument marshalling only: every function checks tensors, takes their device
pointers and the current CUDA stream, and calls the C ABI declared in
``include/ordmerge.h`` through ctypes.  All computation runs in the library's
CUDA kernels; there is no CPU path.  PyTorch is used for device memory and
streams.

Import fails loudly if the library has not been built
(``python -m ordered_merge_gb300.build`` or ``__graft_entry__.build()``).

Functions carry the C names (``om_merge_i32`` ...) with unprefixed aliases
(``merge_i32`` ...).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

OM_OK, OM_EINVAL, OM_ERANGE, OM_ENOMEM, OM_ECUDA, OM_EDEVICE = range(6)

KIND_PARTITION, KIND_TILE_MERGE, KIND_BLOCK_SORT, KIND_CORANK, KIND_BASELINE, KIND_ONE_PASS = range(6)

# om_key_type codes and their element sizes
KEY_TYPES = {"i32": (0, 4), "u32": (1, 4), "f32": (2, 4), "i64": (3, 8), "u64": (4, 8), "f64": (5, 8)}
OM_ASCENDING, OM_DESCENDING = 0, 1


class OrdMergeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)} ({status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m ordered_merge_gb300.build` "
            "(the merge has no CPU fallback)"
        )
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.om_corank_i32.argtypes = [I64, P, I64, P, I64]
    lib.om_corank_i32.restype = I64
    lib.om_corank_i32_batch.argtypes = [P, I64, P, I64, P, I64, P, P]
    lib.om_corank_i32_batch.restype = I32
    lib.om_partition_i32.argtypes = [P, I64, P, I64, I64, I64, P, P]
    lib.om_partition_i32.restype = I32
    lib.om_merge_i32.argtypes = [P, I64, P, I64, P, P]
    lib.om_merge_i32.restype = I32
    lib.om_merge_i32_noalloc.argtypes = [P, I64, P, I64, P, P]
    lib.om_merge_i32_noalloc.restype = I32
    lib.om_merge_pairs_u32.argtypes = [P, P, I64, P, P, I64, P, P, P]
    lib.om_merge_pairs_u32.restype = I32
    lib.om_merge_sort_u32.argtypes = [P, P, I64, P]
    lib.om_merge_sort_u32.restype = I32
    lib.om_status_string.argtypes = [I32]
    lib.om_status_string.restype = ctypes.c_char_p
    lib.om_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.om_device_error.restype = I32
    lib.om_trace_enable.argtypes = [I32]
    lib.om_trace_enable.restype = I32
    lib.om_trace_reset.argtypes = []
    lib.om_trace_reset.restype = I32
    lib.om_trace_read.argtypes = [I32, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)]
    lib.om_trace_read.restype = I32
    lib.om_merge_keys.argtypes = [I32, I32, P, I64, P, I64, P, P]
    lib.om_merge_keys.restype = I32
    lib.om_merge_sort_keys.argtypes = [I32, I32, P, P, I64, P]
    lib.om_merge_sort_keys.restype = I32
    lib.om_merge_i32_one_thread.argtypes = [P, I64, P, I64, P, P]
    lib.om_merge_i32_one_thread.restype = I32
    lib.om_merge_i32_slices.argtypes = [P, I64, P, I64, P, I64, P]
    lib.om_merge_i32_slices.restype = I32
    lib.om_release_scratch.argtypes = []
    lib.om_release_scratch.restype = I32
    lib.om_launch_count.argtypes = []
    lib.om_launch_count.restype = ctypes.c_uint64
    lib.om_subtiles_per_range.argtypes = [I64, I64, I64, I64, I64]
    lib.om_subtiles_per_range.restype = I64
    return lib


_lib = _load()


def lib():
    """The ctypes handle of libordmerge.so (for direct C-ABI calls)."""
    return _lib


def _status_string(status: int) -> str:
    return _lib.om_status_string(status).decode()


def _check(status: int, what: str):
    if status != OM_OK:
        raise OrdMergeError(status, what)


def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _on_current_device(t, name: str):
    """The library launches on the current CUDA device: a tensor elsewhere
    would hand that device's addresses to its kernels."""
    import torch

    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")


def _ptr4(t, name: str):
    """Device pointer of a contiguous CUDA tensor of 4-byte elements."""
    _on_current_device(t, name)
    if t.element_size() != 4:
        raise ValueError(f"{name} must have 4-byte elements (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() if t.numel() else None


def om_corank_i32(k: int, A, B) -> int:
    """co_rank(k) of int32 device tensors A, B (synchronous); j = k - i."""
    r = _lib.om_corank_i32(int(k), _ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel())
    if r < 0:
        raise OrdMergeError(int(-r), "om_corank_i32")
    return int(r)


def om_corank_i32_batch(ks, A, B, out=None, stream=None):
    """i[t] = co_rank(ks[t]) for an int64 device tensor ks (asynchronous)."""
    import torch

    if ks.dtype != torch.int64 or not ks.is_cuda or not ks.is_contiguous():
        raise ValueError("ks must be a contiguous int64 CUDA tensor")
    _on_current_device(ks, "ks")
    if out is None:
        out = torch.empty_like(ks)
    if out.dtype != torch.int64 or out.numel() != ks.numel() or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 tensor as long as ks")
    _on_current_device(out, "out")
    _check(
        _lib.om_corank_i32_batch(ks.data_ptr() if ks.numel() else None, ks.numel(), _ptr4(A, "A"), A.numel(),
                                 _ptr4(B, "B"), B.numel(), out.data_ptr() if out.numel() else None,
                                 _stream(stream)),
        "om_corank_i32_batch",
    )
    return out


def om_partition_i32(A, B, tile: int, count: int | None = None, out=None, stream=None):
    """split[t] = co_rank(min(t * tile, len(A) + len(B))) for t < count
    (default: one per tile boundary, ceil((m + n) / tile) + 1), by the
    partition kernel (asynchronous); j_t = min(t * tile, m + n) - split[t]."""
    import torch

    total = A.numel() + B.numel()
    if count is None:
        count = (total + tile - 1) // tile + 1 if tile > 0 else 0
    if out is None:
        out = torch.empty(count, dtype=torch.int64, device=A.device)
    if out.dtype != torch.int64 or out.numel() != count or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 tensor of count elements")
    _on_current_device(out, "out")
    _check(
        _lib.om_partition_i32(_ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel(), int(tile), int(count),
                              out.data_ptr() if out.numel() else None, _stream(stream)),
        "om_partition_i32",
    )
    return out


def om_merge_i32(A, B, C=None, stream=None):
    """C = stable merge of sorted int32 device tensors A and B (ties: A first)."""
    import torch

    if C is None:
        C = torch.empty(A.numel() + B.numel(), dtype=torch.int32, device=A.device)
    if C.numel() != A.numel() + B.numel():
        raise ValueError("C must hold len(A) + len(B) elements")
    _check(
        _lib.om_merge_i32(_ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel(), _ptr4(C, "C"), _stream(stream)),
        "om_merge_i32",
    )
    return C


def om_merge_i32_noalloc(A, B, C=None, stream=None):
    """om_merge_i32 through the entry point that allocates nothing on the
    device (splitters in the library's fixed array; m + n <= 2^30)."""
    import torch

    if C is None:
        C = torch.empty(A.numel() + B.numel(), dtype=torch.int32, device=A.device)
    if C.numel() != A.numel() + B.numel():
        raise ValueError("C must hold len(A) + len(B) elements")
    _check(
        _lib.om_merge_i32_noalloc(_ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel(), _ptr4(C, "C"),
                                  _stream(stream)),
        "om_merge_i32_noalloc",
    )
    return C


def _key_type_of(dtype) -> str:
    import torch

    names = {torch.int32: "i32", torch.float32: "f32", torch.int64: "i64", torch.float64: "f64"}
    for extra, name in (("uint32", "u32"), ("uint64", "u64")):
        if hasattr(torch, extra):
            names[getattr(torch, extra)] = name
    if dtype not in names:
        raise ValueError(f"no key type for {dtype}; pass key_type")
    return names[dtype]


def _ptr_sized(t, name: str, size: int):
    """Device pointer of a contiguous CUDA tensor of `size`-byte elements."""
    _on_current_device(t, name)
    if t.element_size() != size:
        raise ValueError(f"{name} must have {size}-byte elements (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() if t.numel() else None


def om_merge_keys(A, B, C=None, key_type=None, descending=False, stream=None):
    """C = stable merge of sorted device tensors A and B (ties: A first).

    key_type: "i32", "u32", "f32", "i64", "u64" or "f64" (default: from
    A's dtype); the tensors' bits are read as that type, so an int32 tensor
    can carry uint32 keys.  descending: inputs and output nonincreasing.
    """
    import torch

    name = key_type or _key_type_of(A.dtype)
    if name not in KEY_TYPES:
        raise ValueError(f"unknown key type {name!r}")
    code, size = KEY_TYPES[name]
    if C is None:
        C = torch.empty(A.numel() + B.numel(), dtype=A.dtype, device=A.device)
    if C.numel() != A.numel() + B.numel():
        raise ValueError("C must hold len(A) + len(B) elements")
    _check(
        _lib.om_merge_keys(code, OM_DESCENDING if descending else OM_ASCENDING, _ptr_sized(A, "A", size),
                           A.numel(), _ptr_sized(B, "B", size), B.numel(), _ptr_sized(C, "C", size),
                           _stream(stream)),
        "om_merge_keys",
    )
    return C


def om_merge_sort_keys(keys, vals=None, key_type=None, descending=False, stream=None):
    """Stable in-place sort of a device tensor of keys (type from its dtype
    or `key_type`), nondecreasing or (descending) nonincreasing, carrying
    optional 4-byte values (4-byte keys only)."""
    name = key_type or _key_type_of(keys.dtype)
    if name not in KEY_TYPES:
        raise ValueError(f"unknown key type {name!r}")
    code, size = KEY_TYPES[name]
    n = keys.numel()
    if vals is not None and vals.numel() != n:
        raise ValueError("vals must have as many elements as keys")
    _check(
        _lib.om_merge_sort_keys(code, OM_DESCENDING if descending else OM_ASCENDING, _ptr_sized(keys, "keys", size),
                                _ptr4(vals, "vals") if vals is not None else None, n, _stream(stream)),
        "om_merge_sort_keys",
    )
    return keys, vals


def om_merge_i32_one_thread(A, B, C=None, stream=None):
    """The two-pointer merge in one device thread (comparison only)."""
    import torch

    if C is None:
        C = torch.empty(A.numel() + B.numel(), dtype=torch.int32, device=A.device)
    if C.numel() != A.numel() + B.numel():
        raise ValueError("C must hold len(A) + len(B) elements")
    _check(_lib.om_merge_i32_one_thread(_ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel(), _ptr4(C, "C"),
                                        _stream(stream)), "om_merge_i32_one_thread")
    return C


def om_merge_i32_slices(A, B, C=None, per_thread=1, stream=None):
    """One thread per slice of `per_thread` outputs, no shared memory
    (comparison only)."""
    import torch

    if C is None:
        C = torch.empty(A.numel() + B.numel(), dtype=torch.int32, device=A.device)
    if C.numel() != A.numel() + B.numel():
        raise ValueError("C must hold len(A) + len(B) elements")
    _check(_lib.om_merge_i32_slices(_ptr4(A, "A"), A.numel(), _ptr4(B, "B"), B.numel(), _ptr4(C, "C"),
                                    int(per_thread), _stream(stream)), "om_merge_i32_slices")
    return C


def om_merge_pairs_u32(keysA, valsA, keysB, valsB, keysC=None, valsC=None, stream=None):
    """Stable merge of (uint32 key, uint32 value) pairs; keys compared unsigned.

    uint32 data may be carried in int32 tensors (bits are reinterpreted).
    """
    import torch

    m, n = keysA.numel(), keysB.numel()
    if valsA.numel() != m or valsB.numel() != n:
        raise ValueError("each value array must match its key array")
    if keysC is None:
        keysC = torch.empty(m + n, dtype=keysA.dtype, device=keysA.device)
    if valsC is None:
        valsC = torch.empty(m + n, dtype=valsA.dtype, device=valsA.device)
    if keysC.numel() != m + n or valsC.numel() != m + n:
        raise ValueError("outputs must hold len(A) + len(B) elements")
    _check(
        _lib.om_merge_pairs_u32(_ptr4(keysA, "keysA"), _ptr4(valsA, "valsA"), m, _ptr4(keysB, "keysB"),
                                _ptr4(valsB, "valsB"), n, _ptr4(keysC, "keysC"), _ptr4(valsC, "valsC"),
                                _stream(stream)),
        "om_merge_pairs_u32",
    )
    return keysC, valsC


def om_merge_sort_u32(keys, vals=None, stream=None):
    """Stable in-place sort of uint32 keys (unsigned order), carrying vals."""
    n = keys.numel()
    if vals is not None and vals.numel() != n:
        raise ValueError("vals must match keys")
    _check(
        _lib.om_merge_sort_u32(_ptr4(keys, "keys"), _ptr4(vals, "vals") if vals is not None else None, n,
                               _stream(stream)),
        "om_merge_sort_u32",
    )
    return keys, vals


def om_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    w = ctypes.c_uint32(0)
    st = _lib.om_device_error(_stream(stream), ctypes.byref(w))
    if st not in (OM_OK, OM_EDEVICE):
        raise OrdMergeError(st, "om_device_error")
    return int(w.value)


def om_trace_enable(on: bool = True):
    _check(_lib.om_trace_enable(1 if on else 0), "om_trace_enable")


def om_trace_reset():
    _check(_lib.om_trace_reset(), "om_trace_reset")


def om_trace_read(kind: int):
    """(launches, total_ms) of one kernel kind since the last reset."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(_lib.om_trace_read(kind, ctypes.byref(n), ctypes.byref(ms)), "om_trace_read")
    return int(n.value), float(ms.value)


def om_release_scratch():
    """Return the library's cached scratch on the current device to the system."""
    _check(_lib.om_release_scratch(), "om_release_scratch")


def om_launch_count() -> int:
    return int(_lib.om_launch_count())


def om_subtiles_per_range(segs: int, seg_len: int, subtile: int, bytes_per_output: int, resident_ctas: int) -> int:
    """Sub-tiles per CTA output range the library picks for one launch (host only)."""
    return int(_lib.om_subtiles_per_range(segs, seg_len, subtile, bytes_per_output, resident_ctas))


corank_i32 = om_corank_i32
corank_i32_batch = om_corank_i32_batch
merge_i32 = om_merge_i32
partition_i32 = om_partition_i32
merge_i32_noalloc = om_merge_i32_noalloc
merge_pairs_u32 = om_merge_pairs_u32
merge_keys = om_merge_keys
merge_sort_keys = om_merge_sort_keys
merge_i32_one_thread = om_merge_i32_one_thread
merge_i32_slices = om_merge_i32_slices
merge_sort_u32 = om_merge_sort_u32
device_error = om_device_error
release_scratch = om_release_scratch

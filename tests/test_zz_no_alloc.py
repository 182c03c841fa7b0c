"""om_merge_i32_noalloc: the merge for callers that cannot allocate device
memory on the call path (for example a process whose device memory is fully
reserved by another allocator, or code that must not enter an allocator).

Called directly through the C ABI (ctypes, device pointers, the current
stream) and compared with om_merge_i32 and with the CPU oracle on the same
inputs, on calls in a row with different sizes, so each later call runs on
the splitter array the call before left behind.  The inputs include heavy
ties and one-sided merges, so range boundaries (the partition kernel's
splitters) fall inside runs of equal keys and at the ends of a side.  The
file is named to be collected last; it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import host

pytestmark = pytest.mark.gpu


def _noalloc(om):
    lib = om.lib()
    f = lib.om_merge_i32_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _inputs(seed, m, n, span):
    rng = np.random.default_rng(seed)
    A = np.sort(rng.integers(-span, span, m)).astype(np.int32)
    B = np.sort(rng.integers(-span, span, n)).astype(np.int32)
    return torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()


def _one_sided(seed, m, n, a_first):
    rng = np.random.default_rng(seed)
    lo, hi = (np.sort(rng.integers(-1000, 0, m)), np.sort(rng.integers(0, 1000, n)))
    A, B = (lo, hi) if a_first else (hi + 1, lo - 1000)
    return torch.from_numpy(A.astype(np.int32)).cuda(), torch.from_numpy(B.astype(np.int32)).cuda()


CALLS = [
    ("uniform", lambda: _inputs(100, 3_000_001, 2_999_999, 1 << 30)),
    ("heavy_ties", lambda: _inputs(101, 700_003, 1_200_007, 3)),
    ("all_A_first", lambda: _one_sided(102, 1_500_000, 900_001, True)),
    ("all_B_first", lambda: _one_sided(103, 400_007, 2_100_000, False)),
]


def test_noalloc_matches_merge_i32_and_oracle(gpu):
    f = _noalloc(gpu)
    stream = torch.cuda.current_stream().cuda_stream
    for name, make in CALLS:
        A, B = make()
        m, n = A.numel(), B.numel()
        want = gpu.merge_i32(A, B)  # the existing entry point
        got = torch.full((m + n,), -7, dtype=torch.int32, device="cuda")
        st = f(A.data_ptr(), m, B.data_ptr(), n, got.data_ptr(), stream)
        assert st == gpu.OM_OK, gpu.lib().om_status_string(st)
        torch.cuda.synchronize()
        assert gpu.device_error() == 0
        assert torch.equal(got, want), f"{name}: differs from om_merge_i32"
        assert np.array_equal(host(got), oracle.merge_i32(host(A), host(B))), f"{name}: differs from the oracle"


def test_noalloc_large_merge_and_limit(gpu):
    f = _noalloc(gpu)
    stream = torch.cuda.current_stream().cuda_stream
    # 2^28 outputs: thousands of output ranges, all splitters in the fixed array
    m = n = 1 << 27
    A, B = _inputs(7, m, n, 1 << 31)
    want = gpu.merge_i32(A, B)
    got = torch.empty_like(want)
    assert f(A.data_ptr(), m, B.data_ptr(), n, got.data_ptr(), stream) == gpu.OM_OK
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    # beyond the array's capacity: rejected before anything is launched
    too_many = (1 << 30) + 1
    assert f(A.data_ptr(), too_many - 5, B.data_ptr(), 5, got.data_ptr(), stream) == gpu.OM_ERANGE

"""om_merge_i32_noalloc: the merge for callers that cannot allocate device
memory on the call path (for example a process whose device memory is fully
reserved by another allocator, or code that must not enter an allocator).

Called directly through the C ABI (ctypes, device pointers, the current
stream) and compared with om_merge_i32 on the same inputs, on two calls in a
row with different sizes, so the second call runs on the splitter array the
first call left behind.  The file is named to be collected last; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def test_noalloc_matches_merge_i32_two_calls(gpu):
    f = _noalloc(gpu)
    stream = torch.cuda.current_stream().cuda_stream
    for call, (m, n, span) in enumerate([(3_000_001, 2_999_999, 1 << 30), (700_003, 1_200_007, 50)]):
        A, B = _inputs(100 + call, m, n, span)
        want = gpu.merge_i32(A, B)  # the existing entry point
        got = torch.full((m + n,), -7, dtype=torch.int32, device="cuda")
        st = f(A.data_ptr(), m, B.data_ptr(), n, got.data_ptr(), stream)
        assert st == gpu.OM_OK, gpu.lib().om_status_string(st)
        torch.cuda.synchronize()
        assert gpu.device_error() == 0
        assert torch.equal(got, want), f"call {call}: differs from om_merge_i32"


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
    too_many = 1_006_510_080 + 1
    assert f(A.data_ptr(), too_many - 5, B.data_ptr(), 5, got.data_ptr(), stream) == gpu.OM_ERANGE

"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
function include/ordmerge.h declares, and rejects bad arguments on the host
before touching the device (no compute calls: these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ordmerge.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    path = __graft_entry__._lib_build_module().build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(om_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for required in ["om_corank_i32", "om_merge_i32", "om_merge_pairs_u32", "om_merge_sort_u32"]:
        assert required in names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(lib):
    import ordered_merge_gb300 as om

    for s in range(6):
        assert om.lib().om_status_string(s).decode().startswith("OM_")


def test_host_argument_checks():
    """Invalid arguments are rejected by host code with a status, not a crash,
    and never reach the GPU."""
    import ordered_merge_gb300 as om

    L = om.lib()
    # negative lengths
    assert L.om_merge_i32(None, -1, None, 0, None, None) == om.OM_EINVAL
    assert L.om_merge_pairs_u32(None, None, 0, None, None, -5, None, None, None) == om.OM_EINVAL
    assert L.om_merge_sort_u32(None, None, -2, None) == om.OM_EINVAL
    # empty merge / trivial sort are no-ops
    assert L.om_merge_i32(None, 0, None, 0, None, None) == om.OM_OK
    assert L.om_merge_sort_u32(None, None, 1, None) == om.OM_OK
    # NULL with a nonzero length
    assert L.om_merge_i32(None, 4, 0x1000, 4, 0x2000, None) == om.OM_EINVAL
    assert L.om_merge_i32(0x1000, 4, 0x2000, 4, None, None) == om.OM_EINVAL
    # misaligned pointers
    assert L.om_merge_i32(0x1002, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    # output overlapping an input
    assert L.om_merge_i32(0x1000, 4, 0x2000, 4, 0x1008, None) == om.OM_EINVAL
    assert L.om_merge_i32(0x1000, 4, 0x2000, 4, 0x1FF0, None) == om.OM_EINVAL
    # m + n overflow
    assert L.om_merge_i32(0x1000, 2**62, 0x2000, 2**62, 0x3000, None) == om.OM_ERANGE
    # pairs: key/value 16-byte phase mismatch
    assert L.om_merge_pairs_u32(0x1000, 0x2004, 4, 0x3000, 0x4000, 4, 0x5000, 0x6000, None) == om.OM_EINVAL
    # sort: vals overlapping keys
    assert L.om_merge_sort_u32(0x1000, 0x1008, 16, None) == om.OM_EINVAL
    # co-rank: k outside [0, m+n], negative length
    assert L.om_corank_i32(11, 0x1000, 5, 0x2000, 5) == -om.OM_ERANGE
    assert L.om_corank_i32(-1, 0x1000, 5, 0x2000, 5) == -om.OM_ERANGE
    assert L.om_corank_i32(0, 0x1000, -5, 0x2000, 5) == -om.OM_EINVAL
    # co-rank with one side empty is forced and needs no device
    assert L.om_corank_i32(3, None, 0, 0x2000, 5) == 0
    assert L.om_corank_i32(3, 0x1000, 5, None, 0) == 3


def test_merge_keys_host_argument_checks():
    """om_merge_keys: unknown type or order, alignment to the key size and
    overlap in key-size units are rejected on the host."""
    import ordered_merge_gb300 as om

    L = om.lib()
    i64, f32 = om.KEY_TYPES["i64"][0], om.KEY_TYPES["f32"][0]
    assert L.om_merge_keys(6, 0, 0x1000, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_keys(-1, 0, 0x1000, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_keys(f32, 2, 0x1000, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_keys(f32, 0, None, 0, None, 0, None, None) == om.OM_OK
    assert L.om_merge_keys(f32, 0, None, -1, None, 0, None, None) == om.OM_EINVAL
    assert L.om_merge_keys(f32, 0, 0x1000, 2**62, 0x2000, 2**62, 0x3000, None) == om.OM_ERANGE
    # 8-byte keys need 8-byte alignment; 4 is not enough
    assert L.om_merge_keys(i64, 0, 0x1004, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_keys(i64, 1, 0x1000, 4, 0x2000, 4, 0x300C, None) == om.OM_EINVAL
    assert L.om_merge_keys(f32, 0, 0x1002, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    # overlap counts 8 bytes per element: C = [0x2000, 0x2040) meets B at 0x2020
    assert L.om_merge_keys(i64, 0, 0x1000, 4, 0x2020, 4, 0x2000, None) == om.OM_EINVAL
    assert L.om_merge_keys(i64, 0, None, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL


def test_merge_sort_keys_host_argument_checks():
    import ordered_merge_gb300 as om

    L = om.lib()
    i64, f32 = om.KEY_TYPES["i64"][0], om.KEY_TYPES["f32"][0]
    assert L.om_merge_sort_keys(9, 0, 0x1000, None, 16, None) == om.OM_EINVAL
    assert L.om_merge_sort_keys(f32, 3, 0x1000, None, 16, None) == om.OM_EINVAL
    assert L.om_merge_sort_keys(f32, 0, None, None, 1, None) == om.OM_OK       # trivial
    assert L.om_merge_sort_keys(f32, 0, None, None, -1, None) == om.OM_EINVAL
    assert L.om_merge_sort_keys(f32, 0, None, None, 16, None) == om.OM_EINVAL
    assert L.om_merge_sort_keys(i64, 0, 0x1004, None, 16, None) == om.OM_EINVAL  # 8-byte alignment
    assert L.om_merge_sort_keys(i64, 0, 0x1000, 0x9000, 16, None) == om.OM_EINVAL  # no values with 8-byte keys
    assert L.om_merge_sort_keys(f32, 0, 0x1000, 0x2004, 16, None) == om.OM_EINVAL  # 16-byte phase differs
    assert L.om_merge_sort_keys(f32, 1, 0x1000, 0x1010, 16, None) == om.OM_EINVAL  # overlap
    assert L.om_merge_sort_keys(f32, 0, 0x1000, None, (1 << 40) + 1, None) == om.OM_ERANGE


def test_comparison_merges_host_argument_checks():
    import ordered_merge_gb300 as om

    L = om.lib()
    assert L.om_merge_i32_slices(0x1000, 4, 0x2000, 4, 0x3000, 0, None) == om.OM_EINVAL   # per_thread < 1
    assert L.om_merge_i32_slices(0x1000, -1, 0x2000, 4, 0x3000, 4, None) == om.OM_EINVAL
    assert L.om_merge_i32_slices(None, 0, None, 0, None, 4, None) == om.OM_OK
    assert L.om_merge_i32_slices(0x1000, 4, 0x2000, 4, 0x1008, 4, None) == om.OM_EINVAL  # overlap
    assert L.om_merge_i32_one_thread(0x1002, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL  # misaligned
    assert L.om_merge_i32_one_thread(None, 0, None, 0, None, None) == om.OM_OK
    assert L.om_merge_i32_one_thread(0x1000, 2**62, 0x2000, 2**62, 0x3000, None) == om.OM_ERANGE


def test_partition_and_noalloc_host_argument_checks():
    import ordered_merge_gb300 as om

    L = om.lib()
    # partition: tile < 1, negative count or length, NULL or misaligned split, overlap with an input
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 0, 3, 0x3000, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 4, -1, 0x3000, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, -4, 0x2000, 4, 4, 3, 0x3000, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 4, 0, None, None) == om.OM_OK  # nothing to do
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 4, 3, None, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 4, 3, 0x3004, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 4, 3, 0x1008, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1002, 4, 0x2000, 4, 4, 3, 0x3000, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 2**62, 0x2000, 2**62, 4, 3, 0x3000, None) == om.OM_ERANGE
    # no-alloc merge: the same rules as om_merge_i32, and the fixed size limit
    assert L.om_merge_i32_noalloc(None, 0, None, 0, None, None) == om.OM_OK
    assert L.om_merge_i32_noalloc(0x1000, -1, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_i32_noalloc(0x1002, 4, 0x2000, 4, 0x3000, None) == om.OM_EINVAL
    assert L.om_merge_i32_noalloc(0x1000, 4, 0x2000, 4, 0x1008, None) == om.OM_EINVAL
    assert L.om_merge_i32_noalloc(0x1000, (1 << 30) - 4, 0x2000, 5, 0x3000, None) == om.OM_ERANGE


def test_partition_split_next_to_inputs_is_not_overlap():
    """The split array is counted in 8-byte elements and the inputs in 4-byte
    ones: a split array that starts right after A or B does not overlap them.
    A count too large for one launch makes the call stop with OM_ERANGE just
    after the overlap check, so nothing reaches a device."""
    import ordered_merge_gb300 as om

    L = om.lib()
    huge = 1 << 36
    # A = [0x1000, 0x1010) and B = [0x100, 0x110) below the split array
    assert L.om_partition_i32(0x1000, 4, 0x100, 4, 2, huge, 0x1010, None) == om.OM_ERANGE
    # B = [0x2000, 0x2010) and A below: split starting at B's end
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 2, huge, 0x2010, None) == om.OM_ERANGE
    # starting inside B, or covering A: rejected as overlap
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 2, huge, 0x2008, None) == om.OM_EINVAL
    assert L.om_partition_i32(0x1000, 4, 0x2000, 4, 2, 3, 0x0FF8, None) == om.OM_EINVAL

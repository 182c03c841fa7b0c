"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks
that the pins in test_oracle_pins.py catch every one of them.

Each mutant is a one-token edit of oracle/merge_oracle.c: a flipped tie rule,
a floor instead of a ceiling step, mirrored search bounds, a dropped tail
copy, swapped run order in the sort.  A mutant that no pin catches would mean
the pins cannot tell that mistake from the right answer.
"""
import os
import subprocess
import sys

import pytest

import oracle
from test_oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "merge_oracle.c")

# Not listed: a floor step in the "j too big" branch.  On sorted input that
# branch always sees j - j_low >= 2 (j_low is only ever set by an "i too big"
# step, which puts it strictly below the answer's j, or starts at max(0, k-m)
# where that branch cannot fire), so the floor never stalls and the mutant is
# equivalent: no input can tell it apart.  An exhaustive search over all
# sorted inputs of total length <= 8 on a 4-letter alphabet agreed.
#
# Not listed either: taking B first on a tie in the keys-only uint32 merge.
# Equal uint32 keys are the same bits, so the output cannot show which side
# went first; the float merge's tie rule is pinned instead, through -0.0 and
# +0.0, which compare equal but differ in bits.
#
# (name, exact text in the oracle, replacement, occurrence index to replace)
MUTANTS = [
    ("pairs_ties_take_B_first", "if (keysB[j] < keysA[i]) {", "if (keysB[j] <= keysA[i]) {", 0),
    ("merge_drops_B_tail", "    while (j < n) C[k++] = B[j++];\n", "\n", 0),
    ("merge_drops_A_tail", "    while (i < m) C[k++] = A[i++];\n", "\n", 0),
    ("corank_floor_step", "delta = (i - i_low + 1) >> 1;", "delta = (i - i_low) >> 1;", 0),
    ("corank_symmetric_test", "B[j - 1] >= A[i]) {\n            verdict = 2;", "B[j - 1] > A[i]) {\n            verdict = 2;", 0),
    ("corank_mirrored_low_bound", "int64_t i_low = (k - n > 0) ? k - n : 0;", "int64_t i_low = (k - m > 0) ? k - m : 0;", 0),
    ("corank_start_low", "int64_t i = (k < m) ? k : m;\n    int64_t j = k - i;\n    int64_t i_low", "int64_t i = 0;\n    int64_t j = k - i;\n    int64_t i_low", 0),
    ("count_corank_B_first_on_tie", "if (i < m && (j >= n || A[i] <= B[j])) {", "if (i < m && (j >= n || A[i] < B[j])) {", 0),
    ("merge_at_B_first_on_tie", "int take_a = (i < m) && (j >= n || A[i] <= B[j]);", "int take_a = (i < m) && (j >= n || A[i] < B[j]);", 0),
    ("sort_later_run_first", "oracle_merge_pairs_u32(src_k + lo, src_v + lo, mid - lo,\n                                   src_k + mid, src_v + mid, hi - mid,",
     "oracle_merge_pairs_u32(src_k + mid, src_v + mid, hi - mid,\n                                   src_k + lo, src_v + lo, mid - lo,", 0),
    ("u32_signed_compare", "void oracle_merge_u32(const uint32_t *A, int64_t m, const uint32_t *B,",
     "void oracle_merge_u32(const int32_t *A, int64_t m, const int32_t *B,", 0),
    ("f32_B_first_on_tie", "if (B[j] < A[i]) {", "if (B[j] <= A[i]) {", 2),
    ("f32_drops_B_tail", "    while (j < n) C[k++] = B[j++];\n", "\n", 2),
    ("keys_i64_unsigned_compare", "        int64_t x = ((const int64_t *)A)[i], y = ((const int64_t *)B)[j];",
     "        uint64_t x = ((const int64_t *)A)[i], y = ((const int64_t *)B)[j];", 0),
    ("keys_u64_signed_compare", "        uint64_t x = ((const uint64_t *)A)[i], y = ((const uint64_t *)B)[j];",
     "        int64_t x = ((const uint64_t *)A)[i], y = ((const uint64_t *)B)[j];", 0),
    ("keys_f64_compared_as_bits", "        double x = ((const double *)A)[i], y = ((const double *)B)[j];",
     "        int64_t x = ((const int64_t *)A)[i], y = ((const int64_t *)B)[j];", 0),
    ("keys_f32_desc_B_first_on_tie", "return desc ? (y > x) : (y < x);", "return desc ? (y >= x) : (y < x);", 2),
    ("keys_f64_desc_B_first_on_tie", "return desc ? (y > x) : (y < x);", "return desc ? (y >= x) : (y < x);", 5),
    ("keys_i32_desc_reversed", "return desc ? (y > x) : (y < x);", "return desc ? (y < x) : (y < x);", 0),
    ("keys_drops_B_tail", "    for (; j < n; ++j, ++k) {\n        memcpy(c + (size_t)k * e, b + (size_t)j * e, e);\n        if (vc != NULL) vc[k] = vb[j];\n    }\n", "\n", 0),
    ("sort_keys_later_run_first",
     "src_k + (size_t)lo * e, src_v ? src_v + lo : NULL, mid - lo,\n                                   src_k + (size_t)mid * e, src_v ? src_v + mid : NULL, hi - mid,",
     "src_k + (size_t)mid * e, src_v ? src_v + mid : NULL, hi - mid,\n                                   src_k + (size_t)lo * e, src_v ? src_v + lo : NULL, mid - lo,", 0),
    ("sort_keys_drops_B_values", "        if (vc != NULL) vc[k] = vb[j];\n    }", "    }", 0),
    ("sort_keys_stops_one_pass_early", "for (int64_t width = 1; width < n; width *= 2) {", "for (int64_t width = 2; width < n; width *= 2) {", 1),
    ("sort_stops_one_pass_early", "for (int64_t width = 1; width < n; width *= 2) {", "for (int64_t width = 2; width < n; width *= 2) {", 0),
    ("corank_u32_signed_compare",
     "int64_t oracle_corank_pages_u32(int64_t k, const uint32_t *A, int64_t m,\n                                const uint32_t *B, int64_t n)",
     "int64_t oracle_corank_pages_u32(int64_t k, const int32_t *A, int64_t m,\n                                const int32_t *B, int64_t n)", 0),
    ("corank_u32_symmetric_test", "B[j - 1] >= A[i]) {\n            int64_t delta", "B[j - 1] > A[i]) {\n            int64_t delta", 0),
    ("corank_u32_i_too_big_on_tie", "A[i - 1] > B[j]) {\n            int64_t delta", "A[i - 1] >= B[j]) {\n            int64_t delta", 0),
    ("corank_u32_floor_step", "int64_t delta = (i - i_low + 1) >> 1;", "int64_t delta = (i - i_low) >> 1;", 0),
]


def _build_mutant(tmp_path, name, old, new, occ=0):
    src = open(SRC).read()
    assert src.count(old) > occ, f"mutation site for {name} not found in the oracle"
    at = -1
    for _ in range(occ + 1):
        at = src.index(old, at + 1)
    mutated = src[:at] + new + src[at + len(old):]
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c)])
    return str(so)


_RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
from test_oracle_pins import ALL_CHECKS
lib = oracle.load({so!r})
caught = []
for check in ALL_CHECKS:
    try:
        if check.__name__ == "check_brute_force":
            check(lib, max_len=4)
        elif check.__name__ == "check_typed_keys":
            check(lib, max_len=3)
        elif check.__name__ == "check_merge_keys":
            check(lib, max_len=3, limit=25)
        elif check.__name__ == "check_merge_sort_keys":
            check(lib, max_len=4)
        else:
            check(lib)
    except Exception:
        caught.append(check.__name__)
print("CAUGHT", ",".join(caught))
"""


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, occ):
    so = _build_mutant(tmp_path, name, old, new, occ)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests_dir), tests=tests_dir, so=so)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        return  # the mutant crashed the checks: caught
    line = [l for l in proc.stdout.splitlines() if l.startswith("CAUGHT")][-1]
    caught = [c for c in line[len("CAUGHT"):].strip().split(",") if c]
    assert caught, f"no pin caught mutant {name}"

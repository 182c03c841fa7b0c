"""Pins for the CPU oracle (CPU only, no GPU).

Each check ties an oracle routine to something other than itself: the pages'
worked example and trace, a hand-derived tie case, closed forms of the
evens/odds and heavy-tie workloads, brute force over every tiny sorted input,
and Python's guaranteed-stable ``sorted`` / numpy's stable argsort as library
routines.  ``test_oracle_mutants.py`` plants mistakes in a copy of the oracle
and checks that these pins catch each one.

The check functions take the oracle library handle so the mutant test can run
them against a mutated build.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- checks --

def check_worked_example(lib):
    """Co-rank page: trace table, three-thread splits, thread-1 slice."""
    rows = _read_golden("corank_trace_example.txt")
    A = [int(x) for x in next(r for r in rows if r[0] == "A")[1:]]
    B = [int(x) for x in next(r for r in rows if r[0] == "B")[1:]]
    k = int(next(r for r in rows if r[0] == "k")[1])
    want_i, want_j = (int(x) for x in next(r for r in rows if r[0] == "result")[1:])
    i, trace = oracle.corank_pages(k, A, B, trace=True, lib=lib)
    assert (i, k - i) == (want_i, want_j)
    want_trace = [r[1:] for r in rows if r[0] == "trace"]
    assert len(trace) == len(want_trace)
    for got, want in zip(trace, want_trace):
        it, i_low, ii, jj, j_low = (int(x) for x in want[:5])
        a_im1, b_j, b_jm1, a_i = want[5:9]
        assert (got["i_low"], got["i"], got["j"], got["j_low"]) == (i_low, ii, jj, j_low)
        # the compared values printed in the table
        assert int(a_im1) == A[ii - 1] and int(b_j) == B[jj]
        if b_jm1 != "-":
            assert int(b_jm1) == B[jj - 1] and int(a_i) == A[ii]
        assert got["verdict"] == want[9].replace("_", " ")
        assert got["delta"] == int(want[10])
    for r in rows:
        if r[0] == "split":
            kk, si, sj = (int(x) for x in r[1:])
            assert oracle.corank_pages(kk, A, B, lib=lib) == si
            assert oracle.corank_count(kk, A, B, lib=lib) == si
            assert kk - si == sj
    C = oracle.merge_i32(A, B, lib=lib)
    sl = next(r for r in rows if r[0] == "slice")
    start = int(sl[1])
    vals = [int(x) for x in sl[2:]]
    assert list(C[start:start + len(vals)]) == vals
    assert list(C) == sorted(A + B)


def check_tie_case(lib):
    """Hand-derived tie case on the page's tiny inputs, with sources."""
    rows = {r[0]: r[1:] for r in _read_golden("tie_case_small.txt")}
    A = [int(x) for x in rows["A"]]
    B = [int(x) for x in rows["B"]]
    C = [int(x) for x in rows["C"]]
    src = rows["src"]
    assert list(oracle.merge_i32(A, B, lib=lib)) == C
    va = [i for i in range(len(A))]
    vb = [(1 << 31) | i for i in range(len(B))]
    kc, vc = oracle.merge_pairs_u32(A, va, B, vb, lib=lib)
    assert list(kc) == C
    got_src = [("B%d" % (v & 0x7FFFFFFF)) if v >> 31 else ("A%d" % v) for v in vc]
    assert got_src == src
    for k in range(len(C)):
        # co-rank = number of A sources among the first k outputs
        want_i = sum(1 for s in src[:k] if s[0] == "A")
        assert oracle.corank_pages(k, A, B, lib=lib) == want_i
        assert oracle.corank_count(k, A, B, lib=lib) == want_i
        v, from_a = oracle.merge_at_i32(k, A, B, lib=lib)
        assert v == C[k] and from_a == (src[k][0] == "A")


def _sorted_seqs(max_len, alphabet):
    for L in range(max_len + 1):
        yield from itertools.combinations_with_replacement(alphabet, L)


def check_brute_force(lib, max_len=5, alphabet=(0, 1, 2)):
    """Every pair of sorted inputs up to max_len over a 3-letter alphabet:
    the merge equals Python's stable sort of the tagged concatenation, and
    both co-rank routines equal the count of A tags among the first k."""
    seqs = [list(s) for s in _sorted_seqs(max_len, alphabet)]
    for A in seqs:
        for B in seqs:
            tagged = sorted([(a, 0, p) for p, a in enumerate(A)] + [(b, 1, p) for p, b in enumerate(B)],
                            key=lambda t: t[0])  # sorted() is stable: A's items stay first on ties
            want = [t[0] for t in tagged]
            assert list(oracle.merge_i32(A, B, lib=lib)) == want
            va = list(range(len(A)))
            vb = [(1 << 31) | p for p in range(len(B))]
            kc, vc = oracle.merge_pairs_u32(A, va, B, vb, lib=lib)
            assert list(kc) == want
            assert list(vc) == [p if s == 0 else (1 << 31) | p for _, s, p in tagged]
            a_count = 0
            for k in range(len(A) + len(B) + 1):
                assert oracle.corank_pages(k, A, B, lib=lib) == a_count, (A, B, k)
                assert oracle.corank_count(k, A, B, lib=lib) == a_count, (A, B, k)
                if k < len(want):
                    v, from_a = oracle.merge_at_i32(k, A, B, lib=lib)
                    assert v == want[k] and from_a == (tagged[k][1] == 0)
                    a_count += tagged[k][1] == 0


def check_corank_pages_u32(lib, max_len=4, alphabet=(0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF)):
    """The pages' co-rank loop with unsigned compares (O2 on uint32 keys):
    for every pair of sorted inputs up to max_len over an alphabet that
    straddles the sign bit (where a signed compare would reorder keys), and
    for random heavy-tie inputs over the full uint32 range, the result
    equals the number of A tags among the first k items of Python's stable
    sort of the tagged concatenation (the co-rank definition)."""
    def want_coranks(A, B):
        tagged = sorted([(a, 0) for a in A] + [(b, 1) for b in B], key=lambda t: t[0])
        out, a_count = [0], 0
        for _, side in tagged:
            a_count += side == 0
            out.append(a_count)
        return out

    seqs = [list(s) for s in _sorted_seqs(max_len, alphabet)]
    for A in seqs:
        for B in seqs:
            want = want_coranks(A, B)
            for k in range(len(A) + len(B) + 1):
                assert oracle.corank_pages_u32(k, A, B, lib=lib) == want[k], (A, B, k)
    rng = np.random.default_rng(17)
    for _ in range(30):
        m, n = (int(x) for x in rng.integers(0, 90, 2))
        pool = rng.integers(0, 1 << 32, 6, dtype=np.uint64)  # few distinct keys: heavy ties
        A = sorted(int(x) for x in rng.choice(pool, m))
        B = sorted(int(x) for x in rng.choice(pool, n))
        want = want_coranks(A, B)
        for k in range(m + n + 1):
            assert oracle.corank_pages_u32(k, A, B, lib=lib) == want[k], (A, B, k)


def check_evens_odds_closed_form(lib, scale_log2=0):
    """Evens/odds workload: with n = len(B) and A = 0,2,4,... longer by t0:
    C[k] = k for k < 2n, and C[2n + t] = 2n + 2t for the A-only tail;
    co_rank(k) = ceil(k / 2) for k <= 2n and k - n above."""
    d = synth.make_host("evens_odds", scale_log2)
    A, B = d["A"], d["B"]
    m, n = A.size, B.size
    C = oracle.merge_i32(A, B, lib=lib)
    k = np.arange(m + n, dtype=np.int64)
    want = np.where(k < 2 * n, k, 2 * n + 2 * (k - 2 * n))
    assert np.array_equal(C.astype(np.int64), want)
    rng = np.random.default_rng(11)
    ks = np.concatenate([[0, 1, 2, 2 * n - 1, 2 * n, 2 * n + 1, m + n - 1, m + n],
                         rng.integers(0, m + n + 1, 64)])
    for kk in ks:
        kk = int(kk)
        want_i = (kk + 1) // 2 if kk <= 2 * n else kk - n
        assert oracle.corank_pages(kk, A, B, lib=lib) == want_i
    for kk in ks[:12]:
        assert oracle.corank_count(int(kk), A, B, lib=lib) == ((int(kk) + 1) // 2 if kk <= 2 * n else int(kk) - n)


def check_pairs_ties_closed_form(lib, scale_log2=10):
    """Heavy-tie pairs workload: for every key v in order, C holds all of A's
    entries with key v (values = their A positions, ascending) and then all
    of B's (values = 1<<31 | B positions, ascending)."""
    d = synth.make_host("pairs_ties", scale_log2)
    ka, va, kb, vb = d["keysA"], d["valsA"], d["keysB"], d["valsB"]
    kc, vc = oracle.merge_pairs_u32(ka, va, kb, vb, lib=lib)
    want_k, want_v = [], []
    pa = pb = 0
    for v in range(16):
        ca = int(np.count_nonzero(ka == v))
        cb = int(np.count_nonzero(kb == v))
        want_k += [v] * (ca + cb)
        want_v += list(range(pa, pa + ca)) + [(1 << 31) | p for p in range(pb, pb + cb)]
        pa += ca
        pb += cb
    assert np.array_equal(kc, np.array(want_k, dtype=np.uint32))
    assert np.array_equal(vc, np.array(want_v, dtype=np.uint32))


def check_invariants_random(lib, trials=40, seed=5):
    """Nondecreasing output, permutation of the inputs, A-first ties, and
    i + j = k with the acceptance test at every split, on random inputs."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        m = int(rng.integers(0, 300))
        n = int(rng.integers(0, 300))
        span = int(rng.choice([3, 50, 1 << 31]))
        A = np.sort(rng.integers(-span, span, m)).astype(np.int32)
        B = np.sort(rng.integers(-span, span, n)).astype(np.int32)
        C = oracle.merge_i32(A, B, lib=lib)
        assert np.all(np.diff(C.astype(np.int64)) >= 0)
        assert np.array_equal(np.sort(C), np.sort(np.concatenate([A, B])))
        for k in range(0, m + n + 1, max(1, (m + n) // 17)):
            i = oracle.corank_pages(k, A, B, lib=lib)
            j = k - i
            assert max(0, k - n) <= i <= min(k, m)
            assert i == 0 or j == n or A[i - 1] <= B[j]
            assert j == 0 or i == m or B[j - 1] < A[i]
            assert i == oracle.corank_count(k, A, B, lib=lib)
        va = np.arange(m, dtype=np.uint32)
        vb = np.arange(n, dtype=np.uint32) | np.uint32(1 << 31)
        kc, vc = oracle.merge_pairs_u32(A.view(np.uint32) ^ np.uint32(1 << 31), va,
                                        B.view(np.uint32) ^ np.uint32(1 << 31), vb, lib=lib)
        # within each run of equal keys: every A tag before every B tag, each ascending
        for key in np.unique(kc):
            vals = vc[kc == key]
            tags = vals >> np.uint32(31)
            assert np.all(np.diff(tags.astype(np.int64)) >= 0)
            assert np.all(np.diff((vals[tags == 0]).astype(np.int64)) > 0)
            assert np.all(np.diff((vals[tags == 1] & np.uint32(0x7FFFFFFF)).astype(np.int64)) > 0)
        # flipping the sign bit maps int32 order onto uint32 order
        assert np.array_equal((kc ^ np.uint32(1 << 31)).view(np.int32), C)


def check_merge_sort(lib, seed=9):
    """O4 against numpy's stable argsort (a library stable sort), including
    heavy ties, and the sort definition itself (nondecreasing permutation)."""
    rng = np.random.default_rng(seed)
    for n, hi in [(0, 10), (1, 10), (2, 3), (7, 3), (100, 5), (1000, 1 << 32), (4099, 40)]:
        keys = rng.integers(0, hi, n, dtype=np.uint64).astype(np.uint32)
        vals = np.arange(n, dtype=np.uint32)
        sk, sv = oracle.merge_sort_pairs_u32(keys, vals, lib=lib)
        order = np.argsort(keys, kind="stable")
        assert np.array_equal(sk, keys[order])
        assert np.array_equal(sv, vals[order])
        assert np.all(np.diff(sk.astype(np.int64)) >= 0)


def _stable_merge_by(A, B, key):
    """Python's stable sort of A's items then B's items; returns (value, side)."""
    tagged = sorted([(a, 0) for a in A] + [(b, 1) for b in B], key=lambda t: key(t[0]))
    return tagged


def check_typed_keys(lib, max_len=4):
    """O1 on uint32 and float32 keys.

    uint32: every pair of sorted inputs over an alphabet that straddles the
    sign bit equals the stable sort of the concatenation by unsigned value,
    so a signed compare (0x80000000 before 0) fails.  float32: the alphabet
    holds -inf, a negative, -0.0 and +0.0 (equal as floats, different bits),
    a subnormal and +inf; the merge must equal the stable sort by float value
    bit for bit, so comparing raw bits (negatives reversed) or taking B first
    on a tie (+0.0 of B ahead of -0.0 of A) fails."""
    u_alpha = (0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF)
    seqs = [list(s) for s in _sorted_seqs(max_len, u_alpha)]
    for A in seqs:
        for B in seqs:
            want = [v for v, _ in _stable_merge_by(A, B, key=int)]
            got = oracle.merge_u32(np.array(A, np.uint32), np.array(B, np.uint32), lib=lib)
            assert [int(x) for x in got] == want, (A, B)
    f_alpha = np.array([-np.inf, -1.5, -0.0, 0.0, 1e-45, np.inf], dtype=np.float32)
    # sorted by float order, -0.0 and +0.0 equal; every order of the two zeros
    # inside a sequence is a valid sorted input, so enumerate bit patterns
    bits = [int(x) for x in f_alpha.view(np.uint32)]
    fval = {b: float(np.array([b], np.uint32).view(np.float32)[0]) for b in bits}
    fseqs = []
    for L in range(max_len + 1):
        for combo in itertools.product(bits, repeat=L):
            if all(fval[combo[t]] <= fval[combo[t + 1]] for t in range(L - 1)):
                fseqs.append(list(combo))
    rng = np.random.default_rng(17)
    pick = rng.choice(len(fseqs), size=min(len(fseqs), 140), replace=False)
    sub = [fseqs[int(t)] for t in pick] + [[], [bits[2]], [bits[3]]]
    for A in sub:
        for B in sub:
            want = [v for v, _ in _stable_merge_by(A, B, key=lambda b: fval[b])]
            got = oracle.merge_f32(np.array(A, np.uint32).view(np.float32),
                                   np.array(B, np.uint32).view(np.float32), lib=lib)
            assert [int(x) for x in got.view(np.uint32)] == want, (A, B)
    # larger random inputs against numpy's stable argsort of the concatenation
    for m, n in [(0, 7), (7, 0), (1000, 999), (4097, 33)]:
        a = np.sort(rng.integers(0, 1 << 32, m, dtype=np.uint64)).astype(np.uint32)
        b = np.sort(rng.integers(0, 1 << 32, n, dtype=np.uint64)).astype(np.uint32)
        cat = np.concatenate([a, b])
        assert np.array_equal(oracle.merge_u32(a, b, lib=lib), cat[np.argsort(cat, kind="stable")])
        fa = np.sort(rng.choice(f_alpha, m).astype(np.float32) * rng.integers(1, 4, m).astype(np.float32))
        fb = np.sort(rng.choice(f_alpha, n).astype(np.float32) * rng.integers(1, 4, n).astype(np.float32))
        fcat = np.concatenate([fa, fb])
        got = oracle.merge_f32(fa, fb, lib=lib)
        assert np.array_equal(got.view(np.uint32), fcat[np.argsort(fcat, kind="stable")].view(np.uint32))


_KEY_ALPHABETS = {
    np.int32: [np.iinfo(np.int32).min, -1, 0, 1, np.iinfo(np.int32).max],
    np.uint32: [0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF],
    np.float32: [-np.inf, -1.5, -0.0, 0.0, 1e-45, np.inf],
    np.int64: [np.iinfo(np.int64).min, -(1 << 32), -1, 0, 1 << 32, np.iinfo(np.int64).max],
    np.uint64: [0, 1, (1 << 63) - 1, 1 << 63, (1 << 64) - 1],
    np.float64: [-np.inf, -2.5e300, -0.0, 0.0, 5e-324, np.inf],
}


def _sorted_inputs(values, dtype, max_len, descending, rng, limit):
    """Sorted sequences (in the merge order) over `values`, as bit patterns:
    every arrangement the order allows, including -0.0 / +0.0 in either
    order, sampled down to `limit`."""
    arr = np.array(values, dtype=dtype)
    ubits = {4: np.uint32, 8: np.uint64}[arr.itemsize]
    pats = [int(b) for b in arr.view(ubits)]
    num = {p: arr[t].item() for t, p in enumerate(pats)}
    seqs = []
    for L in range(max_len + 1):
        for combo in itertools.product(pats, repeat=L):
            vals = [num[p] for p in combo]
            ok = all((vals[t] >= vals[t + 1]) if descending else (vals[t] <= vals[t + 1]) for t in range(L - 1))
            if ok:
                seqs.append(list(combo))
    if len(seqs) > limit:
        keep = rng.choice(len(seqs), size=limit, replace=False)
        seqs = [seqs[int(t)] for t in keep] + [[]]
    return seqs, num, ubits


def _stable_desc_order(x):
    """Indices of a stable descending sort, from numpy's stable ascending
    argsort: sort the reversed array, reverse the result, map back."""
    r = np.argsort(x[::-1], kind="stable")[::-1]
    return x.size - 1 - r


def check_merge_keys(lib, max_len=3, limit=60):
    """O1 for all six key types, ascending and descending.

    Brute force: every pair of sorted inputs (sampled) over an alphabet of
    the type's extremes (sign bits, -0.0 and +0.0, subnormals, infinities)
    equals Python's stable sort of the concatenation by numeric value, bit
    for bit; sorted(..., reverse=True) is documented stable, so descending
    ties keep A first.  A wrong compare type (signed for unsigned, bits for
    floats), a flipped tie rule or a reversed order each fails here.  Random
    inputs: equal to numpy's stable argsort of the concatenation (for
    descending, through the reversal construction above)."""
    rng = np.random.default_rng(23)
    for dtype, alpha in _KEY_ALPHABETS.items():
        for desc in (False, True):
            seqs, num, ubits = _sorted_inputs(alpha, dtype, max_len, desc, rng, limit)
            for A in seqs:
                for B in seqs:
                    tagged = sorted([(num[p], p) for p in A] + [(num[p], p) for p in B],
                                    key=lambda t: t[0], reverse=desc)
                    want = [p for _, p in tagged]
                    a = np.array(A, dtype=ubits).view(dtype)
                    b = np.array(B, dtype=ubits).view(dtype)
                    got = oracle.merge_keys(a, b, descending=desc, lib=lib)
                    assert [int(x) for x in got.view(ubits)] == want, (dtype, desc, A, B)
            for m, n in [(0, 9), (9, 0), (500, 700), (2049, 31)]:
                src = np.array(alpha, dtype=dtype)
                a = src[rng.integers(0, src.size, m)]
                b = src[rng.integers(0, src.size, n)]
                if np.issubdtype(dtype, np.integer):
                    info = np.iinfo(dtype)
                    a = np.concatenate([a[: m // 2], rng.integers(info.min, info.max, m - m // 2, dtype=dtype,
                                                                  endpoint=True)]) if m else a
                    b = np.concatenate([b[: n // 2], rng.integers(info.min, info.max, n - n // 2, dtype=dtype,
                                                                  endpoint=True)]) if n else b
                else:
                    a = (a * rng.integers(1, 5, m)).astype(dtype)
                    b = (b * rng.integers(1, 5, n)).astype(dtype)
                a = np.sort(a, kind="stable")
                b = np.sort(b, kind="stable")
                if desc:
                    a, b = a[::-1].copy(), b[::-1].copy()
                cat = np.concatenate([a, b])
                order = _stable_desc_order(cat) if desc else np.argsort(cat, kind="stable")
                got = oracle.merge_keys(a, b, descending=desc, lib=lib)
                assert np.array_equal(got.view(ubits), cat[order].view(ubits)), (dtype, desc, m, n)


def check_merge_sort_keys(lib, max_len=5):
    """O4 on all six key types, both orders, with and without values.

    Brute force: every sequence up to max_len over three keys of the type
    (for floats -0.0, +0.0 and 1.0, so equal keys with different bits show
    whether input order is kept) sorts as Python's stable sorted() by value
    (reverse=True is documented stable).  Random inputs with heavy ties and
    the type's extremes: keys (bit for bit) and values equal the
    permutation of numpy's stable argsort (descending through the reversal
    construction)."""
    rng = np.random.default_rng(29)
    for dtype, alpha in _KEY_ALPHABETS.items():
        arr = np.array(alpha, dtype=dtype)
        ubits = {4: np.uint32, 8: np.uint64}[arr.itemsize]
        small = np.array([-0.0, 0.0, 1.0] if arr.dtype.kind == "f" else [alpha[0], alpha[2], alpha[-1]], dtype=dtype)
        for desc in (False, True):
            for L in range(max_len + 1):
                for combo in itertools.product(range(3), repeat=L):
                    keys = small[list(combo)]
                    tags = np.arange(L, dtype=np.uint32)
                    want = sorted(zip(keys.tolist(), keys.view(ubits).tolist(), tags.tolist()),
                                  key=lambda t: t[0], reverse=desc)
                    gk, gv = oracle.merge_sort_keys(keys, tags, descending=desc, lib=lib)
                    assert gk.view(ubits).tolist() == [w[1] for w in want], (dtype, desc, combo)
                    assert gv.tolist() == [w[2] for w in want], (dtype, desc, combo)
            for n in [0, 1, 2, 7, 100, 1000, 4099]:
                keys = arr[rng.integers(0, arr.size, n)]
                if arr.dtype.kind in "iu" and n > 4:
                    info = np.iinfo(dtype)
                    keys[: n // 2] = rng.integers(info.min, info.max, n // 2, dtype=dtype, endpoint=True)
                vals = np.arange(n, dtype=np.uint32)
                order = _stable_desc_order(keys) if desc else np.argsort(keys, kind="stable")
                gk, gv = oracle.merge_sort_keys(keys, vals, descending=desc, lib=lib)
                assert np.array_equal(gk.view(ubits), keys[order].view(ubits)), (dtype, desc, n)
                assert np.array_equal(gv, vals[order]), (dtype, desc, n)
                gk2, none = oracle.merge_sort_keys(keys, None, descending=desc, lib=lib)
                assert none is None and np.array_equal(gk2.view(ubits), gk.view(ubits))


ALL_CHECKS = [
    check_worked_example,
    check_tie_case,
    check_brute_force,
    check_corank_pages_u32,
    check_evens_odds_closed_form,
    check_pairs_ties_closed_form,
    check_invariants_random,
    check_merge_sort,
    check_typed_keys,
    check_merge_keys,
    check_merge_sort_keys,
]


# ------------------------------------------------------------------ tests --

@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)


def test_evens_odds_closed_form_full_size(oracle_lib):
    """The full evens/odds workload (4,194,915 outputs), not a scaled copy."""
    check_evens_odds_closed_form(oracle_lib, scale_log2=0)


def test_pairs_ties_closed_form_larger(oracle_lib):
    check_pairs_ties_closed_form(oracle_lib, scale_log2=6)


def test_corank_step_bound(oracle_lib):
    """The pages' loop takes at most bitlength(min(m, n)) + 1 iterations
    (the interval starts no wider than min(m, n) and halves each step; the
    extra row is the accepting one)."""
    d = synth.make_host("evens_odds", 6)
    A, B = d["A"], d["B"]
    bound = int(min(A.size, B.size)).bit_length() + 1
    for k in [0, 1, 5, 1000, A.size, A.size + B.size]:
        _, rows = oracle.corank_pages(k, A, B, trace=True, lib=oracle_lib)
        assert len(rows) <= bound


def test_merge_sort_matches_python_sorted(oracle_lib):
    rng = np.random.default_rng(3)
    keys = rng.integers(0, 7, 257).astype(np.uint32)
    vals = np.arange(257, dtype=np.uint32)
    sk, sv = oracle.merge_sort_pairs_u32(keys, vals, lib=oracle_lib)
    want = sorted(zip(keys.tolist(), vals.tolist()), key=lambda t: t[0])
    assert list(zip(sk.tolist(), sv.tolist())) == want

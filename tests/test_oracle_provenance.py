"""Pins of the oracle's path provenance (no GPU).

`oracle.smooth_track` returns, besides the fp64 fixed point, the fewest edges
of a shortest upper-bound path (HU), of a best lower-bound path (HL) and the
summed |edge weight| of that lower-bound path (ML).  These numbers state the
rounding bound of fp32 results off the 1/1024 grid, so they are pinned here
against an enumeration of every simple path of tiny bound graphs, against a
chain whose paths are known by construction, and against the plain fp64
rounds.  The path structure is that of the triangle inequalities of GPU Gems 2
ch. 43, section 2 (u edges within a copy of the atoms, one -l edge between
the copies).
"""
import itertools

import numpy as np
import pytest

from workloads import molecules as W


def brute_force(U0, L0):
    """Lexicographic (length, edges) over all simple u paths, and (value,
    edges) over all lower-bound paths i..a, -l(a, b), b..j; n <= 6."""
    n = U0.shape[0]
    bu = np.full((n, n), np.inf)
    bh = np.zeros((n, n), np.int64)
    for i in range(n):
        bu[i, i] = 0.0
    for length in range(2, n + 1):
        for path in itertools.permutations(range(n), length):
            s = sum(U0[path[t], path[t + 1]] for t in range(length - 1))
            i, j, h = path[0], path[-1], length - 1
            if s < bu[i, j] or (s == bu[i, j] and h < bh[i, j]):
                bu[i, j], bh[i, j] = s, h
    bl = np.full((n, n), -np.inf)
    hl = np.zeros((n, n), np.int64)
    ml = np.zeros((n, n))
    ties = np.zeros((n, n), bool)
    for i, j in itertools.product(range(n), repeat=2):
        for a, b in itertools.product(range(n), repeat=2):
            v = L0[a, b] - bu[i, a] - bu[b, j]
            h = bh[i, a] + 1 + bh[b, j]
            m = L0[a, b] + bu[i, a] + bu[b, j]
            if v > bl[i, j] or (v == bl[i, j] and h < hl[i, j]):
                ties[i, j] = v == bl[i, j] and m != ml[i, j]
                bl[i, j], hl[i, j], ml[i, j] = v, h, m
            elif v == bl[i, j] and h == hl[i, j] and m != ml[i, j]:
                ties[i, j] = True
    return bu, bh, bl, hl, ml, ties


@pytest.mark.parametrize("seed", range(8))
def test_hops_against_enumeration_with_ties(oracle_lib, seed):
    """Small integer weights: many shortest paths tie, and the fewest edges
    among them must be found."""
    n = 4 + seed % 3
    rng = np.random.default_rng(900 + seed)
    U0 = rng.integers(0, 4, size=(n, n)).astype(np.float64)
    if seed % 2 == 0:
        U0 = np.minimum(U0, U0.T)
    np.fill_diagonal(U0, 0)
    L0 = rng.integers(0, 3, size=(n, n)).astype(np.float64)
    np.fill_diagonal(L0, 0)
    bu, bh, bl, hl, _, _ = brute_force(U0, L0)
    U, L, HU, HL, ML = oracle_lib.smooth_track(U0, L0)
    np.testing.assert_array_equal(U, bu)
    np.testing.assert_array_equal(HU, bh)
    np.testing.assert_array_equal(L, bl)
    np.testing.assert_array_equal(HL, hl)


@pytest.mark.parametrize("seed", range(6))
def test_magnitudes_against_enumeration(oracle_lib, seed):
    """Real weights: the best lower-bound path is unique, and ML is the sum
    of |weights| along it."""
    n = 4 + seed % 3
    rng = np.random.default_rng(950 + seed)
    U0 = rng.random((n, n)) * 5 + 0.5
    np.fill_diagonal(U0, 0)
    L0 = rng.random((n, n)) * 6
    np.fill_diagonal(L0, 0)
    bu, bh, bl, hl, ml, ties = brute_force(U0, L0)
    U, L, HU, HL, ML = oracle_lib.smooth_track(U0, L0)
    np.testing.assert_allclose(U, bu, rtol=1e-13)
    np.testing.assert_allclose(L, bl, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(HU, bh)
    np.testing.assert_array_equal(HL, hl)
    np.testing.assert_allclose(ML[~ties], ml[~ties], rtol=1e-13)


def test_chain_hops(oracle_lib):
    """A chain known only between neighbours: the shortest path from i to j
    is the chain itself, |i - j| edges; the best lower bound of a pair comes
    from its own -l edge when nothing beats it."""
    n = 40
    U0 = np.full((n, n), 1000.0)
    L0 = np.full((n, n), 1.0)
    for i in range(n - 1):
        U0[i, i + 1] = U0[i + 1, i] = 3.8
        L0[i, i + 1] = L0[i + 1, i] = 3.7
    np.fill_diagonal(U0, 0)
    np.fill_diagonal(L0, 0)
    U, L, HU, HL, ML = oracle_lib.smooth_track(U0, L0)
    idx = np.arange(n)
    np.testing.assert_array_equal(HU, np.abs(idx[:, None] - idx[None, :]))
    np.testing.assert_allclose(U, 3.8 * np.abs(idx[:, None] - idx[None, :]), rtol=1e-12)
    # neighbours keep their own bound: one edge, magnitude 3.7
    assert all(HL[i, i + 1] == 1 and ML[i, i + 1] == 3.7 for i in range(n - 1))
    # the lower bound of every cell is the length of its path
    assert np.all(ML >= np.abs(L) - 1e-12)


def test_values_equal_plain_rounds(oracle_lib):
    """The tracked rounds form the same fp64 candidates as the plain rounds."""
    U0, L0 = W.random_bounds(60, 31, p_known=0.3, p_bad=0.02)
    rng = np.random.default_rng(5)
    U0 = U0 / 1024.0 + rng.random(U0.shape) * 1e-3
    L0 = np.maximum(L0 / 1024.0 - rng.random(L0.shape) * 1e-3, 0)
    np.fill_diagonal(U0, 0)
    np.fill_diagonal(L0, 0)
    U, L, HU, HL, ML = oracle_lib.smooth_track(U0, L0)
    Up, Lp = oracle_lib.smooth(U0.copy(), L0.copy())
    np.testing.assert_array_equal(U, Up)
    np.testing.assert_array_equal(L, Lp)
    assert HU.min() == 0 and np.all(np.diag(HU) == 0) and HU.max() < 60
    assert HL.min() >= 1 and np.all(ML >= 0)


# ---------------------------------------------------------------- planted mistakes

import ctypes  # noqa: E402
import os  # noqa: E402
import subprocess  # noqa: E402

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "oracle.c")

TRACK_MUTANTS = {
    "ties_keep_more_edges": ("if (s < U[c] || (s == U[c] && hs < HU[c])) {",
                             "if (s < U[c] || (s == U[c] && hs > HU[c])) {"),
    "upper_edges_not_added": ("const int32_t hs = hucol[i] + hurow[j];",
                              "const int32_t hs = hucol[i];"),
    "lower_edges_not_added": ("const int32_t ha = hlrow[j] + hucol[i];",
                              "const int32_t ha = hlrow[j];"),
    "magnitude_drops_u": ("ML[c] = mrow[j] + ucol[i];", "ML[c] = mrow[j];"),
    "raise_keeps_old_magnitude": ("mc = mkk + ucol[i];", "(void)mkk;"),
}


def track_variant(tmp_path, name, patch):
    src = open(SRC).read()
    old, new = patch
    assert src.count(old) == 1, name
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("%s.so" % name)
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                    str(c), "-o", str(so)], check=True)
    f = ctypes.CDLL(str(so)).oracle_smooth_track_f64
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 2
    f.restype = ctypes.c_int

    def run(U0, L0):
        n = U0.shape[0]
        U, L = U0.astype(np.float64).copy(), L0.astype(np.float64).copy()
        HU, HL = np.empty((n, n), np.int32), np.empty((n, n), np.int32)
        ML = np.empty((n, n))
        assert f(U.ctypes.data, L.ctypes.data, HU.ctypes.data, HL.ctypes.data,
                 ML.ctypes.data, n, n) == 0
        return U, L, HU, HL, ML
    return run


def golden_matrices():
    """The worked examples (tests/golden): exact multiples of 1/8, so many
    paths tie, and example C needs the closure raise (l_22 > 0)."""
    import json
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                           "examples.json")) as f:
        exs = json.load(f)["examples"]
    out = []
    for ex in exs:
        n = ex["n"]
        lo, hi = ex["unknown"]
        U0 = np.full((n, n), float(hi))
        L0 = np.full((n, n), float(lo))
        for i, j, l, u in ex["pairs"]:
            U0[i, j] = U0[j, i] = u
            L0[i, j] = L0[j, i] = l
        np.fill_diagonal(U0, 0)
        np.fill_diagonal(L0, 0)
        out.append((ex["name"], U0, L0))
    return out


@pytest.mark.parametrize("idx", range(3))
def test_golden_examples(oracle_lib, idx):
    name, U0, L0 = golden_matrices()[idx]
    bu, bh, bl, hl, ml, ties = brute_force(U0, L0)
    U, L, HU, HL, ML = oracle_lib.smooth_track(U0, L0)
    np.testing.assert_array_equal(U, bu)
    np.testing.assert_array_equal(L, bl)
    np.testing.assert_array_equal(HU, bh)
    np.testing.assert_array_equal(HL, hl)
    np.testing.assert_array_equal(ML[~ties], ml[~ties])
    if name == "C":
        # l*_33 = l_02 - u*_30 - u*_23: three u edges, one -l edge, one u edge
        assert L[3, 3] == 0.5 and HL[3, 3] == 5 and ML[3, 3] == 17.5


def pins_pass(run):
    """The enumeration pins above, as one predicate."""
    for name, U0, L0 in golden_matrices():
        bu, bh, bl, hl, ml, ties = brute_force(U0, L0)
        U, L, HU, HL, ML = run(U0, L0)
        if not (np.array_equal(HL, hl) and np.array_equal(ML[~ties], ml[~ties])):
            return False
    for seed in range(8):
        n = 4 + seed % 3
        rng = np.random.default_rng(900 + seed)
        U0 = rng.integers(0, 4, size=(n, n)).astype(np.float64)
        np.fill_diagonal(U0, 0)
        L0 = rng.integers(0, 3, size=(n, n)).astype(np.float64)
        np.fill_diagonal(L0, 0)
        bu, bh, bl, hl, _, _ = brute_force(U0, L0)
        U, L, HU, HL, _ = run(U0, L0)
        if not (np.array_equal(HU, bh) and np.array_equal(HL, hl)):
            return False
    for seed in range(6):
        n = 4 + seed % 3
        rng = np.random.default_rng(950 + seed)
        U0 = rng.random((n, n)) * 5 + 0.5
        np.fill_diagonal(U0, 0)
        L0 = rng.random((n, n)) * 6
        np.fill_diagonal(L0, 0)
        bu, bh, bl, hl, ml, ties = brute_force(U0, L0)
        U, L, HU, HL, ML = run(U0, L0)
        if not np.allclose(ML[~ties], ml[~ties], rtol=1e-13):
            return False
    return True


@pytest.mark.parametrize("name", sorted(TRACK_MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    assert not pins_pass(track_variant(tmp_path, name, TRACK_MUTANTS[name]))


def test_unmutated_source_passes(tmp_path):
    assert pins_pass(track_variant(tmp_path, "same", ("int rc = 0;", "int rc = 0;")))

"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties the oracle to something it does not compute by itself:
hand-worked examples, a library shortest-path routine, the closed form of the
lower-bound fixed point, invariants of the triangle inequalities, a
brute-force enumeration of bound-graph paths, and the generating geometry.
The rules pinned are those of GPU Gems 2 ch. 43 ("GPU Computing for Protein
Structure Prediction"), section 2 (triangle inequality, upper before lower)
and section 3 (Floyd-Warshall rounds over the middle atom k).
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.sparse.csgraph import floyd_warshall

from workloads import molecules as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "examples.json")


def load_examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def example_matrices(ex, dtype):
    n = ex["n"]
    lo, hi = ex["unknown"]
    U = np.full((n, n), hi)
    L = np.full((n, n), lo)
    np.fill_diagonal(U, 0)
    np.fill_diagonal(L, 0)
    for i, j, l, u in ex["pairs"]:
        U[i, j] = U[j, i] = u
        L[i, j] = L[j, i] = l
    if dtype == "i32":
        return (np.round(U * 1024).astype(np.int32), np.round(L * 1024).astype(np.int32), 1024.0)
    dt = np.float32 if dtype == "f32" else np.float64
    return U.astype(dt), L.astype(dt), 1.0


@pytest.mark.parametrize("dtype", ["f32", "f64", "i32"])
@pytest.mark.parametrize("ex", load_examples(), ids=lambda e: e["name"])
def test_worked_examples(oracle_lib, ex, dtype):
    U0, L0, s = example_matrices(ex, dtype)
    U, L = oracle_lib.smooth(U0, L0)
    np.testing.assert_array_equal(U / s, np.array(ex["U"], dtype=float))
    np.testing.assert_array_equal(L / s, np.array(ex["L"], dtype=float))
    assert oracle_lib.count_infeasible(U, L) == ex["flags"]
    Ul, Ll = oracle_lib.smooth(U0, L0, rule=oracle_lib.RULE_LITERAL)
    np.testing.assert_array_equal(Ul, U)
    if ex["literal_same"]:
        np.testing.assert_array_equal(Ll, L)
    else:
        np.testing.assert_array_equal(Ll / s, np.array(ex["literal_L"], dtype=float))
        assert oracle_lib.count_infeasible(Ul, Ll) == ex["literal_flags"]


def test_example_witness(oracle_lib):
    """Example A is consistent: the printed coordinates lie inside every bound."""
    ex = [e for e in load_examples() if e["name"] == "A"][0]
    U0, L0, _ = example_matrices(ex, "f64")
    U, L = oracle_lib.smooth(U0, L0)
    x = np.array(ex["witness"], dtype=float)
    d = np.sqrt(((x[:, None] - x[None]) ** 2).sum(-1))
    assert np.all(L0 <= d) and np.all(d <= U0)
    assert np.all(L <= d) and np.all(d <= U)


# ---------------------------------------------------------------- upper bound


def random_weights(n, seed, directed):
    rng = np.random.default_rng(seed)
    q = rng.integers(1, 60 * 1024, size=(n, n)).astype(np.int32)   # >= 1/1024, never 0
    big = rng.random((n, n)) < 0.6                                   # most pairs "unknown"
    q[big] = W.sentinel_q(n)
    if not directed:
        q = np.triu(q, 1)
        q = q + q.T
    np.fill_diagonal(q, 0)
    return q


@pytest.mark.parametrize("n", [1, 2, 3, 5, 17, 64])
@pytest.mark.parametrize("directed", [False, True])
def test_upper_is_shortest_paths(oracle_lib, n, directed):
    """U after smoothing equals all-pairs shortest paths (scipy Floyd-Warshall)."""
    q = random_weights(n, 10 + n, directed)
    ref = floyd_warshall(q.astype(np.float64), directed=True)
    Ui = oracle_lib.smooth_upper(q)
    np.testing.assert_array_equal(Ui.astype(np.float64), ref)
    Uf = oracle_lib.smooth_upper(W.to_f32(q))
    np.testing.assert_array_equal(Uf.astype(np.float64) * 1024, ref)
    Ud = oracle_lib.smooth_upper(q.astype(np.float64))
    np.testing.assert_array_equal(Ud, ref)


def test_upper_only_matches_upper_of_bounds(oracle_lib):
    U0, L0 = W.random_bounds(40, 3, p_bad=0.05)
    U1 = oracle_lib.smooth_upper(U0)
    U2, _ = oracle_lib.smooth(U0, L0)
    np.testing.assert_array_equal(U1, U2)


# ---------------------------------------------------------------- lower bound


def closed_form_lower(U0, L0):
    """l*_ij = max(l_ij, max_{a,b} l_ab - u*_ia - u*_bj), u* by scipy, in fp64.

    Computed as two max-minus products: T[i,b] = max_a (l_ab - u*_ia), then
    l*_ij = max(l_ij, max_b (T[i,b] - u*_bj)).
    """
    Us = floyd_warshall(U0.astype(np.float64), directed=True)
    L0 = L0.astype(np.float64)
    T = np.max(L0[None, :, :] - Us[:, :, None], axis=1)
    Lc = np.max(T[:, :, None] - Us[None, :, :], axis=1)
    return Us, np.maximum(L0, Lc)


@pytest.mark.parametrize("n,p_bad,sym", [(2, 0.0, True), (5, 0.3, True), (16, 0.0, True),
                                         (16, 0.1, True), (33, 0.05, False),
                                         (48, 0.02, True), (48, 0.0, False)])
def test_lower_matches_closed_form(oracle_lib, n, p_bad, sym):
    U0, L0 = W.random_bounds(n, 100 + n, p_known=0.4, p_bad=p_bad, symmetric=sym)
    U0 = np.where((U0 == 0) & ~np.eye(n, dtype=bool), 1, U0).astype(np.int32)
    Us, Ls = closed_form_lower(U0, L0)
    Ui, Li = oracle_lib.smooth(U0, L0)
    np.testing.assert_array_equal(Ui.astype(np.float64), Us)
    np.testing.assert_array_equal(Li.astype(np.float64), Ls)
    Uf, Lf = oracle_lib.smooth(W.to_f32(U0), W.to_f32(L0))
    np.testing.assert_array_equal(Lf.astype(np.float64) * 1024, Ls)


def brute_force_paths(U0, L0):
    """Enumerate every simple path of the doubled bound graph (n <= 5).

    u*_ij = min over simple paths i..j of the summed u; l*_ij = max over paths
    i..a (u edges), one edge a->b (-l_ab), b..j (u edges) of l_ab - sums.
    """
    n = U0.shape[0]
    best_u = np.full((n, n), np.inf)
    for i in range(n):
        best_u[i, i] = 0.0
    for length in range(2, n + 1):
        for path in itertools.permutations(range(n), length):
            s = sum(U0[path[t], path[t + 1]] for t in range(length - 1))
            best_u[path[0], path[-1]] = min(best_u[path[0], path[-1]], s)
    best_l = np.full((n, n), -np.inf)
    for i, a, b, j in itertools.product(range(n), repeat=4):
        best_l[i, j] = max(best_l[i, j], L0[a, b] - best_u[i, a] - best_u[b, j])
    return best_u, np.maximum(best_l, L0)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(oracle_lib, seed):
    n = 3 + seed % 3
    U0, L0 = W.random_bounds(n, 500 + seed, p_known=0.7, p_bad=0.2,
                             symmetric=seed % 2 == 0, maxval=10.0)
    U0 = U0.astype(np.float64) / 1024
    L0 = L0.astype(np.float64) / 1024
    bu, bl = brute_force_paths(U0, L0)
    U, L = oracle_lib.smooth(U0, L0)
    np.testing.assert_array_equal(U, bu)
    np.testing.assert_array_equal(L, bl)


# ---------------------------------------------------------------- invariants


def check_invariants(U, L, consistent, tol=0.0):
    n = U.shape[0]
    Uf = U.astype(np.float64)
    Lf = L.astype(np.float64)
    # every triangle inequality holds at the fixed point, for every k
    assert np.all(Uf[:, None, :] <= Uf[:, :, None] + Uf[None, :, :] + tol)
    assert np.all(Lf[:, None, :] >= Lf[:, :, None] - Uf[None, :, :] - tol)   # l_ik - u_kj
    assert np.all(Lf[:, None, :] >= Lf[None, :, :] - Uf[:, :, None] - tol)   # l_kj - u_ik
    assert np.all(np.diag(Uf) == 0)
    if consistent:
        assert np.all(np.diag(Lf) == 0)
        assert np.all(Lf <= Uf)
    del n


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_invariants_on_chain(oracle_lib, dtype):
    m = W.chain_bounds(96, 77, 0.05)
    U0, L0 = m["U"], m["L"]
    if dtype == "f32":
        U0, L0 = W.to_f32(U0), W.to_f32(L0)
    U, L = oracle_lib.smooth(U0, L0)
    check_invariants(U, L, consistent=True)
    # symmetric in, symmetric out
    np.testing.assert_array_equal(U, U.T)
    np.testing.assert_array_equal(L, L.T)
    # monotone: bounds only tighten
    assert np.all(U <= U0) and np.all(L >= L0)
    # idempotent: a second smoothing changes nothing
    U2, L2 = oracle_lib.smooth(U, L)
    np.testing.assert_array_equal(U2, U)
    np.testing.assert_array_equal(L2, L)
    # the generating coordinates stay inside the smoothed bounds
    x = m["coords"]
    d = np.sqrt(((x[:, None] - x[None]) ** 2).sum(-1))
    s = 1.0 if dtype == "f32" else 1024.0
    assert np.all(L / s <= d + 1e-9) and np.all(d <= U / s + 1e-9)


def test_invariants_inconsistent(oracle_lib):
    """With inverted pairs the triangle inequalities still hold at the fixed point."""
    U0, L0 = W.random_bounds(40, 9, p_known=0.4, p_bad=0.05)
    U, L = oracle_lib.smooth(U0, L0)
    check_invariants(U, L, consistent=False)
    assert oracle_lib.count_infeasible(U, L) > 0


def test_rules_agree_when_consistent(oracle_lib):
    for seed in range(3):
        m = W.chain_bounds(64, 200 + seed, 0.1)
        a = oracle_lib.smooth(m["U"], m["L"])
        b = oracle_lib.smooth(m["U"], m["L"], rule=oracle_lib.RULE_LITERAL)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_fp32_equals_q10_on_grid(oracle_lib):
    """On the 1/1024 grid with values below 2**14, fp32 smoothing is exact."""
    for m in (W.chain_bounds(200, 31, 0.05),
              W.chain_bounds(150, 32, 0.02, near=6.0, jitter=True, long_halfwidth=1.5)):
        Ui, Li = oracle_lib.smooth(m["U"], m["L"])
        Uf, Lf = oracle_lib.smooth(W.to_f32(m["U"]), W.to_f32(m["L"]))
        np.testing.assert_array_equal(Uf * 1024, Ui.astype(np.float32))
        np.testing.assert_array_equal(Lf * 1024, Li.astype(np.float32))
    U0, L0 = W.random_bounds(70, 5, p_bad=0.03)
    Ui, Li = oracle_lib.smooth(U0, L0)
    Uf, Lf = oracle_lib.smooth(W.to_f32(U0), W.to_f32(L0))
    np.testing.assert_array_equal(Uf * 1024, Ui.astype(np.float32))
    np.testing.assert_array_equal(Lf * 1024, Li.astype(np.float32))


def test_round_ranges_compose(oracle_lib):
    U0, L0 = W.random_bounds(50, 11, p_bad=0.02)
    full = oracle_lib.smooth(U0, L0)
    a = oracle_lib.smooth(U0, L0, k_begin=0, k_end=17)
    b = oracle_lib.smooth(a[0], a[1], k_begin=17, k_end=50)
    np.testing.assert_array_equal(b[0], full[0])
    np.testing.assert_array_equal(b[1], full[1])


def test_leading_dimension(oracle_lib):
    """Columns beyond n are never read or written."""
    n, ld = 37, 44
    U0, L0 = W.random_bounds(n, 12, p_bad=0.02)
    Up = np.full((n, ld), -7, dtype=np.int32)
    Lp = np.full((n, ld), -9, dtype=np.int32)
    Up[:, :n], Lp[:, :n] = U0, L0
    ref = oracle_lib.smooth(U0, L0)
    U, L = oracle_lib.smooth(Up, Lp, n=n)
    np.testing.assert_array_equal(U[:, :n], ref[0])
    np.testing.assert_array_equal(L[:, :n], ref[1])
    assert np.all(U[:, n:] == -7) and np.all(L[:, n:] == -9)


# ---------------------------------------------------------------- sampled rows


@pytest.mark.parametrize("n,p_bad,sym", [(1, 0, True), (9, 0.1, True), (40, 0.03, True),
                                         (57, 0.02, False), (64, 0.0, True)])
def test_closure_rows_match_rounds(oracle_lib, n, p_bad, sym):
    """Dijkstra rows of the fixed point equal the round-by-round result."""
    U0, L0 = W.random_bounds(n, 300 + n, p_bad=p_bad, symmetric=sym)
    U, L = oracle_lib.smooth(U0, L0)
    rows = np.arange(n)
    Ur, Lr = oracle_lib.closure_rows(U0, L0, rows)
    np.testing.assert_array_equal(Ur, U.astype(np.float64))
    np.testing.assert_array_equal(Lr, L.astype(np.float64))


# ---------------------------------------------------------------- the generator


@pytest.mark.parametrize("idx", [0, 1])
def test_generated_chains_are_consistent(idx):
    m = W.make_config(idx)
    n, U, L, x = m["n"], m["U"], m["L"], m["coords"]
    d = np.sqrt(((x[:, None] - x[None]) ** 2).sum(-1)) * 1024
    assert np.array_equal(U, U.T) and np.array_equal(L, L.T)
    assert np.all(np.diag(U) == 0) and np.all(np.diag(L) == 0)
    assert np.all(L <= d + 1e-6) and np.all(d <= U + 1e-6)
    assert U.max() == W.sentinel_q(n)
    assert np.all(U[np.arange(n - 1), np.arange(1, n)] < W.sentinel_q(n))


def test_generated_globule_small():
    """Globule generator: a self-avoiding lattice chain; short pairs <= 6 A known."""
    rng = np.random.default_rng(0)
    sites, x = W.lattice_globule((6, 5, 4), rng)
    assert len(np.unique(sites, axis=0)) == len(sites) == 120
    steps = np.abs(np.diff(sites, axis=0)).sum(1)
    assert np.all(steps == 1)
    m = W.globule_bounds((6, 5, 4), 5, 0.05, p_bad=0.02)
    U, L, x = m["U"], m["L"], m["coords"]
    d = np.sqrt(((x[:, None] - x[None]) ** 2).sum(-1))
    near = (d <= 6.0) & (d > 0)
    assert np.all(U[near] < W.sentinel_q(120))
    assert np.count_nonzero(L > U) > 0          # inconsistent pairs present

"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

Bit-exact in int32 (1/1024 A) and in the per-round mode; fp32 blocked results
on the 1/1024 grid are bit-exact too (every sum that can win is exact below
2^14 A), which is stricter than the stated fp32 gate of 1e-5 relative /
1e-4 A absolute.  That gate is exercised on off-grid inputs in
test_fp32_off_grid_within_tolerance.
"""
import numpy as np
import pytest

import blocked_floyd_warshall_gb300 as bsm
import oracle
from workloads import molecules as W

from gpu_util import dev, gpu_bounds, gpu_upper, host, same_bits, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    bsm.build()
    bsm.library()


def as_dtype(Uq, Lq, dtype):
    if dtype == "f32":
        return W.to_f32(Uq), W.to_f32(Lq)
    return Uq, Lq


SIZES_PERK = [1, 2, 3, 4, 5, 7, 31, 33, 64, 255, 256]
# the last 64-wide tile ends on every kind of 16-row stripe boundary: inside
# the first stripe (1, 2, 3, 5), on one (16, 48, 96 = 64 + 32), inside a later
# one (31, 63, 300 = 256 + 44)
SIZES_BLOCKED = [1, 2, 3, 5, 16, 31, 48, 63, 64, 65, 96, 127, 128, 129, 255, 256, 257, 300, 383,
                 385, 513]
# blocked-mode schedules: automatic, forced tile sizes, with and without look-ahead
SCHEDULES = {
    "auto": 0,
    "t64": bsm.BS_TILE_64,
    "t128": bsm.BS_TILE_128,
    "t64_serial": bsm.BS_TILE_64 | bsm.BS_NO_LOOKAHEAD,
    "t128_serial": bsm.BS_TILE_128 | bsm.BS_NO_LOOKAHEAD,
    "sym": bsm.BS_SYMMETRIC,
    "one": bsm.BS_ONE_LAUNCH,
    "one_sym": bsm.BS_ONE_LAUNCH | bsm.BS_SYMMETRIC,
    "pairs": bsm.BS_PAIRED_ROUNDS,
    "pairs_sym": bsm.BS_PAIRED_ROUNDS | bsm.BS_SYMMETRIC,
    "pairs64": bsm.BS_PAIRED_ROUNDS | bsm.BS_TILE_64,
}
# every algorithm: the blocked schedules and both per-round forms
ALGOS = dict(SCHEDULES, perk=bsm.BS_PERK, perk2=bsm.BS_PERK | bsm.BS_PERK_PAIRED)


@pytest.mark.parametrize("n", SIZES_PERK)
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("rule", ["closure", "literal"])
@pytest.mark.parametrize("form", ["plain", "paired"])
def test_per_round_matches_oracle(n, dtype, rule, form):
    """Both per-round forms: one round per pass (the plain reference mode) and
    two rounds per pass."""
    Uq, Lq = W.random_bounds(n, 1000 + n, p_known=0.3, p_bad=0.03)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    flags = bsm.BS_PERK | (bsm.BS_RULE_LITERAL if rule == "literal" else 0)
    if form == "paired":
        flags |= bsm.BS_PERK_PAIRED
    r = oracle.RULE_LITERAL if rule == "literal" else oracle.RULE_CLOSURE
    Uo, Lo = oracle.smooth(U0, L0, rule=r)
    Ug, Lg, ok = gpu_bounds(U0, L0, flags)
    assert ok
    assert same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n", SIZES_BLOCKED)
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("sched", sorted(SCHEDULES))
def test_blocked_matches_oracle(n, dtype, sched):
    Uq, Lq = W.random_bounds(n, 2000 + n, p_known=0.2, p_bad=0.02)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    Uo, Lo = oracle.smooth(U0, L0)
    Ug, Lg, ok = gpu_bounds(U0, L0, SCHEDULES[sched])
    assert ok
    assert same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n", [1, 2, 5, 63, 64, 65, 127, 129, 257, 300, 513])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("sched", ["auto", "t64", "t128", "t64_serial", "t128_serial", "one",
                                   "pairs", "pairs64"])
def test_symmetric_mode_matches_oracle(n, dtype, sched):
    """Half the tiles computed and mirrored: bit-identical to the oracle."""
    Uq, Lq = W.random_bounds(n, 2500 + n, p_known=0.2, p_bad=0.02)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    Uo, Lo = oracle.smooth(U0, L0)
    Ug, Lg, ok = gpu_bounds(U0, L0, SCHEDULES[sched] | bsm.BS_SYMMETRIC, ld=n + 4)
    assert ok
    assert same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n", [65, 300, 513])
@pytest.mark.parametrize("algo", ["t64", "t128", "one", "pairs", "pairs64"])
def test_symmetric_upper_only(n, algo):
    Uq, _ = W.random_bounds(n, 5500 + n, p_known=0.25)
    Uo = oracle.smooth_upper(Uq)
    Ug, ok = gpu_upper(Uq, SCHEDULES[algo] | bsm.BS_SYMMETRIC, ld=n + 1)
    assert ok and same_bits(Ug, Uo)


@pytest.mark.parametrize("n", [997, 1001, 1003])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("sched", ["auto", "sym", "t128", "one", "pairs", "pairs_sym", "pairs64"])
def test_blocked_tails_near_1000(n, dtype, sched):
    """Sizes around the n = 1000 chain with ragged last tiles (37, 41, 43 rows
    of 64; 101, 105, 107 of 128), a padded leading dimension n + 5 with
    canaries, every cell against the oracle."""
    Uq, Lq = W.random_bounds(n, 6100 + n, p_known=0.05, p_bad=0.005)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    Uo, Lo = oracle.smooth(U0, L0)
    Ug, Lg, ok = gpu_bounds(U0, L0, SCHEDULES[sched], ld=n + 5)
    assert ok
    assert same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n", [129, 300])
@pytest.mark.parametrize("sched", ["t64", "t128", "pairs", "pairs64"])
def test_blocked_asymmetric(n, sched):
    Uq, Lq = W.random_bounds(n, 3000 + n, p_known=0.3, p_bad=0.02, symmetric=False)
    Uo, Lo = oracle.smooth(Uq, Lq)
    Ug, Lg, ok = gpu_bounds(Uq, Lq, SCHEDULES[sched])
    assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n,ld,offset", [(130, 140, 0), (130, 133, 0), (257, 260, 1),
                                         (97, 101, 3), (200, 200, 1)])
@pytest.mark.parametrize("algo", ["t64", "t128", "perk", "perk2", "one", "pairs", "pairs64"])
def test_leading_dimension_and_misalignment(n, ld, offset, algo):
    """ld > n keeps the padding untouched; ld % 4 != 0 or a base not 16-byte
    aligned takes the scalar-IO instantiation with identical results."""
    Uq, Lq = W.random_bounds(n, 4000 + n, p_bad=0.02)
    U0, L0 = W.to_f32(Uq), W.to_f32(Lq)
    flags = ALGOS[algo]
    Uo, Lo = oracle.smooth(U0, L0)
    Ug, Lg, ok = gpu_bounds(U0, L0, flags, ld=ld, offset=offset)
    assert ok
    assert same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("n", [1, 5, 128, 129, 300, 513])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("algo", ["t64", "t128", "perk", "perk2", "one", "pairs", "pairs64"])
def test_upper_only(n, dtype, algo):
    Uq, _ = W.random_bounds(n, 5000 + n, p_known=0.25)
    U0 = W.to_f32(Uq) if dtype == "f32" else Uq
    Uo = oracle.smooth_upper(U0)
    Ug, ok = gpu_upper(U0, ALGOS[algo], ld=n + 3)
    assert ok and same_bits(Ug, Uo)


@pytest.mark.parametrize("n,pad", [(1, 4), (64, 4), (131, 4), (131, 1), (131, 5), (257, 3)])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_feasibility_count_and_mask(n, pad, dtype):
    """Rows of 16-byte multiples take the 4-cell path (with a tail when n is
    not a multiple of 4); others the 1-cell path.  Padding columns untouched."""
    Uq, Lq = W.random_bounds(n, 6000 + n, p_known=0.4, p_bad=0.05)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    Uo, Lo = oracle.smooth(U0, L0)
    ld = n + pad
    t = torch()
    U = dev(np.pad(Uo, ((0, 0), (0, pad))))
    L = dev(np.pad(Lo, ((0, 0), (0, pad))))
    mask = t.full((n, ld), 7, dtype=t.uint8, device="cuda")
    cnt = bsm.bs_check_feasible(U, L, n, ld, None, None, mask)
    assert cnt == oracle.count_infeasible(Uo, Lo)
    m = host(mask)
    assert np.array_equal(m[:, :n].astype(bool), Lo > Uo)
    assert np.all(m[:, n:] == 7)


def test_feasibility_count_example_c():
    """The worked example with 16 flags (closure) and 15 (printed rule, per round)."""
    U0 = np.full((4, 4), 100.0, np.float32)
    L0 = np.full((4, 4), 1.0, np.float32)
    np.fill_diagonal(U0, 0)
    np.fill_diagonal(L0, 0)
    for i, j, lo, hi in [(0, 1, 3, 4), (1, 2, 3, 4), (0, 2, 9, 10), (2, 3, 0.125, 0.25)]:
        U0[i, j] = U0[j, i] = hi
        L0[i, j] = L0[j, i] = lo
    for flags, expect in [(0, 16), (bsm.BS_PERK, 16), (bsm.BS_PERK | bsm.BS_RULE_LITERAL, 15)]:
        U, L = dev(U0), dev(L0)
        bsm.bs_smooth_bounds(U, L, flags=flags)
        assert bsm.bs_check_feasible(U, L) == expect


def off_grid(n, seed, p_bad, symmetric=True):
    """Bounds with values off the 1/1024 grid (fp32), optionally inverted pairs."""
    rng = np.random.default_rng(seed)
    Uq, Lq = W.random_bounds(n, seed, p_known=0.3, p_bad=p_bad, symmetric=symmetric)
    U0 = (Uq / 1024.0 + rng.random((n, n)) * 1e-3).astype(np.float32)
    L0 = np.maximum(Lq / 1024.0 - rng.random((n, n)) * 1e-3, 0).astype(np.float32)
    if symmetric:
        U0 = np.minimum(U0, U0.T)
        L0 = np.minimum(L0, L0.T)
    np.fill_diagonal(U0, 0)
    np.fill_diagonal(L0, 0)
    return U0, L0


@pytest.mark.parametrize("n,p_bad", [(300, 0.0), (300, 0.02), (700, 0.01)])
@pytest.mark.parametrize("sched", ["t64", "t128", "sym", "pairs", "pairs_sym", "pairs64"])
def test_fp32_off_grid_within_tolerance(n, p_bad, sched):
    """Off the 1/1024 grid fp32 sums round, so the schedule changes the last
    bits.  Against the fp64 oracle on the same fp32 inputs:
      * the stated gate: |g - o| <= 1e-4 A or <= 1e-5 |o|, every cell;
      * U: a computed upper bound is the fp32 sum of the edges of one path of
        at most n-1 edges, each add rounding to nearest, so
        |g - o| <= (n-1) 2^-24 o;
      * the L > U flags agree wherever |L - U| exceeds the tolerance."""
    U0, L0 = off_grid(n, 7000 + n, p_bad)
    Uo, Lo = oracle.smooth(U0.astype(np.float64), L0.astype(np.float64))
    Ug, Lg, ok = gpu_bounds(U0, L0, SCHEDULES[sched])
    assert ok
    for g, o in ((Ug, Uo), (Lg, Lo)):
        err = np.abs(g.astype(np.float64) - o)
        assert np.all((err <= 1e-4) | (err <= 1e-5 * np.abs(o)))
    assert np.all(np.abs(Ug - Uo) <= (n - 1) * 2.0 ** -24 * Uo + 1e-30)
    margin = np.abs(Lo - Uo)
    clear = margin > 2e-4 + 2e-5 * np.maximum(np.abs(Lo), np.abs(Uo))
    assert np.array_equal((Lg > Ug)[clear], (Lo > Uo)[clear])
    # the fp32 round-by-round oracle differs from fp64 by rounding only as well
    Uf, Lf = oracle.smooth(U0, L0)
    assert np.max(np.abs(Uf.astype(np.float64) - Uo)) <= np.max(Uo) * (n - 1) * 2.0 ** -24


def gamma(m):
    """Relative rounding bound of a sum of m + 1 fp32 terms, any order."""
    u = 2.0 ** -24
    m = np.maximum(m, 0).astype(np.float64)
    return m * u / (1 - m * u)


@pytest.mark.parametrize("n,p_bad,seed", [(300, 0.0, 1), (300, 0.02, 2), (700, 0.01, 3),
                                          (517, 0.005, 4)])
@pytest.mark.parametrize("sched", ["auto", "t64", "t128", "sym", "perk", "perk2", "pairs",
                                   "pairs_sym"])
def test_fp32_off_grid_per_cell_bound(n, p_bad, seed, sched):
    """Off the 1/1024 grid, every fp32 cell against the fp64 oracle, with a
    bound from the cell's own path (oracle provenance: edges h and summed
    |weight| M of a best path).  Every computed value is a rounded sum or
    difference of computed values and rounding is monotone, so
      U: U64 (1 - g(n-2)) <= Ug <= U64 (1 + g(hU - 1))
      L: L64 - g(hL - 1) M <= Lg <= L64 + g(n) (2 max L0 + 1)
    with g(m) = m u / (1 - m u), u = 2^-24 (the second L bound: a path that
    wins has no more u weight than twice its l weight).  Slack 1e-12 relative
    covers the oracle's own fp64 rounding."""
    U0, L0 = off_grid(n, 8000 + seed, p_bad)
    U64, L64, HU, HL, ML = oracle.smooth_track(U0.astype(np.float64), L0.astype(np.float64))
    flags = ALGOS[sched]
    Ug, Lg, ok = gpu_bounds(U0, L0, flags)
    assert ok
    Ug, Lg = Ug.astype(np.float64), Lg.astype(np.float64)
    eps = 1e-12
    assert np.all(Ug <= U64 * (1 + gamma(HU - 1)) * (1 + eps))
    assert np.all(Ug >= U64 * (1 - gamma(np.full_like(HU, n - 2))) * (1 - eps))
    assert np.all(Lg >= L64 - gamma(HL - 1) * ML * (1 + eps) - eps * ML)
    top = gamma(np.array(n)) * (2 * float(L0.max()) + 1)
    assert np.all(Lg <= L64 + top * (1 + eps))
    # the per-cell bound lies inside the stated gate (1e-4 A or 1e-5 relative)
    assert np.all((gamma(HU - 1) <= 1e-5) | (gamma(HU - 1) * U64 <= 1e-4))


# ------------------------------------------------------------------ edge cases


def edge_cases():
    """Degenerate inputs the method admits (each pair: U, L as Q10 int32)."""
    cases = {}
    n = 150
    # int32 at the precondition ceiling: unknown U = 2^30 - 1, long known bonds
    U, L = W.random_bounds(n, 9400, p_known=0.05, p_bad=0.01)
    U = np.where(U == W.sentinel_q(n), (1 << 30) - 1, U).astype(np.int32)
    big = np.random.default_rng(1).random((n, n)) < 0.02
    U = np.where(big & (U < (1 << 29)), U + (1 << 28), U).astype(np.int32)
    U = np.minimum(U, U.T)
    np.fill_diagonal(U, 0)
    cases["int32_ceiling"] = (U, L)
    # zero-length bonds: distinct atoms at the same place
    U, L = W.random_bounds(n, 9401, p_known=0.3)
    z = np.random.default_rng(2).random((n, n)) < 0.01
    z = z | z.T
    U = np.where(z, 0, U).astype(np.int32)
    L = np.where(z, 0, L).astype(np.int32)
    cases["zero_bonds"] = (U, L)
    # two disconnected molecules: no path between the halves
    U, L = W.blank_bounds(n)
    h = n // 2
    Ua, La = W.random_bounds(h, 9402, p_known=0.3)
    Ub, Lb = W.random_bounds(n - h, 9403, p_known=0.3)
    U[:h, :h], L[:h, :h] = Ua, La
    U[h:, h:], L[h:, h:] = Ub, Lb
    cases["disconnected"] = (U, L)
    # nothing known
    cases["all_unknown"] = W.blank_bounds(n)
    return cases


@pytest.mark.parametrize("case", sorted(edge_cases()))
@pytest.mark.parametrize("algo", ["t64", "t128", "perk", "perk2", "one", "pairs", "pairs64"])
def test_edge_cases(case, algo):
    Uq, Lq = edge_cases()[case]
    flags = ALGOS[algo]
    for U0, L0 in ((Uq, Lq), (W.to_f32(Uq), W.to_f32(Lq))):
        if case == "int32_ceiling" and U0.dtype == np.float32:
            continue                      # above 2^24 units the fp32 grid is not exact
        Uo, Lo = oracle.smooth(U0, L0)
        Ug, Lg, ok = gpu_bounds(U0, L0, flags)
        assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)
    if case == "all_unknown":
        np.testing.assert_array_equal(Uo, Uq.astype(Uo.dtype) / (1 if Uo.dtype == np.int32 else 1024))


@pytest.mark.parametrize("algo", ["t64", "t128", "perk", "perk2", "one", "pairs"])
def test_infinite_upper_bounds(algo):
    """fp32 U may be +inf for unknown pairs; inf + x = inf never wins."""
    Uq, Lq = W.random_bounds(200, 9500, p_known=0.1, p_bad=0.01)
    Uq[190:, :] = Lq[190:, :] = 0
    Uq[:, 190:] = Lq[:, 190:] = 0
    Uq[190:, :] = W.sentinel_q(200)              # atoms 190.. are constrained by nothing
    Uq[:, 190:] = W.sentinel_q(200)
    Lq[190:, :] = 1024
    Lq[:, 190:] = 1024
    np.fill_diagonal(Uq, 0)
    np.fill_diagonal(Lq, 0)
    U0, L0 = W.to_f32(Uq), W.to_f32(Lq)
    U0 = np.where(Uq == W.sentinel_q(200), np.float32(np.inf), U0).astype(np.float32)
    Uo, Lo = oracle.smooth(U0, L0)
    assert np.isinf(Uo).any()
    Ug, Lg, ok = gpu_bounds(U0, L0, ALGOS[algo])
    assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.mark.parametrize("flags", [0, bsm.BS_ONE_LAUNCH])
def test_batch_beyond_grid_limit(flags):
    """More molecules than a grid's z dimension holds (65535): launches are
    split in chunks; every molecule still matches a single-molecule call."""
    t = torch()
    B, n = 70000, 4
    rng = np.random.default_rng(9600)
    base = [W.random_bounds(n, 9600 + s, p_known=0.8, p_bad=0.1) for s in range(7)]
    pick = rng.integers(0, 7, B)
    Uq = np.stack([base[p][0] for p in pick])
    Lq = np.stack([base[p][1] for p in pick])
    U, L = dev(W.to_f32(Uq)), dev(W.to_f32(Lq))
    bsm.bs_smooth_bounds_batched(U, L, flags=flags)
    Ug, Lg = host(U), host(L)
    ref = [oracle.smooth(W.to_f32(u), W.to_f32(l)) for u, l in base]
    for b in (0, 1, 65534, 65535, 65536, B - 1) + tuple(rng.integers(0, B, 50)):
        assert same_bits(Ug[b], ref[pick[b]][0]) and same_bits(Lg[b], ref[pick[b]][1])
    counts = bsm.bs_check_feasible_noalloc(U[:4096], L[:4096])
    assert counts == [oracle.count_infeasible(*ref[p]) for p in pick[:4096]]
    del t


# ------------------------------------------------------------------ benchmark molecules


@pytest.mark.parametrize("idx", [0, 1])
@pytest.mark.parametrize("algo", ["blocked", "perk", "symmetric", "one"])
def test_chain_configs(idx, algo):
    m = W.make_config(idx)
    flags = {"blocked": 0, "perk": bsm.BS_PERK, "symmetric": bsm.BS_SYMMETRIC,
             "one": bsm.BS_ONE_LAUNCH}[algo]
    for U0, L0 in ((W.to_f32(m["U"]), W.to_f32(m["L"])), (m["U"], m["L"])):
        Uo, Lo = oracle.smooth(U0, L0)
        Ug, Lg, ok = gpu_bounds(U0, L0, flags)
        assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)
        assert oracle.count_infeasible(Uo, Lo) == 0


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_mid_size_default_schedule(dtype):
    """n = 2000 (ragged against 64-wide tiles) on the default schedule, which
    at this size is 64-wide tiles with look-ahead: full matrix vs the oracle."""
    Uq, Lq = W.random_bounds(2000, 2024, p_known=0.1, p_bad=0.001)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    Uo, Lo = oracle.smooth(U0, L0)
    Ug, Lg, ok = gpu_bounds(U0, L0)
    assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)


@pytest.fixture(scope="module")
def globule4096():
    m = W.make_config(2)
    Uo, Lo = oracle.smooth(m["U"], m["L"])          # int32, all 4096 rounds
    return m, Uo, Lo


@pytest.mark.parametrize("sched", ["auto", "t64", "t128_serial", "sym", "pairs", "pairs_sym",
                                   "pairs64"])
def test_globule_4096_int32_blocked(globule4096, sched):
    m, Uo, Lo = globule4096
    Ug, Lg, ok = gpu_bounds(m["U"], m["L"], SCHEDULES[sched])
    assert ok and same_bits(Ug, Uo) and same_bits(Lg, Lo)
    U, L = dev(Ug), dev(Lg)
    assert bsm.bs_check_feasible(U, L) == oracle.count_infeasible(Uo, Lo) > 0


def test_globule_4096_fp32_blocked_and_per_round(globule4096):
    m, Uo, Lo = globule4096
    U0, L0 = W.to_f32(m["U"]), W.to_f32(m["L"])
    expect_flags = oracle.count_infeasible(Uo, Lo)
    for flags in (0, bsm.BS_PERK, bsm.BS_PERK | bsm.BS_PERK_PAIRED):
        Ug, Lg, ok = gpu_bounds(U0, L0, flags)
        assert ok
        # fp32 on the grid equals int32 / 1024 exactly
        assert np.array_equal(Ug * 1024, Uo.astype(np.float32))
        assert np.array_equal(Lg * 1024, Lo.astype(np.float32))
        assert bsm.bs_check_feasible(dev(Ug), dev(Lg)) == expect_flags


@pytest.mark.parametrize("sched", ["auto", "t128", "sym", "one", "one_sym", "pairs", "pairs_sym",
                                   "pairs64"])
def test_batched_chains(sched):
    """Batch of 256 molecules n=512 in one call; every 32nd molecule against the
    oracle, all molecules against a per-molecule GPU call."""
    m = W.make_config(3)
    B, n = m["batch"], m["n"]
    U0, L0 = W.to_f32(m["U"]), W.to_f32(m["L"])
    U, L = dev(U0), dev(L0)
    bsm.bs_smooth_bounds_batched(U, L, flags=SCHEDULES[sched])
    Ug, Lg = host(U), host(L)
    for b in range(0, B, 32):
        Uo, Lo = oracle.smooth(U0[b], L0[b])
        assert same_bits(Ug[b], Uo) and same_bits(Lg[b], Lo)
    for b in range(B):
        Us, Ls, _ = gpu_bounds(U0[b], L0[b])
        assert same_bits(Ug[b], Us) and same_bits(Lg[b], Ls)
    del n


@pytest.mark.parametrize("n,B", [(200, 3), (300, 4), (257, 12), (130, 40)])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("sched", ["auto", "sym", "one", "pairs64"])
def test_batched_small_molecules(n, B, dtype, sched):
    """Small batches of small molecules: the launches take the strip forms
    (four or two CTAs per tile) or the 256-thread form depending on the
    tiles per SM; every molecule against the oracle."""
    mols = [W.random_bounds(n, 8100 + 7 * B + b, p_bad=0.01) for b in range(B)]
    Uq = np.stack([m[0] for m in mols])
    Lq = np.stack([m[1] for m in mols])
    U0, L0 = (W.to_f32(Uq), W.to_f32(Lq)) if dtype == "f32" else (Uq, Lq)
    U, L = dev(U0), dev(L0)
    bsm.bs_smooth_bounds_batched(U, L, flags=SCHEDULES[sched])
    Ug, Lg = host(U), host(L)
    for b in range(B):
        Uo, Lo = oracle.smooth(U0[b], L0[b])
        assert same_bits(Ug[b], Uo) and same_bits(Lg[b], Lo)


@pytest.mark.parametrize("seed", range(6))
def test_small_schedules_random_sizes(seed):
    """Random sizes and batches across the small-matrix schedules (the
    merged look-ahead below half an SM's worth of rest tiles, the tight one
    up to an SM's worth, then the loose one), random dtype and symmetry,
    every molecule against the oracle."""
    rng = np.random.default_rng(7100 + seed)
    n = int(rng.integers(130, 1000))
    B = int(rng.integers(1, 4))
    dtype = "f32" if rng.integers(2) else "i32"
    flags = bsm.BS_SYMMETRIC if rng.integers(2) else 0
    mols = [W.random_bounds(n, 7200 + 10 * seed + b, p_known=0.25, p_bad=0.01) for b in range(B)]
    Uq = np.stack([m[0] for m in mols])
    Lq = np.stack([m[1] for m in mols])
    U0, L0 = (W.to_f32(Uq), W.to_f32(Lq)) if dtype == "f32" else (Uq, Lq)
    U, L = dev(U0), dev(L0)
    bsm.bs_smooth_bounds_batched(U, L, flags=flags)
    Ug, Lg = host(U), host(L)
    for b in range(B):
        Uo, Lo = oracle.smooth(U0[b], L0[b])
        assert same_bits(Ug[b], Uo) and same_bits(Lg[b], Lo), (n, B, dtype, flags, b)


def test_batched_per_round_and_strided():
    """Per-round mode and a batch stride larger than one molecule."""
    B, n, ld = 5, 70, 72
    stride = n * ld + 16
    t = torch()
    Us = [W.random_bounds(n, 8000 + b, p_bad=0.02) for b in range(B)]
    Ubuf = t.full((B * stride,), -1.0, dtype=t.float32, device="cuda")
    Lbuf = t.full((B * stride,), -1.0, dtype=t.float32, device="cuda")
    for b, (uq, lq) in enumerate(Us):
        Ubuf[b * stride: b * stride + n * ld].view(n, ld)[:, :n] = dev(W.to_f32(uq))
        Lbuf[b * stride: b * stride + n * ld].view(n, ld)[:, :n] = dev(W.to_f32(lq))
    for flags in (bsm.BS_PERK, bsm.BS_PERK | bsm.BS_PERK_PAIRED, 0, bsm.BS_TILE_128,
                  bsm.BS_ONE_LAUNCH):
        U, L = Ubuf.clone(), Lbuf.clone()
        bsm.bs_smooth_bounds_batched(U, L, n, ld, stride, B, None, bsm.BS_FP32 | flags)
        Uh, Lh = host(U), host(L)
        for b, (uq, lq) in enumerate(Us):
            Uo, Lo = oracle.smooth(W.to_f32(uq), W.to_f32(lq))
            blk = slice(b * stride, b * stride + n * ld)
            assert same_bits(Uh[blk].reshape(n, ld)[:, :n], Uo)
            assert same_bits(Lh[blk].reshape(n, ld)[:, :n], Lo)
            assert np.all(Uh[blk].reshape(n, ld)[:, n:] == -1.0)
            assert np.all(Uh[b * stride + n * ld: (b + 1) * stride] == -1.0)


@pytest.fixture(scope="module")
def globule16384():
    """n = 16384 globule and the oracle's shortest-path rows for 64 sources:
    both sides of several 128-tile boundaries and 52 seeded random rows."""
    m = W.make_config(4)
    n = m["n"]
    edges = [0, 1, 127, 128, 4097, 8191, 8192, 12000, 16255, 16256, n - 2, n - 1]
    rnd = np.random.default_rng(64).choice(n, 64, replace=False)
    rows = np.array(sorted(set(edges) | set(rnd.tolist())))[:64]
    Ur, Lr = oracle.closure_rows(m["U"], m["L"], rows)
    return m, rows, Ur, Lr


def upper_bellman_holds(U0q, Ug, block=32):
    """Every cell of the smoothed upper bound against the shortest-path
    (Bellman) equations of the bound graph: U[j,j] = 0 and, for i != j,
    U[i,j] = min(U0[i,j], min over the known neighbours k of i of
    U0[i,k] + U[k,j]).  With positive weights the distances are the only
    solution, so this checks all n^2 cells exactly without an n^3 oracle.
    Plain PyTorch on the device, in float64 on Q10 values (exact)."""
    t = torch()
    n = U0q.shape[0]
    sent = W.sentinel_q(n)
    known = (U0q < sent) & ~np.eye(n, dtype=bool)
    deg = known.sum(1)
    kmax = int(deg.max())
    nbr = np.zeros((n, kmax), np.int64)
    wgt = np.full((n, kmax), np.inf)
    for i in range(n):
        ks = np.nonzero(known[i])[0]
        nbr[i, :len(ks)] = ks
        wgt[i, :len(ks)] = U0q[i, ks]
    nbr_d, wgt_d = t.from_numpy(nbr).cuda(), t.from_numpy(wgt).cuda()
    Ud = Ug.to(t.float64) * 1024
    U0d = t.from_numpy(U0q.astype(np.float64)).cuda()
    for i0 in range(0, n, block):
        i1 = min(n, i0 + block)
        cand = (wgt_d[i0:i1, :, None] + Ud[nbr_d[i0:i1]]).min(dim=1).values
        rhs = t.minimum(U0d[i0:i1], cand)
        rows = t.arange(i0, i1, device=rhs.device)
        rhs[rows - i0, rows] = 0
        if not bool((rhs == Ud[i0:i1]).all()):
            return False
    return True


def lower_bellman_holds(U0q, L0q, Ug, Lg, block=32):
    """Every cell of the smoothed lower bound against the shortest-path
    equations of the doubled bound graph (-L[i,j] is the distance from i's
    first copy to j's second), given the smoothed U:
      L[i,j] = max(L0[i,j], max_k L[k,j] - U0[i,k], max_b L0[i,b] - U[b,j])
    over the known neighbours k, b of i.  Pairs left out cannot win here:
    an unknown pair's term L0[i,b] - U[b,j] <= 1 A <= L0[i,j] (every
    off-diagonal L0 is at least the unknown value, asserted), and an unknown
    u edge leaves L[k,j] - U0[i,k] < 0 since L <= U < U0 there.  For fixed U
    the equations are a shortest-path problem with positive weights, so
    their solution is unique.  Plain PyTorch float64 on Q10 values."""
    t = torch()
    n = U0q.shape[0]
    sent = W.sentinel_q(n)
    off = ~np.eye(n, dtype=bool)
    unknown_l = int(L0q[off & (U0q >= sent)].max())
    assert int(L0q[off].min()) >= unknown_l
    known = (U0q < sent) & off
    kmax = int(known.sum(1).max())
    nbr = np.zeros((n, kmax), np.int64)
    wu = np.full((n, kmax), np.inf)       # U0[i, k]
    wl = np.full((n, kmax), -np.inf)      # L0[i, b]
    for i in range(n):
        ks = np.nonzero(known[i])[0]
        nbr[i, :len(ks)] = ks
        wu[i, :len(ks)] = U0q[i, ks]
        wl[i, :len(ks)] = L0q[i, ks]
    nbr_d = t.from_numpy(nbr).cuda()
    wu_d, wl_d = t.from_numpy(wu).cuda(), t.from_numpy(wl).cuda()
    Ud = Ug.to(t.float64) * 1024
    Ld = Lg.to(t.float64) * 1024
    L0d = t.from_numpy(L0q.astype(np.float64)).cuda()
    for i0 in range(0, n, block):
        i1 = min(n, i0 + block)
        nb = nbr_d[i0:i1]
        via_u = (Ld[nb] - wu_d[i0:i1, :, None]).max(dim=1).values
        via_l = (wl_d[i0:i1, :, None] - Ud[nb]).max(dim=1).values
        rhs = t.maximum(L0d[i0:i1], t.maximum(via_u, via_l))
        if not bool((rhs == Ld[i0:i1]).all()):
            return False
    return True


@pytest.mark.parametrize("sched", ["auto", "sym"])
def test_globule_16384_sampled_rows(globule16384, sched):
    """n = 16384, fp32, blocked, as timed by the benchmark: 64 sampled rows
    of U and L against the oracle's shortest-path rows, every cell of U and
    of L against the shortest-path equations, plus properties of every cell."""
    m, rows, Ur, Lr = globule16384
    t = torch()
    U, L = dev(W.to_f32(m["U"])), dev(W.to_f32(m["L"]))
    bsm.bs_smooth_bounds(U, L, flags=SCHEDULES[sched])
    t.cuda.synchronize()
    Ug = U[t.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64) * 1024
    Lg = L[t.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64) * 1024
    assert np.array_equal(Ug, Ur) and np.array_equal(Lg, Lr)
    # every cell of U and L: the shortest-path equations of the bound graph
    assert upper_bellman_holds(m["U"], U)
    assert lower_bellman_holds(m["U"], m["L"], U, L)
    # every cell: symmetric, consistent (no flags), diagonal zero
    assert bool((U == U.T).all()) and bool((L == L.T).all())
    assert bsm.bs_check_feasible(U, L) == 0
    assert bool((t.diagonal(U) == 0).all()) and bool((t.diagonal(L) == 0).all())
    # the generating coordinates lie inside every smoothed bound (sampled rows)
    x = m["coords"]
    d = np.sqrt(((x[rows][:, None] - x[None]) ** 2).sum(-1)) * 1024
    assert np.all(Lg <= d + 1e-6) and np.all(d <= Ug + 1e-6)


@pytest.mark.parametrize("sched", ["auto", "sym"])
def test_globule_16384_every_cell_against_oracle(globule16384, sched):
    """n = 16384, fp32, blocked, as timed by the benchmark, against the
    oracle's own full result: every cell of U and L bit for bit, through the
    SHA-256 digests of the oracle's output that tests/golden/
    make_oracle_digest.py stored (whole matrices and blocks of 128 rows).  The
    input's digests are checked first, so a generator that drew a different
    molecule on this host is reported as such."""
    import json
    import os
    from golden.make_oracle_digest import digest
    m = globule16384[0]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "globule16384_oracle.json")
    with open(path) as f:
        ref = json.load(f)
    U0, L0 = W.to_f32(m["U"]), W.to_f32(m["L"])
    assert ref["n"] == m["n"]
    assert digest(U0)["sha256"] == ref["input"]["U"]["sha256"], "generator drew another input"
    assert digest(L0)["sha256"] == ref["input"]["L"]["sha256"], "generator drew another input"
    t = torch()
    U, L = dev(U0), dev(L0)
    del U0, L0
    bsm.bs_smooth_bounds(U, L, flags=SCHEDULES[sched])
    t.cuda.synchronize()
    for name, mat in (("U", U), ("L", L)):
        got = digest(host(mat))
        bad = [b for b, (x, y) in enumerate(zip(got["blocks"], ref["output"][name]["blocks"]))
               if x != y]
        assert not bad, "%s differs from the oracle in row blocks %s" % (name, bad[:16])
        assert got["sha256"] == ref["output"][name]["sha256"]
    assert bsm.bs_check_feasible(U, L) == ref["flags"]


# ------------------------------------------------------------------ checks and errors


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_validate_flag(dtype):
    Uq, Lq = W.random_bounds(40, 9000, p_bad=0.02)
    U0, L0 = as_dtype(Uq, Lq, dtype)
    U, L = dev(U0), dev(L0)
    bsm.bs_smooth_bounds(U, L, flags=bsm.BS_VALIDATE)        # valid input passes
    bad_diag = U0.copy()
    bad_diag[3, 3] = 1
    bad_neg = L0.copy()
    bad_neg[2, 5] = -1
    cases = [(bad_diag, L0, bsm.BS_ERR_INPUT), (U0, bad_neg, bsm.BS_ERR_INPUT)]
    if dtype == "f32":
        bad_nan = L0.copy()
        bad_nan[1, 2] = np.nan
        bad_inf = L0.copy()
        bad_inf[1, 2] = np.inf
        cases += [(U0, bad_nan, bsm.BS_ERR_INPUT), (U0, bad_inf, bsm.BS_ERR_INPUT)]
    else:
        big = U0.copy()
        big[0, 1] = 1 << 30
        cases += [(big, L0, bsm.BS_ERR_RANGE)]
    for u, l, code in cases:
        with pytest.raises(bsm.BSError) as e:
            bsm.bs_smooth_bounds(dev(u), dev(l), flags=bsm.BS_VALIDATE)
        assert e.value.status == code


def test_symmetric_flag_checks():
    """BS_VALIDATE rejects asymmetric input in symmetric mode."""
    Uq, Lq = W.random_bounds(40, 9100, p_bad=0.02, symmetric=False)
    U, L = dev(W.to_f32(Uq)), dev(W.to_f32(Lq))
    with pytest.raises(bsm.BSError) as e:
        bsm.bs_smooth_bounds(U, L, flags=bsm.BS_SYMMETRIC | bsm.BS_VALIDATE)
    assert e.value.status == bsm.BS_ERR_INPUT
    Us, Ls = W.random_bounds(40, 9101, p_bad=0.02)
    bsm.bs_smooth_bounds(dev(W.to_f32(Us)), dev(W.to_f32(Ls)),
                         flags=bsm.BS_SYMMETRIC | bsm.BS_VALIDATE)


@pytest.mark.parametrize("sched,n", [("t64", 300), ("t128", 300), ("sym", 300), ("perk", 300),
                                     ("auto", 1000), ("one", 300), ("pairs", 1000)])
def test_cuda_graph_capture_and_replay(sched, n):
    """A smoothing captured into a CUDA graph (look-ahead fork and join
    included) replays to the same result, twice, on fresh inputs.  n = 1000
    has more rest tiles than SMs: captured, it takes the order in which the
    rest of each round waits for the next block row and column."""
    t = torch()
    flags = ALGOS[sched]
    Uq, Lq = W.random_bounds(n, 9300, p_bad=0.02)
    U0, L0 = dev(W.to_f32(Uq)), dev(W.to_f32(Lq))
    Uo, Lo = oracle.smooth(W.to_f32(Uq), W.to_f32(Lq))
    U, L = U0.clone(), L0.clone()
    bsm.bs_smooth_bounds(U, L, flags=flags)          # first call on the device: set-up
    t.cuda.synchronize()
    s = t.cuda.Stream()
    g = t.cuda.CUDAGraph()
    U.copy_(U0)
    L.copy_(L0)
    t.cuda.synchronize()
    with t.cuda.graph(g, stream=s):
        bsm.bs_smooth_bounds(U, L, flags=flags)
    for _ in range(2):
        U.copy_(U0)
        L.copy_(L0)
        g.replay()
        t.cuda.synchronize()
        assert same_bits(host(U), Uo) and same_bits(host(L), Lo)


@pytest.mark.parametrize("n", [700, 1000, 2000])
def test_concurrent_calls_on_own_streams(n):
    """Three host threads smooth three molecules at once, each on its own
    stream (each call takes its own look-ahead stream and events); then work
    queued on each caller's stream after the call sees the finished result
    (the look-ahead stream is joined back into the caller's stream)."""
    import threading
    t = torch()
    mols = [W.random_bounds(n, 9500 + b, p_bad=0.01) for b in range(3)]
    want = [oracle.smooth(W.to_f32(u), W.to_f32(l)) for u, l in mols]
    bsm.bs_smooth_bounds(dev(W.to_f32(mols[0][0])), dev(W.to_f32(mols[0][1])))   # set-up
    t.cuda.synchronize()
    streams = [t.cuda.Stream() for _ in mols]
    bufs = [(dev(W.to_f32(u)), dev(W.to_f32(l))) for u, l in mols]
    outs = [(t.empty_like(u), t.empty_like(l)) for u, l in bufs]
    errors = []

    def work(b):
        try:
            with t.cuda.stream(streams[b]):
                U, L = bufs[b]
                bsm.bs_smooth_bounds(U, L, stream=streams[b])
                outs[b][0].copy_(U)          # queued after the call on the same stream
                outs[b][1].copy_(L)
        except Exception as e:               # reported below, in the test thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(b,)) for b in range(len(mols))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for b, s in enumerate(streams):
        s.synchronize()
        assert same_bits(host(outs[b][0]), want[b][0]) and same_bits(host(outs[b][1]), want[b][1])


def test_literal_rule_rejected_in_blocked_mode():
    U, L = dev(np.zeros((4, 4), np.float32)), dev(np.zeros((4, 4), np.float32))
    with pytest.raises(bsm.BSError) as e:
        bsm.bs_smooth_bounds(U, L, flags=bsm.BS_RULE_LITERAL)
    assert e.value.status == bsm.BS_ERR_ARG


def test_empty_and_launch_counting():
    t = torch()
    U = t.zeros((0, 0), dtype=t.float32, device="cuda")
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(U, U.clone())
    assert bsm.bs_launch_count() == before
    Uq, Lq = W.random_bounds(300, 1, p_bad=0.01)
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq)), dev(W.to_f32(Lq)),
                         flags=bsm.BS_TILE_128 | bsm.BS_NO_LOOKAHEAD)
    assert bsm.bs_launch_count() - before == 3 * 3        # three phases x three block rounds
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq)), dev(W.to_f32(Lq)), flags=bsm.BS_TILE_64)
    # 5 block rounds: 5 x (phase 1, phase 2); 9 rest tiles, fewer than half
    # the SMs: phase 3 of rounds 0..3 is one launch without the next
    # diagonal tile (phase 1 of the next round takes it), then the last round
    assert bsm.bs_launch_count() - before == 5 + 5 + 4 + 1
    before = bsm.bs_launch_count()
    Ul, Ll = dev(W.to_f32(Uq)), dev(W.to_f32(Lq))
    bsm.bs_smooth_bounds(Ul, Ll, flags=bsm.BS_PERK)
    # the plain per-round mode: a pass and a row/column launch per round
    assert bsm.bs_launch_count() - before == 2 * 300
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq)), dev(W.to_f32(Lq)),
                         flags=bsm.BS_PERK | bsm.BS_PERK_PAIRED)
    # two rounds per pass: 150 passes, each with its row/column launch
    assert bsm.bs_launch_count() - before == 2 * 150
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq)), dev(W.to_f32(Lq)), flags=bsm.BS_ONE_LAUNCH)
    # the one-launch form: a single kernel for the whole smoothing
    assert bsm.bs_launch_count() - before == 1
    assert bsm.bs_one_launch_cluster() in (8, 16)
    Uq7, Lq7 = W.random_bounds(700, 1, p_bad=0.01)
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq7)), dev(W.to_f32(Lq7)), flags=bsm.BS_TILE_64)
    # 11 block rounds, 81 rest tiles: phase 3 split in two for rounds 0..9
    assert bsm.bs_launch_count() - before == 11 + 11 + 10 * 2 + 1
    before = bsm.bs_launch_count()
    bsm.bs_smooth_bounds(dev(W.to_f32(Uq)), dev(W.to_f32(Lq)),
                         flags=bsm.BS_TILE_64 | bsm.BS_NO_LOOKAHEAD)
    assert bsm.bs_launch_count() - before == 5 * 3


def test_profile_records_every_launch():
    Uq, Lq = W.random_bounds(300, 2, p_bad=0.01)
    U, L = dev(W.to_f32(Uq)), dev(W.to_f32(Lq))
    bsm.bs_profile_begin()
    bsm.bs_smooth_bounds(U, L, flags=bsm.BS_TILE_128)
    p = bsm.bs_profile_end()
    # rounds 0, 1: phase 3 split into the rest (caller's stream) and the next
    # block row and column (look-ahead stream)
    assert [p[k]["launches"] for k in bsm.PHASES] == [0, 3, 3, 3, 2, 0]
    assert p["phase3"]["ms"] > 0 and p["phase3_next"]["ms"] > 0
    # block rounds in pairs: on the caller's stream the pair's bulk (no tile at
    # nb = 3), the rest of block row and column 0 and the odd last round
    # whole; on the look-ahead stream the next block row and column, the near
    # ones and the corner tiles
    bsm.bs_profile_begin()
    bsm.bs_smooth_bounds(U, L, flags=bsm.BS_PAIRED_ROUNDS)
    p = bsm.bs_profile_end()
    assert [p[k]["launches"] for k in bsm.PHASES] == [0, 3, 3, 2, 3, 0]
    assert p["phase3"]["ms"] > 0 and p["phase3_next"]["ms"] > 0
    # 64-wide tiles, few rest tiles: phase 3 of each round but the last is
    # one launch on the caller's stream, beside phase 1 of the next round
    bsm.bs_profile_begin()
    bsm.bs_smooth_bounds(U, L, flags=bsm.BS_TILE_64)
    p = bsm.bs_profile_end()
    assert [p[k]["launches"] for k in bsm.PHASES] == [0, 5, 5, 5, 0, 0]
    # the one-launch form: its single kernel, in its own category
    bsm.bs_profile_begin()
    bsm.bs_smooth_bounds(U, L, flags=bsm.BS_ONE_LAUNCH)
    p = bsm.bs_profile_end()
    assert [p[k]["launches"] for k in bsm.PHASES] == [0, 0, 0, 0, 0, 1]
    assert p["one_launch"]["ms"] > 0

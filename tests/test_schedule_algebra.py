"""CPU checks of the identities the GPU schedules rest on (no GPU, no CUDA
code): plain Python on small integer and on-grid fp32 matrices, compared
with the oracle.

1. Two rounds per pass (per-round mode).  Round k+1's operands -- row k+1,
   column k+1 and cell (k+1,k+1) after round k -- formed by each cell from
   values before round k, then both rounds on the cell, give exactly the two
   oracle rounds; rows and columns k, k+1 themselves follow the same
   expressions with the four corner cells as they were before the pass.
2. The pre-update row sub-panel (phase 1 on a cluster).  With D the closure
   of a diagonal block, C = C0 + C0 D its column sub-panel and R = R0 + D R0
   its row sub-panel (min-plus sums and products of the doubled bound
   graph), the update of the rest, C R, equals C R0.
3. The symmetric schedule.  With symmetric inputs, computing only the tiles
   on and above the diagonal -- phase 2 takes, for each block column j, the
   panel tile on the upper side ((K,j) for j > K as a row panel, (j,K) for
   j < K as a column panel) and stores it also transposed; phase 3 stores
   its tiles once -- and writing the lower triangle as the transpose of the
   upper one at the end gives the oracle's result, even with the lower
   triangle poisoned at the start: no step reads a stale tile below the
   diagonal.
4. Launch lists and barrier phases.  The library's schedules -- block rounds
   in pairs, one round per pass (loose, tight, merged look-ahead) and the
   one-launch form's cluster-barrier phases -- written as lists of launches
   with their streams and events: whatever may run side by side touches
   disjoint tiles, every tile takes every round once and in order, and
   running them gives the oracle's result.
"""
import numpy as np
import pytest

import oracle
from workloads import molecules as W


# ---------------------------------------------------------------- one round

def one_round(u, l, uik, lik, ukj, lkj, lkk, closure, T):
    """Round k on cell (i,j) (GPU Gems 2 ch. 43, section 2's rules, upper
    first; the lower column raised by the closure rule or taken as printed)."""
    lc = max(lik, T(lkk - uik)) if closure else lik
    return min(u, T(uik + ukj)), max(l, max(T(lkj - uik), T(lc - ukj)))


def two_rounds(u, l, row_i, col_j, corners, closure, T):
    """Rounds k and k+1 on cell (i,j) from values before round k.
    row_i: U, L at (i,k), (i,k+1); col_j: U, L at (k,j), (k+1,j);
    corners: U, L at (k,k), (k,k+1), (k+1,k), (k+1,k+1)."""
    (uik, lik, uik1, lik1), (ukj, lkj, uk1j, lk1j) = row_i, col_j
    (_, lkk), (ukk1, lkk1), (uk1k, lk1k), (uk1k1, lk1k1) = corners
    u, l = one_round(u, l, uik, lik, ukj, lkj, lkk, closure, T)
    uik1, lik1 = one_round(uik1, lik1, uik, lik, ukk1, lkk1, lkk, closure, T)
    uk1j, lk1j = one_round(uk1j, lk1j, uk1k, lk1k, ukj, lkj, lkk, closure, T)
    _, l11 = one_round(uk1k1, lk1k1, uk1k, lk1k, ukk1, lkk1, lkk, closure, T)
    return one_round(u, l, uik1, lik1, uk1j, lk1j, l11, closure, T)


def smooth_two_per_pass(U, L, closure, step=None):
    """Every pair of rounds as one pass, every value from before the pass
    (`step`: the two-round cell update, two_rounds unless a test plants a
    mistake)."""
    step = step or two_rounds
    U, L = U.copy(), L.copy()
    T = U.dtype.type
    n = U.shape[0]
    k = 0
    while k + 1 < n:
        k1 = k + 1
        U0, L0 = U.copy(), L.copy()
        corners = [(U0[a, b], L0[a, b]) for a, b in ((k, k), (k, k1), (k1, k), (k1, k1))]
        for i in range(n):
            for j in range(n):
                row_i = (U0[i, k], L0[i, k], U0[i, k1], L0[i, k1])
                col_j = (U0[k, j], L0[k, j], U0[k1, j], L0[k1, j])
                U[i, j], L[i, j] = step(U0[i, j], L0[i, j], row_i, col_j, corners, closure, T)
        k += 2
    if k < n:
        U0, L0 = U.copy(), L.copy()
        for i in range(n):
            for j in range(n):
                U[i, j], L[i, j] = one_round(U0[i, j], L0[i, j], U0[i, k], L0[i, k], U0[k, j],
                                             L0[k, j], L0[k, k], closure, T)
    return U, L


@pytest.mark.parametrize("n", [1, 2, 3, 6, 9, 14])
@pytest.mark.parametrize("dtype", ["i32", "f32"])
@pytest.mark.parametrize("closure", [True, False])
def test_two_rounds_per_pass_equal_two_rounds(n, dtype, closure):
    Uq, Lq = W.random_bounds(n, 4400 + n, p_known=0.3, p_bad=0.05)
    U0, L0 = (W.to_f32(Uq), W.to_f32(Lq)) if dtype == "f32" else (Uq, Lq)
    Uo, Lo = oracle.smooth(U0, L0, rule=oracle.RULE_CLOSURE if closure else oracle.RULE_LITERAL)
    Ug, Lg = smooth_two_per_pass(U0, L0, closure)
    assert np.array_equal(Ug.view(np.int32), Uo.view(np.int32))
    assert np.array_equal(Lg.view(np.int32), Lo.view(np.int32))


def test_two_rounds_per_pass_catches_a_wrong_operand():
    """Planted mistake: round k+1 taking row k+1 from before round k."""
    n = 9
    Uq, Lq = W.random_bounds(n, 4499, p_known=0.5, p_bad=0.05)
    Uo, Lo = oracle.smooth(Uq, Lq)

    def wrong(u, l, row_i, col_j, corners, closure, T):
        (uik, lik, uik1, lik1), (ukj, lkj, uk1j, lk1j) = row_i, col_j
        (_, lkk), (ukk1, lkk1), (uk1k, lk1k), (uk1k1, lk1k1) = corners
        u, l = one_round(u, l, uik, lik, ukj, lkj, lkk, closure, T)
        uik1, lik1 = one_round(uik1, lik1, uik, lik, ukk1, lkk1, lkk, closure, T)
        _, l11 = one_round(uk1k1, lk1k1, uk1k, lk1k, ukk1, lkk1, lkk, closure, T)
        return one_round(u, l, uik1, lik1, uk1j, lk1j, l11, closure, T)

    Ug, Lg = smooth_two_per_pass(Uq, Lq, True, step=wrong)
    assert not (np.array_equal(Ug, Uo) and np.array_equal(Lg, Lo))


# ---------------------------------------------------------------- doubled-graph products

def product(A, B):
    """A (x) B in the doubled bound graph: the phase-3 rules with A the column
    operand and B the row operand; pairs (U, L) of integer arrays."""
    AU, AL = A
    BU, BL = B
    U = (AU[:, :, None] + BU[None, :, :]).min(axis=1)
    L = np.maximum((BL[None, :, :] - AU[:, :, None]).max(axis=1),
                   (AL[:, :, None] - BU[None, :, :]).max(axis=1))
    return U, L


def plus(X, Y):
    return np.minimum(X[0], Y[0]), np.maximum(X[1], Y[1])


@pytest.mark.parametrize("seed", range(8))
def test_pre_update_row_panel_gives_the_same_product(seed):
    rng = np.random.default_rng(4500 + seed)
    s, r, c = 6, 9, 7          # block width, column sub-panel rows, row sub-panel columns
    Uq, Lq = W.random_bounds(s, 4600 + seed, p_known=0.4, p_bad=0.05)
    D = tuple(a.astype(np.int64) for a in oracle.smooth(Uq, Lq))          # closed block
    big = 1 << 28
    C0 = (rng.integers(0, big, (r, s)), rng.integers(0, big // 4, (r, s)))
    R0 = (rng.integers(0, big, (s, c)), rng.integers(0, big // 4, (s, c)))
    C = plus(C0, product(C0, D))
    R = plus(R0, product(D, R0))
    X = (rng.integers(0, big, (r, c)), rng.integers(0, big // 4, (r, c)))
    full = plus(X, product(C, R))
    short = plus(X, product(C, R0))
    assert np.array_equal(full[0], short[0]) and np.array_equal(full[1], short[1])


def test_pre_update_identity_needs_the_closure():
    """With an unclosed block in place of D the two products differ for some
    input: the identity is not vacuous."""
    differs = False
    for seed in range(20):
        rng = np.random.default_rng(4700 + seed)
        s, r, c = 6, 9, 7
        Uq, Lq = W.random_bounds(s, 4800 + seed, p_known=0.4, p_bad=0.05)
        D = (Uq.astype(np.int64), Lq.astype(np.int64))                        # not closed
        big = 1 << 28
        C0 = (rng.integers(0, big, (r, s)), rng.integers(0, big // 4, (r, s)))
        R0 = (rng.integers(0, big, (s, c)), rng.integers(0, big // 4, (s, c)))
        C = plus(C0, product(C0, D))
        R = plus(R0, product(D, R0))
        X = (rng.integers(0, big, (r, c)), rng.integers(0, big // 4, (r, c)))
        full = plus(X, product(C, R))
        short = plus(X, product(C, R0))
        if not (np.array_equal(full[0], short[0]) and np.array_equal(full[1], short[1])):
            differs = True
            break
    assert differs


# ---------------------------------------------------------------- symmetric schedule

def smooth_blocked_symmetric(U0, L0, B, panel_mirror=True):
    """The blocked schedule of symmetric mode on integer matrices, tile by
    tile: phase 1 closes tile (K,K) (the oracle on the tile: the closure of
    its middle atoms), phase 2 the upper-side panel tiles with their
    transposes, phase 3 the tiles with I <= J, then the lower triangle as the
    transpose of the upper one.  Every tile below the diagonal is first
    overwritten with values that would change any result they reached.
    `panel_mirror`: phase 2 stores the transposes (a test drops them)."""
    n = U0.shape[0]
    nb = (n + B - 1) // B
    U, L = U0.astype(np.int64), L0.astype(np.int64)
    sl = [slice(t * B, min(n, (t + 1) * B)) for t in range(nb)]
    for I in range(nb):
        for J in range(I):
            U[sl[I], sl[J]] = 0
            L[sl[I], sl[J]] = 1 << 29

    def tile(I, J):
        return U[sl[I], sl[J]].copy(), L[sl[I], sl[J]].copy()

    def put(I, J, X, mirror=False):
        U[sl[I], sl[J]], L[sl[I], sl[J]] = X
        if mirror:
            U[sl[J], sl[I]], L[sl[J], sl[I]] = X[0].T, X[1].T

    for K in range(nb):
        du, dl = tile(K, K)
        D = tuple(a.astype(np.int64) for a in oracle.smooth(du.astype(np.int32),
                                                            dl.astype(np.int32)))
        put(K, K, D)
        for j in range(nb):
            if j > K:
                X = tile(K, j)
                put(K, j, plus(X, product(D, X)), mirror=panel_mirror)
            elif j < K:
                X = tile(j, K)
                put(j, K, plus(X, product(X, D)), mirror=panel_mirror)
        for I in range(nb):
            for J in range(I, nb):
                if K not in (I, J):
                    put(I, J, plus(tile(I, J), product(tile(I, K), tile(K, J))))
    for I in range(nb):
        for J in range(I + 1, nb):
            put(I, J, tile(I, J), mirror=True)
    return U, L


@pytest.mark.parametrize("n,B", [(12, 4), (13, 4), (17, 5), (9, 3), (7, 8)])
@pytest.mark.parametrize("seed", range(3))
def test_symmetric_schedule_equals_the_oracle(n, B, seed):
    Uq, Lq = W.random_bounds(n, 4900 + 10 * n + seed, p_known=0.4, p_bad=0.05)
    Uo, Lo = oracle.smooth(Uq, Lq)
    Us, Ls = smooth_blocked_symmetric(Uq, Lq, B)
    assert np.array_equal(Us, Uo) and np.array_equal(Ls, Lo)


def test_symmetric_schedule_needs_the_panels_on_both_sides():
    """Without phase 2's transposed stores, phase 3 reads poisoned panel
    tiles below the diagonal: the poison reaches the result, so the test
    above would see a stale read."""
    Uq, Lq = W.random_bounds(12, 4990, p_known=0.4, p_bad=0.05)
    Uo, Lo = oracle.smooth(Uq, Lq)
    Us, Ls = smooth_blocked_symmetric(Uq, Lq, 4, panel_mirror=False)
    assert not (np.array_equal(Us, Uo) and np.array_equal(Ls, Lo))


def test_column_panel_is_the_transposed_row_panel_in_fp32():
    """Off the grid too: with symmetric operands the column-panel product
    (X D) and the row-panel product (D X^T) form the same fp32 sums, so one is
    the other's transpose to the bit."""
    rng = np.random.default_rng(4995)
    s, r = 8, 11
    Du = rng.random((s, s)).astype(np.float32) * 40
    Du = np.minimum(Du, Du.T)
    Dl = (Du * rng.random((s, s)).astype(np.float32) * 0.5).astype(np.float32)
    Dl = np.maximum(Dl, Dl.T)
    Xu = rng.random((r, s)).astype(np.float32) * 40
    Xl = (Xu * rng.random((r, s)).astype(np.float32) * 0.5).astype(np.float32)
    col = product((Xu, Xl), (Du, Dl))
    row = product((Du, Dl), (Xu.T.copy(), Xl.T.copy()))
    assert col[0].dtype == np.float32
    assert np.array_equal(col[0], row[0].T) and np.array_equal(col[1], row[1].T)


# ---------------------------------------------------------------- block rounds in pairs

def pair_schedule(nb, sym=False):
    """The launches of the pair schedule (128-wide tiles), in
    the library's host order, as (stream, kind, K, tiles, rounds, waits):
    stream "s" (the caller's) or "side"; kind "p1", "p2" or "p3"; waits: the
    names of events the launch waits for first.  Events are ("rec", name)
    entries.  The sets are written from their definitions (block-rows and
    -columns), not from the device code's index maps.  sym: every phase-3
    set keeps its tiles on and above the diagonal, the panels are written on
    both sides, and a last launch ("mirror") writes the lower triangle."""
    def rng(*excl):
        return [x for x in range(nb) if x not in excl]

    def tiles_next(K):
        return {(K + 1, j) for j in rng(K)} | {(i, K + 1) for i in rng(K, K + 1)}

    def tiles_panels(K):
        return {(K, j) for j in rng(K)} | {(i, K) for i in rng(K)}

    def near(K):
        rows = {K + 2, K + 3} & set(range(nb))
        return {(i, j) for i in rng(K, K + 1) for j in rng(K, K + 1) if i in rows or j in rows}

    out = []

    def add(e):
        if sym and len(e) == 5 and e[1] == "p3":
            e = e[:3] + ({(i, j) for (i, j) in e[3] if i <= j},) + e[4:]
        out.append(e)
    add(("s", "p1", 0, {(0, 0)}, (0,)))
    add(("s", "p2", 0, tiles_panels(0), (0,)))
    add(("rec", "s", "M"))
    add(("wait", "side", "M"))
    add(("side", "p3", 0, tiles_next(0), (0,)))
    add(("side", "p1", 1, {(1, 1)}, (1,)))
    add(("side", "p2", 1, tiles_panels(1), (1,)))
    add(("rec", "side", "P"))
    K = 0
    while K + 1 < nb:
        add(("wait", "s", "P"))
        add(("s", "p3", K, {(i, j) for i in range(nb) for j in range(nb)
                            if not (K <= i < K + 4) and not (K <= j < K + 4)}, (K, K + 1)))
        if K > 0:
            add(("wait", "side", "M"))
        add(("side", "p3", K, near(K), (K, K + 1)))
        add(("rec", "side", "N"))
        add(("side", "p3", K + 1, {(K + 2, K), (K + 3, K), (K, K + 2), (K, K + 3)}
             & {(i, j) for i in range(nb) for j in range(nb)}, (K + 1,)))
        if K + 2 < nb:
            add(("side", "p1", K + 2, {(K + 2, K + 2)}, (K + 2,)))
            add(("side", "p2", K + 2, tiles_panels(K + 2), (K + 2,)))
        if K + 3 < nb:
            add(("side", "p3", K + 2, tiles_next(K + 2), (K + 2,)))
            add(("side", "p1", K + 3, {(K + 3, K + 3)}, (K + 3,)))
            add(("side", "p2", K + 3, tiles_panels(K + 3), (K + 3,)))
            add(("rec", "side", "P"))
        add(("wait", "s", "N"))
        add(("s", "p3", K + 1, {(K, j) for j in range(nb) if not (K + 1 <= j <= K + 3)}
             | {(i, K) for i in range(nb) if not (K <= i <= K + 3)}, (K + 1,)))
        add(("rec", "s", "M"))
        K += 2
    add(("rec", "side", "J"))
    add(("wait", "s", "J"))
    if K == nb - 1:
        add(("s", "p3", K, {(i, j) for i in rng(K) for j in rng(K)}, (K,)))
    if sym:
        add(("s", "mirror", -1, {(i, j) for i in range(nb) for j in range(i)}, ()))
    return out


def launches_with_order(entries):
    """The launches and, for each, the set of launches that happen before it
    (stream order and event waits)."""
    launches, before = [], []
    last = {"s": None, "side": None}       # last launch on each stream
    pending = {"s": set(), "side": set()}  # happens-before set a stream's next launch inherits
    events = {}
    for e in entries:
        if e[0] == "rec":
            events[e[2]] = set(pending[e[1]])
        elif e[0] == "wait":
            pending[e[1]] |= events[e[2]]
        else:
            idx = len(launches)
            launches.append(e)
            hb = set(pending[e[0]])
            before.append(hb)
            pending[e[0]] = hb | {idx}
    return launches, before


def reads_writes(launch):
    _, kind, K, tiles, rounds = launch
    writes = set(tiles)
    if kind == "mirror":
        return {(j, i) for (i, j) in tiles}, writes
    reads = set(tiles)
    for (i, j) in tiles:
        for k in rounds:
            reads |= {(i, k), (k, j)}
    if kind == "p2":
        reads.add((K, K))
    return reads, writes


@pytest.mark.parametrize("nb", list(range(3, 14)))
@pytest.mark.parametrize("sym", [False, True])
def test_pair_schedule_has_no_race(nb, sym):
    """Launches that may run side by side (neither ordered before the other by
    its stream or an event) touch disjoint tiles: no write meets a read or a
    write of the other."""
    launches, before = launches_with_order(pair_schedule(nb, sym))
    rw = [reads_writes(x) for x in launches]
    for b in range(len(launches)):
        for a in range(b):
            if a in before[b]:
                continue
            (ra, wa), (rb, wb) = rw[a], rw[b]
            assert not (wa & (rb | wb)) and not (wb & ra), (nb, launches[a][1:3], launches[b][1:3])


@pytest.mark.parametrize("nb", list(range(3, 14)))
@pytest.mark.parametrize("sym", [False, True])
def test_pair_schedule_updates_every_tile_with_every_round(nb, sym):
    """Each tile (with symmetric inputs: each tile on or above the diagonal)
    takes every block round exactly once, in increasing order, across the
    launches in any order the dependencies allow (checked along the host
    order, which is one of them)."""
    launches, _ = launches_with_order(pair_schedule(nb, sym))
    done = {(i, j): [] for i in range(nb) for j in range(nb)}
    for _, kind, K, tiles, rounds in launches:
        for (i, j) in tiles:
            if kind != "mirror" and (not sym or i <= j):
                done[(i, j)].extend(rounds)
    for (i, j), r in done.items():
        if not sym or i <= j:
            assert r == list(range(nb)), (nb, (i, j), r)


def smooth_pair_schedule(U0, L0, B, sym=False):
    """Run the pair schedule's launches in host order on integer matrices: a
    phase-3 launch reads, for each tile, its operands of every round it
    applies before writing (one pass), then writes the tile.  sym: the tiles
    below the diagonal are poisoned first (values that would change any
    result they reached), as nothing may read them before they are
    written."""
    n = U0.shape[0]
    nb = (n + B - 1) // B
    U, L = U0.astype(np.int64), L0.astype(np.int64)
    sl = [slice(t * B, min(n, (t + 1) * B)) for t in range(nb)]
    if sym:
        for I in range(nb):
            for J in range(I):
                U[sl[I], sl[J]] = 0
                L[sl[I], sl[J]] = 1 << 29

    def tile(I, J):
        return U[sl[I], sl[J]].copy(), L[sl[I], sl[J]].copy()

    return run_schedule(U, L, sl, pair_schedule(nb, sym), sym)


def run_schedule(U, L, sl, entries, sym=False):
    """Execute a launch list (see pair_schedule) in host order on the tiles of
    U and L (int64, in place; sl: the block slices)."""
    def tile(I, J):
        return U[sl[I], sl[J]].copy(), L[sl[I], sl[J]].copy()

    launches, _ = launches_with_order(entries)
    for _, kind, K, tiles, rounds in launches:
        if kind == "mirror":
            for (I, J) in tiles:
                U[sl[I], sl[J]], L[sl[I], sl[J]] = U[sl[J], sl[I]].T, L[sl[J], sl[I]].T
            continue
        if kind in ("p1", "p1pre"):
            du, dl = tile(K, K)
            if kind == "p1pre":     # round K-1's product first, then the closure
                du, dl = plus((du, dl), product(tile(K, K - 1), tile(K - 1, K)))
            U[sl[K], sl[K]], L[sl[K], sl[K]] = (a.astype(np.int64) for a in oracle.smooth(
                du.astype(np.int32), dl.astype(np.int32)))
            continue
        new = {}
        for (I, J) in tiles:
            if kind == "p2" and sym and I > J:
                continue        # the upper-side panel tile, stored on both sides
            X = tile(I, J)
            if kind == "p2":
                D = tile(K, K)
                X = plus(X, product(D, X)) if I == K else plus(X, product(X, D))
            else:
                for k in rounds:
                    X = plus(X, product(tile(I, k), tile(k, J)))
            new[(I, J)] = X
            if kind == "p2" and sym:
                new[(J, I)] = (X[0].T, X[1].T)
        for (I, J), X in new.items():
            U[sl[I], sl[J]], L[sl[I], sl[J]] = X
    return U, L


@pytest.mark.parametrize("n,B", [(12, 4), (13, 3), (17, 2), (25, 3), (9, 3), (21, 2)])
@pytest.mark.parametrize("seed", range(2))
def test_pair_schedule_equals_the_oracle(n, B, seed):
    Uq, Lq = W.random_bounds(n, 5100 + 10 * n + seed, p_known=0.4, p_bad=0.05,
                             symmetric=bool(seed))
    Uo, Lo = oracle.smooth(Uq, Lq)
    Us, Ls = smooth_pair_schedule(Uq, Lq, B)
    assert np.array_equal(Us, Uo) and np.array_equal(Ls, Lo)


@pytest.mark.parametrize("n,B", [(12, 4), (13, 3), (17, 2), (25, 3), (9, 3), (21, 2)])
def test_symmetric_pair_schedule_equals_the_oracle(n, B):
    Uq, Lq = W.random_bounds(n, 5300 + n, p_known=0.4, p_bad=0.05)
    Uo, Lo = oracle.smooth(Uq, Lq)
    Us, Ls = smooth_pair_schedule(Uq, Lq, B, sym=True)
    assert np.array_equal(Us, Uo) and np.array_equal(Ls, Lo)



# ---------------------------------------------------------------- one block round per pass

def single_round_schedule(nb, mode, drop_side_wait=False):
    """The launch list of the look-ahead schedule with one block round per
    pass, as the library enqueues it (mode "loose": the rest of round K starts
    after phase 2 of round K; "tight": after the next block row and column;
    "merged": small 64-wide matrices, phase 3 of round K but tile (K+1,K+1)
    on the caller's stream beside phase 1 of K+1, which applies round K to
    that tile first).  drop_side_wait: a planted mistake, the side stream no
    longer waits for the rest of the previous round."""
    def rng(*excl):
        return [x for x in range(nb) if x not in excl]

    def panels(K):
        return {(K, j) for j in rng(K)} | {(i, K) for i in rng(K)}

    def nxt(K):
        return {(K + 1, j) for j in rng(K)} | {(i, K + 1) for i in rng(K, K + 1)}

    def rest(K):
        return {(i, j) for i in rng(K, K + 1) for j in rng(K, K + 1)}

    out = []
    add = out.append
    add(("s", "p1", 0, {(0, 0)}, (0,)))
    add(("s", "p2", 0, panels(0), (0,)))
    add(("rec", "s", "M1"))                 # stands for the rest of round -1
    forked = False
    for K in range(nb - 1):
        m_cur, m_prev = "M%d" % (K & 1), "M%d" % ((K + 1) & 1)
        if mode == "merged":
            if forked:
                add(("wait", "s", "SD"))
            forked = False
            add(("s", "p3", K, {(i, j) for i in rng(K) for j in rng(K)} - {(K + 1, K + 1)}, (K,)))
            add(("rec", "s", m_cur))
            add(("wait", "side", m_prev))
            forked = True
            add(("side", "p1pre", K + 1, {(K + 1, K + 1)}, (K, K + 1)))
            add(("wait", "side", m_cur))
            add(("side", "p2", K + 1, panels(K + 1), (K + 1,)))
            add(("rec", "side", "SD"))
            continue
        if mode == "loose":
            if forked:
                add(("wait", "s", "SD"))
            forked = False
            add(("s", "p3", K, rest(K), (K,)))
            add(("rec", "s", m_cur))
        if not drop_side_wait:
            add(("wait", "side", m_prev))
        forked = True
        add(("side", "p3", K, nxt(K), (K,)))
        if mode == "tight":
            add(("rec", "side", "ND"))
        add(("side", "p1", K + 1, {(K + 1, K + 1)}, (K + 1,)))
        add(("side", "p2", K + 1, panels(K + 1), (K + 1,)))
        add(("rec", "side", "SD"))
        if mode == "tight":
            add(("wait", "s", "ND"))
            add(("s", "p3", K, rest(K), (K,)))
            add(("rec", "s", m_cur))
    if forked:
        add(("wait", "s", "SD"))
    add(("s", "p3", nb - 1, {(i, j) for i in rng(nb - 1) for j in rng(nb - 1)}, (nb - 1,)))
    return out


@pytest.mark.parametrize("nb", list(range(3, 13)))
@pytest.mark.parametrize("mode", ["loose", "tight", "merged"])
def test_single_round_schedule_has_no_race(nb, mode):
    """The look-ahead schedules of one round per pass: what the two streams
    may run side by side touches disjoint tiles."""
    launches, before = launches_with_order(single_round_schedule(nb, mode))
    rw = [reads_writes(x) for x in launches]
    for b in range(len(launches)):
        for a in range(b):
            if a in before[b]:
                continue
            (ra, wa), (rb, wb) = rw[a], rw[b]
            assert not (wa & (rb | wb)) and not (wb & ra), (nb, mode, launches[a][1:3],
                                                             launches[b][1:3])


@pytest.mark.parametrize("nb", list(range(3, 13)))
@pytest.mark.parametrize("mode", ["loose", "tight", "merged"])
def test_single_round_schedule_updates_every_tile_with_every_round(nb, mode):
    launches, _ = launches_with_order(single_round_schedule(nb, mode))
    done = {(i, j): [] for i in range(nb) for j in range(nb)}
    for _, kind, K, tiles, rounds in launches:
        for t in tiles:
            done[t].extend(rounds)
    for t, r in done.items():
        assert r == list(range(nb)), (nb, mode, t, r)


@pytest.mark.parametrize("n,B", [(12, 4), (13, 3), (17, 2), (9, 3)])
@pytest.mark.parametrize("mode", ["loose", "tight", "merged"])
def test_single_round_schedule_equals_the_oracle(n, B, mode):
    Uq, Lq = W.random_bounds(n, 5400 + n, p_known=0.4, p_bad=0.05, symmetric=False)
    Uo, Lo = oracle.smooth(Uq, Lq)
    nb = (n + B - 1) // B
    U, L = Uq.astype(np.int64), Lq.astype(np.int64)
    sl = [slice(t * B, min(n, (t + 1) * B)) for t in range(nb)]
    Us, Ls = run_schedule(U, L, sl, single_round_schedule(nb, mode))
    assert np.array_equal(Us, Uo) and np.array_equal(Ls, Lo)


def test_race_check_catches_a_missing_wait():
    """Without the side stream's wait for the rest of the previous round,
    NEXT(K) rewrites panels that REST(K-1) may still be reading: the checker
    flags it."""
    launches, before = launches_with_order(single_round_schedule(6, "loose", drop_side_wait=True))
    rw = [reads_writes(x) for x in launches]
    races = [(a, b) for b in range(len(launches)) for a in range(b) if a not in before[b]
             and ((rw[a][1] & (rw[b][0] | rw[b][1])) or (rw[b][1] & rw[a][0]))]
    assert races


# ---------------------------------------------------------------- the one-launch form

def one_launch_phases(nb, sym=False):
    """The one-launch form (one thread-block cluster per molecule) as phases
    between its cluster barriers; each phase lists the units its CTAs run side
    by side, one per tile (kind, K, tiles, rounds): closure of tile (0,0);
    then per block round K the panels, then every other tile of round K beside
    rank 0's update and closure of tile (K+1,K+1) (the whole round when K is
    the last); with symmetric inputs the tiles on and above the diagonal, the
    panels stored on both sides and the lower triangle written at the end."""
    def keep(t):
        return not sym or t[0] <= t[1]

    phases = [[("p1", 0, {(0, 0)}, (0,))]]
    for K in range(nb):
        panels = []
        for j in range(nb):
            if j == K:
                continue
            if sym:
                t = (K, j) if j > K else (j, K)
                panels.append(("p2", K, {t, (t[1], t[0])}, (K,)))
            else:
                panels += [("p2", K, {(K, j)}, (K,)), ("p2", K, {(j, K)}, (K,))]
        phases.append(panels)
        rest = [("p3", K, {(i, j)}, (K,)) for i in range(nb) for j in range(nb)
                if i != K and j != K and keep((i, j))]
        if K + 1 < nb:
            rest = [u for u in rest if (K + 1, K + 1) not in u[2]]
            rest.append(("p1pre", K + 1, {(K + 1, K + 1)}, (K, K + 1)))
        phases.append(rest)
    if sym:
        phases.append([("mirror", -1, {(i, j)}, ()) for i in range(nb) for j in range(i)])
    return phases


@pytest.mark.parametrize("nb", list(range(2, 10)))
@pytest.mark.parametrize("sym", [False, True])
def test_one_launch_phases_have_no_race(nb, sym):
    """Between two cluster barriers the CTAs' units touch disjoint tiles (a
    symmetric panel unit writes its tile and the transpose)."""
    for units in one_launch_phases(nb, sym):
        rw = []
        for kind, K, tiles, rounds in units:
            if kind == "p2":
                reads = set(tiles) | {(K, K)}
            else:
                reads, _ = reads_writes(("", kind, K, tiles, rounds))
            rw.append((reads, set(tiles)))
        for b in range(len(rw)):
            for a in range(b):
                (ra, wa), (rb, wb) = rw[a], rw[b]
                assert not (wa & (rb | wb)) and not (wb & ra), (nb, sym, units[a], units[b])


@pytest.mark.parametrize("n,B", [(12, 4), (13, 3), (9, 3), (8, 8)])
@pytest.mark.parametrize("sym", [False, True])
def test_one_launch_phases_equal_the_oracle(n, B, sym):
    Uq, Lq = W.random_bounds(n, 5500 + n, p_known=0.4, p_bad=0.05, symmetric=sym)
    Uo, Lo = oracle.smooth(Uq, Lq)
    nb = (n + B - 1) // B
    U, L = Uq.astype(np.int64), Lq.astype(np.int64)
    sl = [slice(t * B, min(n, (t + 1) * B)) for t in range(nb)]
    if sym:
        for I in range(nb):
            for J in range(I):
                U[sl[I], sl[J]] = 0
                L[sl[I], sl[J]] = 1 << 29
    for units in one_launch_phases(nb, sym):
        # every unit of a phase reads the state before the phase (they are
        # disjoint, so the order inside a phase does not matter)
        entries = []
        for kind, K, tiles, rounds in units:
            if kind == "p2" and sym:
                t = min(tiles)        # the upper-side tile; the unit mirrors it
                entries.append(("s", "p2", K, {t, (t[1], t[0])}, rounds))
            else:
                entries.append(("s", kind, K, tiles, rounds))
        U, L = run_schedule(U, L, sl, entries, sym)
    assert np.array_equal(U, Uo) and np.array_equal(L, Lo)

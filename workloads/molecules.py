"""Seeded synthetic molecules and their distance-bound matrices.

This module only draws geometry and writes bound matrices.  It performs no
smoothing arithmetic: the CUDA library and the CPU oracle each receive the
arrays built here and compute independently.

Source of the model (GPU Gems 2, ch. 43, "GPU Computing for Protein Structure
Prediction", section 1, the bound graph): a molecule of n atoms is the complete
graph K_n; every pair (i, j) carries an upper bound u_ij and a lower bound l_ij;
pairs with no experimental constraint get the molecular diameter as upper bound
and a near-zero lower bound.  The matrices are dense, symmetric, with a zero
diagonal, and both triangles are stored.

Readings fixed here (the page leaves them open):
  * unknown pairs: U = n * 3.8 Angstrom, L = 1.0 Angstrom;
  * every value is quantised to 1/1024 Angstrom: lower bounds round down, upper
    bounds round up, so an interval that held the true distance still holds it;
  * a negative lower bound is clamped to 0;
  * the random-walk chain redraws any step that would put an atom closer than
    1.0 Angstrom to an earlier atom, so the unknown-pair lower bound of 1.0 never
    exceeds a true distance (the generated coordinates stay a witness).

All integers returned are Q10 fixed point: value * 1024, int32.
"""
from __future__ import annotations

import numpy as np

Q = 1024                 # fixed-point scale: units of 1/1024 Angstrom
BOND = 3.8               # C-alpha spacing in Angstrom
UNKNOWN_L = 1.0          # lower bound of an unconstrained pair
MIN_SEP = 1.0            # excluded volume of the chain walk

# --------------------------------------------------------------------------
# geometry
# --------------------------------------------------------------------------


def chain_walk(n: int, rng: np.random.Generator, step: float = BOND,
               min_sep: float = MIN_SEP) -> np.ndarray:
    """3-D random walk of n atoms, fixed step, directions N(0, I3) normalised.

    A step that lands within `min_sep` of an earlier atom is redrawn.
    """
    x = np.zeros((n, 3))
    for i in range(1, n):
        for _ in range(1000):
            d = rng.standard_normal(3)
            d *= step / np.linalg.norm(d)
            p = x[i - 1] + d
            if i < 2:
                break
            if np.min(np.sum((x[: i - 1] - p) ** 2, axis=1)) >= min_sep * min_sep:
                break
        else:  # pragma: no cover - never seen with 3.8 A steps
            raise RuntimeError("chain_walk: could not place atom %d" % i)
        x[i] = p
    return x


def serpentine(box: tuple[int, int, int]) -> np.ndarray:
    """Hamiltonian path through an (X, Y, Z) lattice box, boustrophedon order.

    Returns (X*Y*Z, 3) int lattice sites; consecutive sites are face neighbours.
    """
    X, Y, Z = box
    sites = []
    for z in range(Z):
        ys = range(Y) if z % 2 == 0 else range(Y - 1, -1, -1)
        for yi, y in enumerate(ys):
            forward = (z * Y + yi) % 2 == 0
            xs = range(X) if forward else range(X - 1, -1, -1)
            for x in xs:
                sites.append((x, y, z))
    return np.asarray(sites, dtype=np.int64)


_NBR6 = np.array([(1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1)],
                 dtype=np.int64)


def backbite(path: np.ndarray, box: tuple[int, int, int], moves: int,
             rng: np.random.Generator) -> np.ndarray:
    """Randomise a Hamiltonian lattice path by backbite moves (Mansfield's method).

    One move: pick an end of the path and one of its six lattice neighbours s.
    If s is inside the box and is not the end's own path neighbour, join the end
    to s and cut the bond from s toward that end; the piece between them is
    reversed.  Every move keeps the walk self-avoiding and space-filling.
    """
    X, Y, Z = box
    n = len(path)
    path = path.copy()
    lin = path[:, 0] + X * (path[:, 1] + Y * path[:, 2])
    pos = np.empty(X * Y * Z, dtype=np.int64)
    pos[lin] = np.arange(n)
    ends = rng.integers(0, 2, size=moves)
    dirs = rng.integers(0, 6, size=moves)
    for m in range(moves):
        e = 0 if ends[m] == 0 else n - 1
        s = path[e] + _NBR6[dirs[m]]
        if s[0] < 0 or s[1] < 0 or s[2] < 0 or s[0] >= X or s[1] >= Y or s[2] >= Z:
            continue
        p = int(pos[s[0] + X * (s[1] + Y * s[2])])
        if e == n - 1:
            if p == n - 2:
                continue
            a, b = p + 1, n          # reverse path[p+1 : n]
        else:
            if p == 1:
                continue
            a, b = 0, p              # reverse path[0 : p]
        path[a:b] = path[a:b][::-1].copy()
        lin[a:b] = lin[a:b][::-1].copy()
        pos[lin[a:b]] = np.arange(a, b)
    return path


def lattice_globule(box: tuple[int, int, int], rng: np.random.Generator,
                    moves_per_atom: int = 20) -> tuple[np.ndarray, np.ndarray]:
    """Compact self-avoiding chain filling the box; returns (sites, coords in A).

    20 backbite moves per atom: each accepted move reverses a stretch of the
    path, so after a few multiples of n moves the serpentine's long-range order
    (contacts only between neighbouring rows of the boustrophedon) is gone."""
    sites = serpentine(box)
    sites = backbite(sites, box, moves_per_atom * len(sites), rng)
    return sites, sites.astype(np.float64) * BOND


# --------------------------------------------------------------------------
# bounds
# --------------------------------------------------------------------------


def sentinel_q(n: int) -> int:
    """Upper bound of an unknown pair: the molecular diameter n * 3.8 A, in Q10."""
    return int(round(n * BOND * Q))


def blank_bounds(n: int) -> tuple[np.ndarray, np.ndarray]:
    """All pairs unknown, zero diagonal (Q10 int32)."""
    U = np.full((n, n), sentinel_q(n), dtype=np.int32)
    L = np.full((n, n), int(UNKNOWN_L * Q), dtype=np.int32)
    np.fill_diagonal(U, 0)
    np.fill_diagonal(L, 0)
    return U, L


def set_pairs(U: np.ndarray, L: np.ndarray, i: np.ndarray, j: np.ndarray,
              lo: np.ndarray, hi: np.ndarray) -> None:
    """Write symmetric bounds [lo, hi] (Angstrom) for pairs (i, j), quantised outward."""
    lo_q = np.floor(np.maximum(lo, 0.0) * Q).astype(np.int64)
    hi_q = np.ceil(np.maximum(hi, 0.0) * Q).astype(np.int64)
    L[i, j] = lo_q
    L[j, i] = lo_q
    U[i, j] = hi_q
    U[j, i] = hi_q


def pair_dist(x: np.ndarray, i: np.ndarray, j: np.ndarray) -> np.ndarray:
    return np.sqrt(np.sum((x[i] - x[j]) ** 2, axis=1))


def bernoulli_pairs(n: int, p: float, rng: np.random.Generator,
                    exclude: np.ndarray | None = None,
                    block: int = 1024) -> tuple[np.ndarray, np.ndarray]:
    """Each unordered pair i < j (not in `exclude`, an n x n bool) kept with prob. p.

    Random numbers are drawn row block by row block, in row order, one double
    per (i, j) with j > i.
    """
    I, J = [], []
    for r0 in range(0, n, block):
        r1 = min(n, r0 + block)
        draw = rng.random((r1 - r0, n))
        keep = draw < p
        rows = np.arange(r0, r1)[:, None]
        keep &= np.arange(n)[None, :] > rows
        if exclude is not None:
            keep &= ~exclude[r0:r1]
        ii, jj = np.nonzero(keep)
        I.append(ii + r0)
        J.append(jj)
    return np.concatenate(I), np.concatenate(J)


def neighbour_pairs(sites: np.ndarray, box: tuple[int, int, int],
                    max_d2: int = 2) -> tuple[np.ndarray, np.ndarray]:
    """Atom pairs whose lattice separation has squared length 1..max_d2 (i < j)."""
    X, Y, Z = box
    n = len(sites)
    at = np.full(X * Y * Z, -1, dtype=np.int64)
    at[sites[:, 0] + X * (sites[:, 1] + Y * sites[:, 2])] = np.arange(n)
    offs = [(a, b, c) for a in (-1, 0, 1) for b in (-1, 0, 1) for c in (-1, 0, 1)
            if 0 < a * a + b * b + c * c <= max_d2]
    I, J = [], []
    for o in offs:
        t = sites + np.asarray(o)
        ok = np.all((t >= 0) & (t < np.asarray(box)), axis=1)
        src = np.nonzero(ok)[0]
        dst = at[t[ok, 0] + X * (t[ok, 1] + Y * t[ok, 2])]
        keep = src < dst
        I.append(src[keep])
        J.append(dst[keep])
    return np.concatenate(I), np.concatenate(J)


# --------------------------------------------------------------------------
# the five benchmark molecules
# --------------------------------------------------------------------------

CONFIG_SEED = 1000       # config c uses seed 1000 + c
BATCH_SEED = 3000        # molecule b of the batched workload uses seed 3000 + b


def chain_bounds(n: int, seed: int, p_long: float, *, near: float | None = None,
                 jitter: bool = False, long_halfwidth: float = 0.5) -> dict:
    """Random-walk chain with bonded pairs (and optionally all pairs <= `near` A).

    near=None : pairs (i, i+1) known at [d-0.5, d+0.5];
    near=6.0  : every pair with d <= 6 A known; jitter=True draws
                L = d - 0.5 r1, U = d + 0.5 r2 with r1, r2 ~ U(0, 1].
    Other pairs are known with probability p_long at [d-w, d+w], w=long_halfwidth.
    """
    rng = np.random.default_rng(seed)
    x = chain_walk(n, rng)
    U, L = blank_bounds(n)
    if near is None:
        short = np.zeros((n, n), dtype=bool)
        i = np.arange(n - 1)
        short[i, i + 1] = True
    else:
        d2 = np.sum((x[:, None, :] - x[None, :, :]) ** 2, axis=2)
        short = np.triu(d2 <= near * near, k=1)
    si, sj = np.nonzero(short)
    sd = pair_dist(x, si, sj)
    if jitter:
        r1 = 1.0 - rng.random(len(si))
        r2 = 1.0 - rng.random(len(si))
        set_pairs(U, L, si, sj, sd - 0.5 * r1, sd + 0.5 * r2)
    else:
        set_pairs(U, L, si, sj, sd - 0.5, sd + 0.5)
    li, lj = bernoulli_pairs(n, p_long, rng, exclude=short)
    ld = pair_dist(x, li, lj)
    set_pairs(U, L, li, lj, ld - long_halfwidth, ld + long_halfwidth)
    return dict(U=U, L=L, coords=x, n=n, seed=seed, consistent=True)


def globule_bounds(box: tuple[int, int, int], seed: int, p_long: float,
                   p_bad: float = 0.0) -> dict:
    """Lattice globule; pairs <= 6 A known at +-0.5, p_long of the rest at +-2,
    p_bad of the remaining pairs given inconsistent bounds [d+1, max(0, d-1)]."""
    rng = np.random.default_rng(seed)
    sites, x = lattice_globule(box, rng)
    n = len(sites)
    U, L = blank_bounds(n)
    si, sj = neighbour_pairs(sites, box)
    sd = pair_dist(x, si, sj)
    set_pairs(U, L, si, sj, sd - 0.5, sd + 0.5)
    known = np.zeros((n, n), dtype=bool)
    known[si, sj] = True
    li, lj = bernoulli_pairs(n, p_long, rng, exclude=known)
    ld = pair_dist(x, li, lj)
    set_pairs(U, L, li, lj, ld - 2.0, ld + 2.0)
    consistent = True
    if p_bad > 0.0:
        known[li, lj] = True
        bi, bj = bernoulli_pairs(n, p_bad, rng, exclude=known)
        bd = pair_dist(x, bi, bj)
        set_pairs(U, L, bi, bj, bd + 1.0, np.maximum(bd - 1.0, 0.0))
        consistent = len(bi) == 0
    del known
    return dict(U=U, L=L, coords=x, n=n, seed=seed, consistent=consistent)


CONFIGS = {
    0: dict(name="chain n=256 fp32", n=256, dtype="fp32"),
    1: dict(name="chain n=1000 fp32, contacts <= 6 A", n=1000, dtype="fp32"),
    2: dict(name="globule n=4096 int32 Q10 and fp32, 0.1% inconsistent", n=4096,
            dtype="int32"),
    3: dict(name="batch of 256 chains n=512 fp32", n=512, batch=256, dtype="fp32"),
    4: dict(name="globule n=16384 fp32", n=16384, dtype="fp32"),
}


def make_config(idx: int, batch: int | None = None) -> dict:
    """Bound matrices of benchmark molecule `idx` (Q10 int32, n x n, row-major).

    For idx 3 the result holds stacked arrays of shape (batch, n, n); `batch`
    may be lowered for tests (molecule b always uses seed 3000 + b).
    """
    seed = CONFIG_SEED + idx
    if idx == 0:
        out = chain_bounds(256, seed, 0.05)
    elif idx == 1:
        out = chain_bounds(1000, seed, 0.02, near=6.0, jitter=True, long_halfwidth=1.5)
    elif idx == 2:
        out = globule_bounds((16, 16, 16), seed, 0.01, p_bad=0.001)
    elif idx == 3:
        nb = CONFIGS[3]["batch"] if batch is None else batch
        mols = [chain_bounds(512, BATCH_SEED + b, 0.08) for b in range(nb)]
        out = dict(U=np.stack([m["U"] for m in mols]), L=np.stack([m["L"] for m in mols]),
                   coords=np.stack([m["coords"] for m in mols]), n=512, seed=BATCH_SEED,
                   consistent=True, batch=nb)
    elif idx == 4:
        out = globule_bounds((32, 32, 16), seed, 0.005)
    else:
        raise ValueError("unknown molecule config %r" % idx)
    out.update(config=idx, name=CONFIGS[idx]["name"])
    return out


# --------------------------------------------------------------------------
# small random cases for parity tests
# --------------------------------------------------------------------------


def random_bounds(n: int, seed: int, *, p_known: float = 0.3, p_bad: float = 0.0,
                  symmetric: bool = True, maxval: float = 50.0,
                  unknown_u: float | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Random Q10 bound matrices without geometry: known pairs get a random
    interval inside [0, maxval]; a fraction p_bad of known pairs is inverted
    (L > U).  With symmetric=False the two triangles are drawn independently."""
    rng = np.random.default_rng(seed)
    unk = n * BOND if unknown_u is None else unknown_u
    U = np.full((n, n), int(round(unk * Q)), dtype=np.int64)
    L = np.full((n, n), int(UNKNOWN_L * Q), dtype=np.int64)
    a = rng.random((n, n)) * maxval
    b = rng.random((n, n)) * maxval
    lo, hi = np.minimum(a, b), np.maximum(a, b)
    bad = rng.random((n, n)) < p_bad
    lo, hi = np.where(bad, hi, lo), np.where(bad, lo, hi)
    known = rng.random((n, n)) < p_known
    Lk = np.floor(lo * Q).astype(np.int64)
    Uk = np.ceil(hi * Q).astype(np.int64)
    U = np.where(known, Uk, U)
    L = np.where(known, Lk, L)
    if symmetric:
        iu = np.triu_indices(n, 1)
        U.T[iu] = U[iu]
        L.T[iu] = L[iu]
    np.fill_diagonal(U, 0)
    np.fill_diagonal(L, 0)
    return U.astype(np.int32), L.astype(np.int32)


def to_f32(q: np.ndarray) -> np.ndarray:
    """Q10 integers to Angstrom in fp32 (exact below 2**24 units)."""
    return (q.astype(np.float32) / np.float32(Q)).astype(np.float32)

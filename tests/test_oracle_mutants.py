"""The oracle pins are strong enough to catch plausible mistakes (no GPU).

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a transposed operand, a missing closure step, a flipped
comparison), compiles the copy, and runs the same pins as test_oracle_pins:
the worked examples, library shortest paths and the closed form of the lower
bound.  Every mutant must fail at least one of them; the unmutated source must
pass all of them.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest
from scipy.sparse.csgraph import floyd_warshall

from workloads import molecules as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drop_lkj_minus_uik": ("W m = a > b ? a : b;", "W m = b;"),
    "drop_lik_minus_ukj": ("W m = a > b ? a : b;", "W m = a;"),
    "sign_of_uik": ("W a = (W)lrow[j] - uik;", "W a = (W)lrow[j] + uik;"),
    "transposed_upper": ("W s = uik + (W)urow[j];", "W s = uik + (W)ucol[j];"),
    "transposed_lower": ("W b = lik - (W)urow[j];", "W b = lik - (W)ucol[j];"),
    "no_closure_step": ("if (c > (W)lcol[i]) lcol[i] = (T)c;", "(void)c;"),
    "min_for_lower": ("if (m > (W)Li[j]) Li[j] = (T)m;", "if (m < (W)Li[j]) Li[j] = (T)m;"),
    "max_for_upper": ("if (s < (W)Ui[j]) Ui[j] = (T)s;", "if (s > (W)Ui[j]) Ui[j] = (T)s;"),
}


def build_variant(tmp_path, name, patch):
    src = open(SRC).read()
    if patch is not None:
        old, new = patch
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                    str(c), "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    f = lib.oracle_smooth_f64
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    f.restype = ctypes.c_int

    def smooth(U0, L0):
        U = np.ascontiguousarray(U0, dtype=np.float64).copy()
        L = np.ascontiguousarray(L0, dtype=np.float64).copy()
        n = U.shape[0]
        assert f(U.ctypes.data, L.ctypes.data, n, n, 0, 0, n) == 0
        return U, L
    return smooth


def pins_pass(smooth):
    with open(os.path.join(ROOT, "tests", "golden", "examples.json")) as fh:
        examples = json.load(fh)["examples"]
    for ex in examples:
        n = ex["n"]
        lo, hi = ex["unknown"]
        U0 = np.full((n, n), hi)
        L0 = np.full((n, n), lo)
        np.fill_diagonal(U0, 0)
        np.fill_diagonal(L0, 0)
        for i, j, l, u in ex["pairs"]:
            U0[i, j] = U0[j, i] = u
            L0[i, j] = L0[j, i] = l
        U, L = smooth(U0, L0)
        if not (np.array_equal(U, np.array(ex["U"], float))
                and np.array_equal(L, np.array(ex["L"], float))):
            return False
    for seed, sym in ((1, True), (2, False)):
        Uq, Lq = W.random_bounds(24, 40 + seed, p_known=0.4, p_bad=0.05, symmetric=sym)
        Uq = np.where((Uq == 0) & ~np.eye(24, dtype=bool), 1, Uq)
        U0 = Uq.astype(np.float64)
        L0 = Lq.astype(np.float64)
        Us = floyd_warshall(U0, directed=True)
        T = np.max(L0[None, :, :] - Us[:, :, None], axis=1)
        Ls = np.maximum(L0, np.max(T[:, :, None] - Us[None, :, :], axis=1))
        U, L = smooth(U0, L0)
        if not (np.array_equal(U, Us) and np.array_equal(L, Ls)):
            return False
    return True


def test_unmutated_passes(tmp_path):
    assert pins_pass(build_variant(tmp_path, "clean", None))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not pins_pass(build_variant(tmp_path, name, MUTANTS[name]))

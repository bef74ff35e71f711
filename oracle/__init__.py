"""CPU oracle for distance-bound smoothing -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The CUDA library never calls it and shares
no code with it.

The arithmetic lives in `oracle.c` (plain C, OpenMP over rows); this module
compiles it with gcc and wraps it for numpy arrays.  See `oracle.c` for what is
computed and which passage of GPU Gems 2 ch. 43 each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

RULE_CLOSURE = 0
RULE_LITERAL = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i64, vp, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        for name in ("oracle_smooth_f32", "oracle_smooth_f64", "oracle_smooth_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, i64, i64, c_int, i64, i64]
            f.restype = c_int
        lib.oracle_closure_rows.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp]
        lib.oracle_closure_rows.restype = c_int
        lib.oracle_smooth_track_f64.argtypes = [vp, vp, vp, vp, vp, i64, i64]
        lib.oracle_smooth_track_f64.restype = c_int
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = c_int
        lib.oracle_set_threads.argtypes = [c_int]
        lib.oracle_set_threads.restype = None
        for name in ("oracle_count_infeasible_f32", "oracle_count_infeasible_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, i64, i64]
            f.restype = i64
        _lib = lib
        return lib


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_threads())


def set_threads(t: int) -> None:
    """Use t OpenMP threads from now on (timing only; results are the same)."""
    _load().oracle_set_threads(int(t))


_FN = {np.dtype(np.float32): "oracle_smooth_f32",
       np.dtype(np.float64): "oracle_smooth_f64",
       np.dtype(np.int32): "oracle_smooth_i32"}


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def smooth(U: np.ndarray, L: np.ndarray | None = None, *, rule: int = RULE_CLOSURE,
           n: int | None = None, k_begin: int = 0, k_end: int | None = None,
           inplace: bool = False):
    """Round-synchronous Floyd-Warshall smoothing of U (and L) over rounds
    k_begin..k_end-1 (all rounds by default).

    U, L: 2-D C-contiguous arrays of shape (n, ld) or (n, n), dtype float32,
    float64 or int32 (Q10).  The n x n leading block is smoothed; columns beyond
    n are untouched.  Returns (U, L) -- copies unless inplace=True.
    """
    lib = _load()
    if U.ndim != 2 or not U.flags.c_contiguous:
        raise ValueError("U must be a C-contiguous 2-D array")
    if not inplace:
        U = U.copy()
        L = None if L is None else L.copy()
    if L is not None and (L.shape != U.shape or L.dtype != U.dtype
                          or not L.flags.c_contiguous):
        raise ValueError("L must match U in shape, dtype and layout")
    n = U.shape[0] if n is None else n
    ld = U.shape[1]
    k_end = n if k_end is None else k_end
    rc = getattr(lib, _FN[U.dtype])(_ptr(U), _ptr(L), n, ld, rule, k_begin, k_end)
    if rc != 0:
        raise ValueError("oracle_smooth: bad arguments (rc=%d)" % rc)
    return U, L


def smooth_track(U0: np.ndarray, L0: np.ndarray):
    """fp64 closure-rule smoothing that also returns each cell's path
    provenance (see oracle_smooth_track_f64 in oracle.c).

    Returns (U, L, HU, HL, ML): the smoothed bounds (float64), the fewest edges
    of a shortest upper-bound path and of a best lower-bound path (int32), and
    the sum of |edge weight| along that lower-bound path (float64).
    """
    lib = _load()
    U = np.array(U0, dtype=np.float64, order="C")
    L = np.array(L0, dtype=np.float64, order="C")
    if U.ndim != 2 or U.shape[0] != U.shape[1] or L.shape != U.shape:
        raise ValueError("U and L must be n x n")
    n = U.shape[0]
    HU = np.empty((n, n), np.int32)
    HL = np.empty((n, n), np.int32)
    ML = np.empty((n, n), np.float64)
    rc = lib.oracle_smooth_track_f64(_ptr(U), _ptr(L), _ptr(HU), _ptr(HL), _ptr(ML), n, n)
    if rc != 0:
        raise ValueError("oracle_smooth_track_f64: bad arguments (rc=%d)" % rc)
    return U, L, HU, HL, ML


def smooth_upper(U: np.ndarray, **kw) -> np.ndarray:
    """Upper-bound smoothing alone: min-plus all-pairs shortest paths."""
    return smooth(U, None, **kw)[0]


def closure_rows(U0: np.ndarray, L0: np.ndarray | None, rows) -> tuple:
    """Rows `rows` of the smoothing fixed point by Dijkstra (fp64).

    U0, L0: the unsmoothed n x n bounds (any real dtype; Q10 ints allowed).
    Returns (U_rows, L_rows) of shape (len(rows), n) in float64 (L_rows None
    when L0 is None).
    """
    lib = _load()
    U0 = np.ascontiguousarray(U0, dtype=np.float64)
    L0 = None if L0 is None else np.ascontiguousarray(L0, dtype=np.float64)
    n, ld = U0.shape[0], U0.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    Uo = np.empty((len(rows), n))
    Lo = None if L0 is None else np.empty((len(rows), n))
    rc = lib.oracle_closure_rows(_ptr(U0), _ptr(L0), n, ld, _ptr(rows), len(rows),
                                 _ptr(Uo), _ptr(Lo))
    if rc != 0:
        raise ValueError("oracle_closure_rows: bad arguments")
    return Uo, Lo


def count_infeasible(U: np.ndarray, L: np.ndarray, n: int | None = None) -> int:
    """Number of cells (diagonal included) of the n x n block with L > U."""
    lib = _load()
    n = U.shape[0] if n is None else n
    U = np.ascontiguousarray(U)
    L = np.ascontiguousarray(L)
    if U.dtype == np.float32:
        return int(lib.oracle_count_infeasible_f32(_ptr(U), _ptr(L), n, U.shape[1]))
    if U.dtype == np.int32:
        return int(lib.oracle_count_infeasible_i32(_ptr(U), _ptr(L), n, U.shape[1]))
    return int(np.count_nonzero(L[:n, :n] > U[:n, :n]))

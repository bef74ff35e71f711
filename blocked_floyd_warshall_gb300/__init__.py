"""Python binding of libbsmooth: distance-bound smoothing on one GPU.

Argument marshalling only.  Every step of the smoothing runs in the CUDA
kernels of `libbsmooth.so` (built in-tree by `build()`); there is no CPU path.
If the library is missing, every call raises.

Functions keep the C names and argument order of `include/bsmooth.h`:

    bs_smooth_upper(U, n, ld, stream, mode)
    bs_smooth_bounds(U, L, n, ld, stream, mode)
    bs_smooth_bounds_batched(U, L, n, ld, batch_stride, batch, stream, mode)
    bs_check_feasible(U, L, n, ld, stream, mode, mask) -> count
    bs_strerror(status)

Matrix arguments are CUDA torch tensors (or raw device addresses as int).
For a tensor, n, ld, batch, batch_stride and the dtype bits of mode default
from its shape, strides and dtype (float32 -> BS_FP32, int32 -> BS_INT32_Q10);
stream defaults to torch's current stream.  A non-zero status raises BSError.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB as LIBRARY_PATH
from ._build import build as _build_lib

BS_OK = 0
BS_ERR_ARG = 1
BS_ERR_ALIGN = 2
BS_ERR_RANGE = 3
BS_ERR_CUDA = 4
BS_ERR_TIMEOUT = 5
BS_ERR_INPUT = 6

BS_FP32 = 0
BS_INT32_Q10 = 1
BS_DTYPE_MASK = 3
BS_BLOCKED = 0
BS_PERK = 1 << 2
BS_RULE_CLOSURE = 0
BS_RULE_LITERAL = 1 << 3
BS_VALIDATE = 1 << 4
BS_TILE_64 = 1 << 5
BS_TILE_128 = 1 << 6
BS_NO_LOOKAHEAD = 1 << 7
BS_SYMMETRIC = 1 << 8
BS_PERK_PAIRED = 1 << 10
BS_ONE_LAUNCH = 1 << 11
BS_PAIRED_ROUNDS = 1 << 12

PHASES = ("round", "phase1", "phase2", "phase3", "phase3_next", "one_launch")

PROBES = {"fadd": 0, "fmnmx": 1, "fmnmx3": 2, "fadd2": 3, "fadd2+fmnmx3": 4,
          "iadd": 5, "imnmx": 6, "viaddmin": 7, "vimnmx3": 8}


class BSError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, bs_strerror(status), status))


class _Profile(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 6), ("launches", ctypes.c_longlong * 6),
                ("overflow", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libbsmooth.so for sm_103a (nvcc) into the package directory."""
    return _build_lib(force=force)


def library() -> ctypes.CDLL:
    """The loaded libbsmooth.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIBRARY_PATH):
            raise RuntimeError("libbsmooth.so is not built (%s); run "
                               "blocked_floyd_warshall_gb300.build()" % LIBRARY_PATH)
        lib = ctypes.CDLL(LIBRARY_PATH)
        vp, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        sig = {
            "bs_smooth_upper": [vp, i, i, vp, i],
            "bs_smooth_bounds": [vp, vp, i, i, vp, i],
            "bs_smooth_bounds_batched": [vp, vp, i, i, ll, i, vp, i],
            "bs_check_feasible": [vp, vp, i, i, vp, i, ctypes.POINTER(ll), vp],
            "bs_profile_begin": [],
            "bs_profile_end": [ctypes.POINTER(_Profile)],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = i
        lib.bs_check_feasible_noalloc.argtypes = [vp, vp, i, i, ll, i, vp, i,
                                                  ctypes.POINTER(ll)]
        lib.bs_check_feasible_noalloc.restype = i
        lib.bs_probe_alu.argtypes = [i, i, ctypes.POINTER(ctypes.c_double)]
        lib.bs_probe_alu.restype = i
        lib.bs_strerror.argtypes = [i]
        lib.bs_strerror.restype = ctypes.c_char_p
        lib.bs_launch_count.argtypes = []
        lib.bs_launch_count.restype = ll
        lib.bs_one_launch_cluster.argtypes = []
        lib.bs_one_launch_cluster.restype = i
        lib.bs_schedule_info.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.bs_schedule_info.restype = i
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling

def _is_tensor(x) -> bool:
    return hasattr(x, "data_ptr") and hasattr(x, "stride")


def _ptr(x):
    if x is None:
        return None
    if _is_tensor(x):
        if not x.is_cuda:
            raise ValueError("matrix must be a CUDA tensor (device memory)")
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


def _dtype_bits(x, mode):
    if mode is not None:
        return mode
    if _is_tensor(x):
        import torch
        if x.dtype == torch.float32:
            return BS_FP32
        if x.dtype == torch.int32:
            return BS_INT32_Q10
        raise ValueError("unsupported dtype %s (float32 or int32)" % x.dtype)
    return BS_FP32


def _geometry(x, n, ld):
    """n and ld from the last two dimensions of a tensor."""
    if _is_tensor(x):
        if n is None:
            n = x.shape[-2]
        if ld is None:
            ld = x.stride(-2)
            if x.stride(-1) != 1:
                raise ValueError("rows must be contiguous (stride(-1) == 1)")
    if n is None or ld is None:
        raise ValueError("n and ld are required for raw pointers")
    return int(n), int(ld)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(st: int, where: str):
    if st != BS_OK:
        raise BSError(st, where)


# ------------------------------------------------------------------ the C ABI

def bs_smooth_upper(U, n=None, ld=None, stream=None, mode=None, *, flags: int = 0) -> None:
    """Smooth upper bounds alone (min-plus all-pairs shortest paths), in place."""
    n, ld = _geometry(U, n, ld)
    m = _dtype_bits(U, mode) | flags
    _check(library().bs_smooth_upper(_ptr(U), n, ld, _stream(stream), m), "bs_smooth_upper")


def bs_smooth_bounds(U, L, n=None, ld=None, stream=None, mode=None, *, flags: int = 0) -> None:
    """Smooth the bound pair (U, L) in place."""
    n, ld = _geometry(U, n, ld)
    m = _dtype_bits(U, mode) | flags
    _check(library().bs_smooth_bounds(_ptr(U), _ptr(L), n, ld, _stream(stream), m),
           "bs_smooth_bounds")


def bs_smooth_bounds_batched(U, L, n=None, ld=None, batch_stride=None, batch=None,
                             stream=None, mode=None, *, flags: int = 0) -> None:
    """Smooth `batch` independent bound pairs; U, L: (batch, n, ld) tensors."""
    n, ld = _geometry(U, n, ld)
    if _is_tensor(U):
        if batch is None:
            batch = U.shape[0] if U.dim() == 3 else 1
        if batch_stride is None:
            batch_stride = U.stride(0) if U.dim() == 3 else n * ld
    if batch is None or batch_stride is None:
        raise ValueError("batch and batch_stride are required for raw pointers")
    m = _dtype_bits(U, mode) | flags
    _check(library().bs_smooth_bounds_batched(_ptr(U), _ptr(L), n, ld, int(batch_stride),
                                              int(batch), _stream(stream), m),
           "bs_smooth_bounds_batched")


def bs_check_feasible(U, L, n=None, ld=None, stream=None, mode=None, mask=None) -> int:
    """Number of cells with L > U (diagonal included); fills `mask` if given."""
    n, ld = _geometry(U, n, ld)
    out = ctypes.c_longlong(0)
    st = library().bs_check_feasible(_ptr(U), _ptr(L), n, ld, _stream(stream),
                                     _dtype_bits(U, mode), ctypes.byref(out), _ptr(mask))
    _check(st, "bs_check_feasible")
    return int(out.value)


BS_NOALLOC_MAX_BATCH = 4096


def bs_check_feasible_noalloc(U, L, n=None, ld=None, batch_stride=None, batch=None,
                              stream=None, mode=None) -> list:
    """Per-molecule L > U counts without any device allocation.

    For callers that cannot allocate device memory (their allocator owns it
    all, or cudaMalloc's synchronisation is not allowed on their path): the
    counters live in a fixed array of BS_NOALLOC_MAX_BATCH entries inside the
    library.  U, L: (batch, n, ld) or (n, ld) tensors.  Calls that overlap on
    the GPU share that array and race; the first call on a device should come
    before any stream capture.
    """
    n, ld = _geometry(U, n, ld)
    if _is_tensor(U):
        if batch is None:
            batch = U.shape[0] if U.dim() == 3 else 1
        if batch_stride is None:
            batch_stride = U.stride(0) if U.dim() == 3 else n * ld
    if batch is None or batch_stride is None:
        raise ValueError("batch and batch_stride are required for raw pointers")
    out = (ctypes.c_longlong * max(1, int(batch)))()
    st = library().bs_check_feasible_noalloc(_ptr(U), _ptr(L), n, ld, int(batch_stride),
                                             int(batch), _stream(stream), _dtype_bits(U, mode),
                                             out)
    _check(st, "bs_check_feasible_noalloc")
    return [int(out[b]) for b in range(int(batch))]


def bs_strerror(status: int) -> str:
    return library().bs_strerror(int(status)).decode()


def bs_launch_count() -> int:
    return int(library().bs_launch_count())


def bs_one_launch_cluster() -> int:
    """CTAs per cluster of BS_ONE_LAUNCH on the current device (0 before the
    first smoothing call on it)."""
    return int(library().bs_one_launch_cluster())


def bs_schedule_info(n: int, batch: int = 1, mode: int = 0, bounds: bool = True) -> tuple:
    """(tile width, block rounds in pairs) a blocked call would take; host
    logic only, no GPU needed."""
    tile, pairs = ctypes.c_int(0), ctypes.c_int(0)
    _check(library().bs_schedule_info(int(n), int(batch), int(mode), int(bool(bounds)),
                                      ctypes.byref(tile), ctypes.byref(pairs)),
           "bs_schedule_info")
    return tile.value, bool(pairs.value)


def bs_profile_begin() -> None:
    _check(library().bs_profile_begin(), "bs_profile_begin")


def bs_profile_end() -> dict:
    """Per-phase summed device milliseconds and launch counts since begin()."""
    p = _Profile()
    _check(library().bs_profile_end(ctypes.byref(p)), "bs_profile_end")
    return {name: {"ms": p.ms[i], "launches": int(p.launches[i])}
            for i, name in enumerate(PHASES)} | {"overflow": bool(p.overflow)}


def bs_probe_alu(which, iters: int = 20000) -> float:
    """Measured thread-instructions per clock per SM for one instruction form
    (a BS_PROBE_* code or a PROBES name)."""
    code = PROBES[which] if isinstance(which, str) else int(which)
    out = ctypes.c_double(0.0)
    _check(library().bs_probe_alu(code, int(iters), ctypes.byref(out)), "bs_probe_alu")
    return float(out.value)

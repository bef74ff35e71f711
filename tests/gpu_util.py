"""Helpers for the GPU parity tests: device copies, padded layouts, comparisons."""
import numpy as np

import blocked_floyd_warshall_gb300 as bsm

CANARY_F = np.float32(-12345.5)
CANARY_I = np.int32(-777777)


def torch():
    import torch as t
    return t


def dev(a):
    return torch().from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def padded(a, ld, offset=0):
    """Device buffer holding `a` (n x n) with leading dimension ld, canaries in
    the padding and `offset` leading elements (to misalign the base)."""
    n = a.shape[0]
    can = CANARY_F if a.dtype == np.float32 else CANARY_I
    flat = np.full(offset + n * ld, can, dtype=a.dtype)
    view = flat[offset:].reshape(n, ld)
    view[:, :n] = a
    buf = dev(flat)
    return buf, buf[offset:].view(n, ld)


def unpad(mat, n):
    return host(mat)[:, :n]


def canaries_ok(mat, n, offset_buf=None, offset=0):
    a = host(mat)
    can = CANARY_F if a.dtype == np.float32 else CANARY_I
    ok = np.all(a[:, n:] == can)
    if offset_buf is not None and offset:
        ok &= bool(np.all(host(offset_buf)[:offset] == can))
    return bool(ok)


def same_bits(a, b):
    """Bit-for-bit equality (fp32 compared as int32 patterns)."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.dtype == np.float32:
        return np.array_equal(a.view(np.int32), b.view(np.int32))
    return np.array_equal(a, b)


def mode_of(a):
    return bsm.BS_FP32 if a.dtype == np.float32 else bsm.BS_INT32_Q10


def gpu_bounds(U0, L0, flags=0, ld=None, offset=0, batched=False):
    """Smooth on the GPU; returns host (U, L) n x n and whether canaries held."""
    n = U0.shape[0]
    ld = n if ld is None else ld
    bu, U = padded(U0, ld, offset)
    bl, L = padded(L0, ld, offset)
    bsm.bs_smooth_bounds(U, L, n, ld, None, mode_of(U0) | flags)
    torch().cuda.synchronize()
    ok = canaries_ok(U, n, bu, offset) and canaries_ok(L, n, bl, offset)
    return unpad(U, n), unpad(L, n), ok


def gpu_upper(U0, flags=0, ld=None):
    n = U0.shape[0]
    ld = n if ld is None else ld
    _, U = padded(U0, ld)
    bsm.bs_smooth_upper(U, n, ld, None, mode_of(U0) | flags)
    torch().cuda.synchronize()
    return unpad(U, n), canaries_ok(U, n)

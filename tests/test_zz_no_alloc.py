"""The allocation-free infeasibility count agrees with bs_check_feasible.

bs_check_feasible_noalloc serves callers that cannot allocate device memory
(their allocator owns all of it, or cudaMalloc's implicit synchronisation is
not allowed on their path); its counters sit in a fixed array inside the
library.  These tests call it through the C ABI, twice in a row on different
data (the second call must not see the first call's counts), and compare each
molecule's count with the allocating entry point.  This file is collected last
and also passes on its own in a fresh process, where the first call performs
the per-device address look-up.
"""
import numpy as np
import pytest

import blocked_floyd_warshall_gb300 as bsm
from workloads import molecules as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    bsm.build()
    bsm.library()
    return t


def smoothed_batch(torch, seed, batch, n, dtype):
    """Molecule 0 is a geometric chain (consistent: no flags); the others are
    random bounds with inverted pairs (flags)."""
    chain = W.chain_bounds(n, seed, 0.1)
    mols = [(chain["U"], chain["L"])]
    mols += [W.random_bounds(n, seed + b, p_known=0.4, p_bad=0.01 * b) for b in range(1, batch)]
    Uq = np.stack([m[0] for m in mols])
    Lq = np.stack([m[1] for m in mols])
    if dtype == "f32":
        Uq, Lq = W.to_f32(Uq), W.to_f32(Lq)
    U = torch.from_numpy(Uq).cuda()
    L = torch.from_numpy(Lq).cuda()
    bsm.bs_smooth_bounds_batched(U, L)
    return U, L


def reference_counts(U, L):
    return [bsm.bs_check_feasible(U[b], L[b]) for b in range(U.shape[0])]


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_noalloc_counts_match_two_calls(torch, dtype):
    U1, L1 = smoothed_batch(torch, 100, 6, 70, dtype)
    U2, L2 = smoothed_batch(torch, 200, 6, 70, dtype)
    first = bsm.bs_check_feasible_noalloc(U1, L1)
    second = bsm.bs_check_feasible_noalloc(U2, L2)
    assert first == reference_counts(U1, L1)
    assert second == reference_counts(U2, L2)
    assert first != second          # different data, so stale counters would show
    assert any(c > 0 for c in first) and any(c == 0 for c in first)


def test_noalloc_strided_and_single(torch):
    n, ld, B = 50, 53, 3
    stride = n * ld + 7
    U0, L0 = smoothed_batch(torch, 300, B, n, "f32")
    Ub = torch.full((B * stride,), 0.0, dtype=torch.float32, device="cuda")
    Lb = torch.full((B * stride,), 0.0, dtype=torch.float32, device="cuda")
    for b in range(B):
        Ub[b * stride: b * stride + n * ld].view(n, ld)[:, :n] = U0[b]
        Lb[b * stride: b * stride + n * ld].view(n, ld)[:, :n] = L0[b]
    got = bsm.bs_check_feasible_noalloc(Ub, Lb, n, ld, stride, B, None, bsm.BS_FP32)
    assert got == reference_counts(U0, L0)
    assert bsm.bs_check_feasible_noalloc(U0[1], L0[1]) == [reference_counts(U0, L0)[1]]


def test_noalloc_rejects_oversized_batch(torch):
    U = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    L = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(bsm.BSError) as e:
        bsm.bs_check_feasible_noalloc(U, L, 4, 4, 16, bsm.BS_NOALLOC_MAX_BATCH + 1, None,
                                      bsm.BS_FP32)
    assert e.value.status == bsm.BS_ERR_ARG

"""ALU issue-rate probes run and return plausible per-SM rates."""
import pytest

import blocked_floyd_warshall_gb300 as bsm

pytestmark = pytest.mark.gpu


def test_probes_plausible():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bsm.build()
    rates = {name: bsm.bs_probe_alu(name, 2000) for name in bsm.PROBES}
    print(rates)
    # an SM issues at most 4 warp-instructions (128 thread-instructions) per clock
    for name, r in rates.items():
        assert 4.0 < r <= 132.0, (name, r)
    assert rates["fadd"] > 60.0


def test_probe_rejects_bad_code():
    with pytest.raises(bsm.BSError):
        bsm.bs_probe_alu(99)

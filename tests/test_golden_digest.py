"""The stored digest of the oracle's n = 16384 run matches the input the
generator draws today (CPU only).

tests/golden/globule16384_oracle.json holds SHA-256 digests of the oracle's
full smoothing of the n = 16384 lattice globule and of its input; the GPU test
compares the GPU's output with the output digests.  This test redraws the
input and checks its digests, so that a change of the generator is caught on
the CPU, before any GPU run, and checks the record's own consistency.
"""
import json
import os

import pytest

from golden.make_oracle_digest import OUT, ROWS_PER_BLOCK, digest
from workloads import make_config, to_f32


@pytest.fixture(scope="module")
def record():
    with open(OUT) as f:
        return json.load(f)


def test_record_is_consistent(record):
    n = record["n"]
    assert n == 16384
    blocks = (n + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK
    for part in ("input", "output"):
        for mat in ("U", "L"):
            d = record[part][mat]
            assert len(d["sha256"]) == 64
            assert len(d["blocks"]) == blocks
    # the benchmark molecule is consistent: smoothing leaves no L > U cell
    assert record["flags"] == 0
    # smoothing changes the matrices
    assert record["output"]["U"]["sha256"] != record["input"]["U"]["sha256"]
    assert record["output"]["L"]["sha256"] != record["input"]["L"]["sha256"]
    assert "oracle" in record["source"] or "oracle/" in record["source"]


def test_generator_draws_the_recorded_input(record):
    m = make_config(4)
    U, L = to_f32(m["U"]), to_f32(m["L"])
    assert digest(U) == record["input"]["U"]
    assert digest(L) == record["input"]["L"]


def test_digest_names_the_rows_that_differ():
    """A change in one row changes that row's block digest only."""
    import numpy as np
    a = np.arange(300 * 300, dtype=np.float32).reshape(300, 300)
    b = a.copy()
    b[200, 7] += 1.0
    da, db = digest(a), digest(b)
    assert da["sha256"] != db["sha256"]
    diff = [i for i, (x, y) in enumerate(zip(da["blocks"], db["blocks"])) if x != y]
    assert diff == [200 // ROWS_PER_BLOCK]
    assert os.path.basename(OUT) == "globule16384_oracle.json"

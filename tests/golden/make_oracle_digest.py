"""Write the oracle's digest of the n = 16384 lattice-globule smoothing.

The full oracle run (GPU Gems 2 ch. 43, section 3: every round k = 0..n-1 over
all n^2 pairs, each round from the matrix the previous one left, section 2's
rules with the upper bound first) takes n^3 = 4.4e12 cell updates: about 40
minutes on 8 x86 cores, 6 minutes on 16 Grace cores.  Its 2 GiB result is too
large to store, so this script stores SHA-256 digests of it instead: of the
whole U and L, and of every block of 128 rows (so that a mismatch names the
rows).  The GPU test smooths the same input and compares digests, which is a
bit-for-bit comparison of every cell.  The digest of the input is stored too,
so a change of the generator is told apart from a change of the result.

Only `oracle/` computes here; the CUDA library is not imported.

    python tests/golden/make_oracle_digest.py        # writes globule16384_oracle.json
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
OUT = os.path.join(HERE, "globule16384_oracle.json")
ROWS_PER_BLOCK = 128


def digest(a: np.ndarray, rows_per_block: int = ROWS_PER_BLOCK) -> dict:
    """SHA-256 of a C-contiguous fp32 n x n array: whole and by row block."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    whole = hashlib.sha256(a.tobytes()).hexdigest()
    blocks = [hashlib.sha256(a[r:r + rows_per_block].tobytes()).hexdigest()[:16]
              for r in range(0, a.shape[0], rows_per_block)]
    return {"sha256": whole, "blocks": blocks}


def main() -> int:
    sys.path.insert(0, ROOT)
    import oracle
    from workloads import make_config, to_f32

    m = make_config(4)
    U, L = to_f32(m["U"]), to_f32(m["L"])
    n = m["n"]
    rec = {
        "what": "oracle (round-synchronous triple loop, closure rule, fp32) on the n=16384 "
                "lattice globule: SHA-256 of the fp32 bytes of U and L, row-major, whole and "
                "per block of %d rows (first 16 hex digits)" % ROWS_PER_BLOCK,
        "source": "GPU Gems 2 ch. 43, section 2 (rules, upper bound first) and section 3 "
                  "(Floyd-Warshall rounds); written by tests/golden/make_oracle_digest.py, "
                  "which calls only oracle/",
        "n": n,
        "input": {"U": digest(U), "L": digest(L)},
    }
    oracle.build()
    t0 = time.perf_counter()
    oracle.smooth(U, L, inplace=True)
    wall = time.perf_counter() - t0
    rec["output"] = {"U": digest(U), "L": digest(L)}
    rec["flags"] = oracle.count_infeasible(U, L)
    rec["oracle_wall_s"] = wall
    rec["oracle_threads"] = oracle.threads()
    rec["host_cores"] = len(os.sched_getaffinity(0))
    with open(OUT, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print("wrote %s (oracle %.0f s on %d threads)" % (OUT, wall, rec["oracle_threads"]))
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""The grid sizes of the phase-3 launches (`p3_tiles`, host and device code
alike) against the tile sets' definitions, on the CPU: a count too small
would leave tiles of a round unupdated, one too large would send CTAs past
the set.  The sets are written here from their definitions (block rows and
columns), as in tests/test_schedule_algebra.py."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "tile_counts.cu")
NAMES = ["ALL", "NEXT", "REST", "PANELS", "ALL_OFF", "REST2", "NEAR2", "PREV2", "CORNER2"]


def expected(name, sym, nb, K):
    """Size of a launch's tile set.  PREV2 and CORNER2 are launched with K the
    pair's second round (base round K - 1); the pair sets need K + 1 < nb."""
    if nb < 2:
        return 0
    tiles = range(nb)

    def up(s):
        return {t for t in s if not sym or t[0] <= t[1]}

    if name == "ALL":
        s = {(i, j) for i in tiles for j in tiles if K not in (i, j)}
    elif name == "ALL_OFF":
        if K + 1 >= nb:
            return 0
        s = {(i, j) for i in tiles for j in tiles if K not in (i, j)} - {(K + 1, K + 1)}
    elif name == "NEXT":
        if K + 1 >= nb:
            return 0
        s = {(i, j) for i in tiles for j in tiles
             if K not in (i, j) and K + 1 in (i, j)}
    elif name == "REST":
        if K + 1 >= nb:
            return 0
        s = {(i, j) for i in tiles for j in tiles if not {i, j} & {K, K + 1}}
    elif name == "PANELS":
        # general: the row and the column panel; symmetric: one side of each pair
        s = {(K, j) for j in tiles if j != K} | {(i, K) for i in tiles if i != K}
        return len(s) // 2 if sym else len(s)
    elif name == "REST2":
        if K + 1 >= nb:
            return 0
        blk = set(range(K, min(K + 4, nb)))
        s = {(i, j) for i in tiles for j in tiles if i not in blk and j not in blk}
    elif name == "NEAR2":
        if K + 1 >= nb:
            return 0
        near = {K + 2, K + 3} & set(tiles)
        s = {(i, j) for i in tiles for j in tiles
             if not {i, j} & {K, K + 1} and {i, j} & near}
    elif name == "PREV2":
        if K < 1:
            return 0
        b = K - 1
        s = {(b, j) for j in tiles if not b + 1 <= j <= b + 3} | \
            {(i, b) for i in tiles if not b <= i <= b + 3}
    elif name == "CORNER2":
        if K < 1:
            return 0
        b = K - 1
        s = {(b + 2, b), (b + 3, b), (b, b + 2), (b, b + 3)} & {(i, j) for i in tiles for j in tiles}
    return len(up(s))


@pytest.fixture(scope="module")
def counts(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc unavailable")
    exe = str(tmp_path_factory.mktemp("tc") / "tile_counts")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + os.path.join(ROOT, "include"), SRC, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    rows = [tuple(int(x) for x in line.split()) for line in out.splitlines()]
    assert rows
    return rows


def test_every_launch_size_matches_its_set(counts):
    bad = []
    for part, sym, nb, K, got in counts:
        want = expected(NAMES[part], sym, nb, K)
        if got != want:
            bad.append((NAMES[part], sym, nb, K, got, want))
    assert not bad, bad[:10]

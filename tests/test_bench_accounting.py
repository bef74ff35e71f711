"""Host-side accounting of bench.py (no GPU): the cell-update counts its
roofline divides by, and its copies of the library's schedule rules."""
import itertools
import json
import os

import pytest

import bench


def brute_phase_cells(n, fb):
    """Count (i, j, k) by phase straight from the blocked schedule's
    definition: round K owns the middle atoms of block K; a cell in block row
    and column K is phase 1, one in exactly one of them phase 2, the rest
    phase 3."""
    p = [0, 0, 0]
    for k in range(n):
        K = k // fb
        for i, j in itertools.product(range(n), repeat=2):
            inr, inc = i // fb == K, j // fb == K
            p[0 if inr and inc else 1 if inr or inc else 2] += 1
    return tuple(p)


@pytest.mark.parametrize("n,fb", [(1, 64), (5, 4), (9, 4), (12, 4), (13, 8)])
def test_phase_cells_match_the_definition(n, fb):
    assert bench.phase_cells(n, fb) == brute_phase_cells(n, fb)
    assert sum(bench.phase_cells(n, fb)) == n ** 3


@pytest.mark.parametrize("n,fb", [(9, 4), (12, 4), (13, 8), (300, 64)])
def test_next_and_diagonal_cells(n, fb):
    """NEXT(K) covers the tiles of block row and column K+1 outside row and
    column K; the diagonal tile (K+1, K+1) is one of them."""
    nb = (n + fb - 1) // fb
    sizes = [min(fb, n - K * fb) for K in range(nb)]
    nxt = diag = 0
    for K in range(nb - 1):
        mk = sizes[K]
        for I in range(nb):
            for J in range(nb):
                if I == K or J == K:
                    continue
                if I == K + 1 or J == K + 1:
                    nxt += sizes[I] * sizes[J] * mk
                if I == J == K + 1:
                    diag += sizes[I] * sizes[J] * mk
    assert bench.next_cells(n, fb) == nxt
    assert bench.diag_cells(n, fb) == diag
    assert diag <= nxt <= bench.phase_cells(n, fb)[2]


def test_merged_lookahead_rule():
    """The library's merged look-ahead: 64-wide tiles and fewer rest tiles
    than half the SMs -- general n <= 640, symmetric n <= 832 on 152 SMs."""
    sms = 152
    assert bench.merged_lookahead(640, 64, 1, sms)
    assert not bench.merged_lookahead(641, 64, 1, sms)
    assert bench.merged_lookahead(832, 64, 1, sms, sym=True)
    assert not bench.merged_lookahead(833, 64, 1, sms, sym=True)
    assert not bench.merged_lookahead(128, 64, 1, sms)          # two block rounds: no look-ahead
    assert not bench.merged_lookahead(256, 128, 1, sms)         # 128-wide tiles
    assert bench.merged_lookahead(300, 64, 4, sms)              # 9 rest tiles x 4 molecules
    assert not bench.merged_lookahead(257, 64, 12, sms)         # 9 x 12 = 108


def test_tile_rule_matches_documented_thresholds():
    """128-wide tiles from 48 block rows of 128 (where block rounds go in
    pairs) or once a 128-wide phase 3 holds >= 9000 tiles over the batch,
    else 64; fp32 and int32 alike (768 tiles for the upper bound alone)."""
    assert bench.tile_size(4096) == 64
    assert bench.tile_size(6016) == 64 and bench.tile_size(6017) == 128   # 47, 48 rows
    assert bench.tile_size(10000) == 128
    assert bench.tile_size(16384) == 128
    assert bench.tile_size(4096, flags=1) == 64 and bench.tile_size(16384, flags=1) == 128
    assert bench.tile_size(6017, flags=1) == 128
    assert bench.tile_size(10000, flags=1 << 8) == 64          # symmetric: 78^2 < 9000
    assert bench.tile_size(3000, batch=18) == 128              # 23^2 x 18 = 9522
    assert bench.tile_size(3000, batch=17) == 64               # 23^2 x 17 = 8993
    assert bench.tile_size(512, batch=256) == 64               # 9 x 256 = 2304
    assert bench.tile_size(4096, upper=True) == 128            # U alone: 961 >= 768
    assert bench.tile_size(3000, upper=True) == 64             # 23^2 = 529


@pytest.mark.parametrize("n", [1, 2, 3, 4096, 4097])
def test_per_round_bytes(n):
    """Per-round mode: one read and one write of U and L per pass; the plain
    form takes one round per pass, the paired form two (and a lone last round
    for n odd)."""
    passes = n // 2 + n % 2
    assert bench.perk_bytes(n, paired=True) == 16 * n * n * passes
    assert bench.perk_bytes(n, paired=False) == 16 * n * n * n


def brute_pair_side_cells(n, fb):
    """Cell updates of the look-ahead stream's phase-3 launches when block
    rounds go in pairs, from the sets' definitions: per pair (K, K+1) block
    row and column K+1 outside row and column K take round K; block rows and
    columns K+2, K+3 outside K, K+1 take rounds K and K+1; tiles (K+2, K),
    (K+3, K), (K, K+2), (K, K+3) take round K+1; then (NEXT of the next pair)
    block row and column K+3 outside K+2 take round K+2 -- that is NEXT(K+2),
    counted with the next pair's K."""
    nb = (n + fb - 1) // fb
    size = [min(fb, n - K * fb) for K in range(nb)]
    cells = 0
    K = 0
    while K + 1 < nb:
        for I in range(nb):
            for J in range(nb):
                if I != K and J != K and (I == K + 1 or J == K + 1):
                    cells += size[I] * size[J] * size[K]
                if (I not in (K, K + 1) and J not in (K, K + 1)
                        and (I in (K + 2, K + 3) or J in (K + 2, K + 3))):
                    cells += size[I] * size[J] * (size[K] + size[K + 1])
                if (I, J) in ((K + 2, K), (K + 3, K), (K, K + 2), (K, K + 3)):
                    cells += size[I] * size[J] * size[K + 1]
        K += 2
    return cells


@pytest.mark.parametrize("n,fb", [(9, 3), (12, 4), (13, 3), (17, 2), (25, 3), (30, 4)])
def test_pair_schedule_main_and_side_cells_cover_phase3(n, fb):
    """With block rounds in pairs the caller's-stream launches and the
    look-ahead stream's together apply every phase-3 cell update once (phase-2
    panels aside)."""
    main, passes = bench.main_stream_phase3(n, fb, pairs=True)
    assert main + brute_pair_side_cells(n, fb) == bench.phase_cells(n, fb)[2]
    if n % fb == 0:
        assert passes * fb <= main          # every pass applies one round or two


def test_pair_schedule_halves_the_passes_at_16384():
    """At n = 16384 nearly every caller's-stream pass applies two rounds: the
    tile cells passed over are about half the cell updates / 128."""
    main, passes = bench.main_stream_phase3(16384, 128)
    assert 0.5 < passes * 128 / main < 0.53


@pytest.mark.parametrize("n,fb", [(9, 4), (12, 4), (13, 8), (300, 64), (1000, 64)])
def test_single_round_main_stream_cells(n, fb):
    """One block round per pass: the caller's stream runs all of phase 3 but
    the next block row and column of each round (the merged form of small
    matrices: all but tile (K+1, K+1)); each pass applies fb middle atoms."""
    p3 = bench.phase_cells(n, fb)[2]
    main, passes = bench.main_stream_phase3(n, fb)
    nb = (n + fb - 1) // fb
    if nb < 3:
        assert main == p3
    elif bench.merged_lookahead(n, fb, 1, 152):
        assert main == p3 - bench.diag_cells(n, fb)
    else:
        assert main == p3 - bench.next_cells(n, fb)
    serial, _ = bench.main_stream_phase3(n, fb, flags=1 << 7)
    assert serial == p3
    if n % fb == 0:
        assert passes * fb == main


def test_pair_schedule_rule():
    """Look-ahead on: 128-wide tiles take block rounds in pairs from 48 block
    rows (n = 6017), 64-wide ones once a pair's bulk ((nb - 4)^2 tiles, or
    (nb - 4)(nb - 3) / 2 with symmetric inputs) holds 2500 tiles over the
    batch; BS_PAIRED_ROUNDS forces them."""
    assert bench.pair_schedule_runs(16384, 128)
    assert bench.pair_schedule_runs(6017, 128)
    assert not bench.pair_schedule_runs(6016, 128)
    assert bench.pair_schedule_runs(16384, 128, sym=True)
    assert bench.pair_schedule_runs(300, 128, flags=1 << 12)
    assert not bench.pair_schedule_runs(16384, 128, flags=1 << 7)
    assert bench.pair_schedule_runs(4096, 64)                        # 60^2 = 3600
    assert not bench.pair_schedule_runs(3000, 64)                    # 43^2 = 1849
    assert bench.pair_schedule_runs(3456, 64)                        # 50^2 = 2500
    assert not bench.pair_schedule_runs(3392, 64)                    # 49^2 = 2401
    assert bench.pair_schedule_runs(512, 64, batch=256)              # 16 x 256 = 4096
    assert not bench.pair_schedule_runs(4096, 64, sym=True)          # 60 x 61 / 2 = 1830
    assert bench.pair_schedule_runs(8192, 64, sym=True)              # 124 x 125 / 2 = 7750
    assert bench.pair_schedule_runs(300, 64, flags=1 << 12)
    assert bench.tile_size(300, flags=1 << 12) == 128
    assert bench.tile_size(300, flags=(1 << 12) | (1 << 5)) == 64


def test_instruction_mix_ceiling():
    """3 adds + 3 comparisons per cell update, two operations per paired
    instruction: at 128 paired instructions per clock per SM, 128 / 3 cells."""
    assert bench.mix_ceiling_cells_per_clk(128.0) == pytest.approx(128.0 / 3)
    assert bench.mix_ceiling_cells_per_clk(None) == pytest.approx(128.0 / 3)
    assert bench.mix_ceiling_cells_per_clk(125.0) == pytest.approx(125.0 / 3)


def test_committed_phase3_capture_is_current():
    """The committed ncu DRAM figure of phase 3 was taken on the current
    kernel code; after any change to that code the capture must be re-taken
    (bench.py reports no traffic while the hashes differ)."""
    with open(os.path.join(bench.ROOT, "profiles", "phase3_traffic.json")) as f:
        d = json.load(f)
    assert d["kernel_hash"] == bench.kernel_hash(), (
        "profiles/phase3_traffic.json is stale: re-take the phase-3 DRAM capture")
    per_pass_cell = d["dram_bytes_per_pass_cell"]
    assert per_pass_cell == pytest.approx(
        (d["dram_bytes_read"] + d["dram_bytes_write"]) / d["tile_cells_per_launch"])


def test_kernel_hash_ignores_comments_only():
    """The hash that ties the committed capture to the kernel sees code, not
    comments or layout: a changed comment keeps it, changed code does not."""
    a = "int f(int x) { return x + 1; }  // add one\n"
    b = "/* the successor */ int f(int x) {\n    return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert bench.code_only('s = "// kept";') == 's = "// kept";'


def test_committed_capture_rate():
    """The capture's own launch alone: its cell updates x 6 over its duration
    against the ALU peak; at most the peak itself."""
    peak = 152 * 128 * 2070e6
    r = bench.committed_capture_rate(peak)
    with open(os.path.join(bench.ROOT, "profiles", "phase3_traffic.json")) as f:
        d = json.load(f)
    assert r is not None
    assert r["frac"] == pytest.approx(6 * d["cells_per_launch"] / (d["gpu_time_ns"] * 1e-9) / peak)
    assert 0.5 < r["frac"] < 1.0


def test_bench_rules_match_the_library():
    """bench.py's copies of the tile and pair rules give what the library
    itself would run (bs_schedule_info, host logic only)."""
    import blocked_floyd_warshall_gb300 as bsm
    bsm.build()
    sizes = [1, 2, 63, 64, 65, 128, 129, 256, 300, 385, 513, 1000, 2048, 3000, 3392, 3456, 3584,
             4096, 5120, 6016, 6017, 6144, 8192, 10000, 12160, 12161, 16384, 20000]
    modes = [0, bsm.BS_TILE_64, bsm.BS_TILE_128, bsm.BS_SYMMETRIC, bsm.BS_PAIRED_ROUNDS,
             bsm.BS_PAIRED_ROUNDS | bsm.BS_TILE_64, bsm.BS_NO_LOOKAHEAD,
             bsm.BS_SYMMETRIC | bsm.BS_TILE_128]
    checked = 0
    for n in sizes:
        for batch in (1, 3, 64, 256):
            if n * n * batch > 2 ** 31:
                continue
            for mode in modes:
                for bounds in (True, False):
                    tile, pairs = bsm.bs_schedule_info(n, batch, mode, bounds)
                    want_tile = bench.tile_size(n, flags=mode, batch=batch, upper=not bounds)
                    assert tile == want_tile, (n, batch, mode, bounds, tile, want_tile)
                    want_pairs = bench.pair_schedule_runs(n, tile, flags=mode,
                                                          sym=bool(mode & bsm.BS_SYMMETRIC),
                                                          batch=batch)
                    assert pairs == want_pairs, (n, batch, mode, bounds, pairs, want_pairs)
                    checked += 1
    assert checked > 1000

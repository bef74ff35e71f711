#!/usr/bin/env python3
"""Benchmark: distance-bound smoothing of the n = 16384 lattice globule (fp32).

One step = one complete bs_smooth_bounds call (blocked three-phase
Floyd-Warshall, all 128 block rounds) on a fresh copy of the bound pair that
is already resident in HBM.  Metric: cell-updates/s = n^3 / time per step,
and its fraction of the FP32 ALU peak (6 ALU ops per cell update:
U add + min, L two subtractions + two maxima; peak = SMs x 128 lanes x
max SM clock).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead
(bounded samples of the same workload on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# mode bits of the per-round forms: one round per pass, two rounds per pass
PERK_FLAGS = {"perk": 1 << 2, "perk2": (1 << 2) | (1 << 10)}
METRIC = "bound-smoothing cell-updates/s (n³/time) and % of GB300 FP32 ALU peak"
UNIT = "cell-updates/s"
OPS_PER_CELL = 6
FP32_LANES_PER_SM = 128
WORKLOADS = {
    "globule16384": dict(config=4, desc="lattice globule n=16384, fp32 U+L, blocked"),
    "globule4096": dict(config=2, consistent=False,   # 0.1 % inverted pairs by design
                        desc="lattice globule n=4096, fp32 U+L, blocked"),
    # profiling size: inputs 4x larger than L2, a few GB on the device
    "globule8192": dict(box=(32, 16, 16), seed=1005, p_long=0.005,
                        desc="lattice globule n=8192 (profiling size), fp32 U+L, blocked"),
    # the small molecules of the benchmark set, for launch lists
    "chain256": dict(config=0, desc="random-walk chain n=256, fp32 U+L, blocked"),
    "chain1000": dict(config=1, desc="random-walk chain n=1000, fp32 U+L, blocked"),
    # 256 molecules in one batched call: a capture target only (--profile-calls)
    "batch256x512": dict(config=3, desc="256 random-walk chains n=512, fp32 U+L, batched"),
}


def make_workload(name):
    from workloads import make_config
    from workloads.molecules import globule_bounds
    wl = WORKLOADS[name]
    if "config" in wl:
        return make_config(wl["config"])
    return globule_bounds(wl["box"], wl["seed"], wl["p_long"])


def tile_size(n, flags=0, batch=1, upper=False):
    """Tile size the library picks (mirrors its rule; forced by the tile bits;
    upper: bs_smooth_upper, U alone)."""
    if flags & (1 << 5):
        return 64
    if flags & ((1 << 6) | (1 << 12)):     # BS_TILE_128, BS_PAIRED_ROUNDS (without BS_TILE_64)
        return 128
    nb = (n + 127) // 128
    if not upper and not flags & (1 << 8) and nb >= PAIRS_FROM:   # general inputs, in pairs
        return 128
    return 128 if (nb - 1) ** 2 * batch >= (768 if upper else 9000) else 64


def phase_cells(n, fb, sym=False):
    """Cell updates (i, j, k) each phase executes in one blocked smoothing.
    Without symmetry the three phases sum to n^3 exactly."""
    nb = (n + fb - 1) // fb
    sizes = [min(fb, n - K * fb) for K in range(nb)]
    p1 = p2 = p3 = 0
    for K, mk in enumerate(sizes):
        rest = n - mk
        p1 += mk ** 3
        p2 += (1 if sym else 2) * rest * mk * mk
        if sym:
            others = [sizes[I] for I in range(nb) if I != K]
            cells = sum(others[a] * others[b] for a in range(len(others))
                        for b in range(a, len(others)))
            p3 += cells * mk
        else:
            p3 += rest * rest * mk
    return p1, p2, p3


def perk_bytes(n, paired=True):
    """DRAM bytes the per-round mode must move per smoothing: U and L read
    and written once per pass over the matrix; a pass takes one round (plain
    form) or two (paired form, with a lone last round when n is odd)."""
    passes = (n + 1) // 2 if paired else n
    return 16.0 * float(n) ** 2 * passes


def mix_ceiling_cells_per_clk(probe_instr_per_clk=None):
    """Cell updates per clock per SM the phase-3 instruction mix allows: a
    cell update is 3 adds (FP32 pipe) and 3 comparisons (ALU pipe), issued as
    paired add.f32x2 and three-input min/max, two operations per instruction.
    With both pipes fed every cycle (the probe interleaving the two forms
    measures the issue rate) that is rate x 2 / 6; without a probe, the
    128 + 128 lanes of the two pipes give 128 / 3."""
    if probe_instr_per_clk:
        return probe_instr_per_clk * 2.0 / 6.0
    return 128.0 / 3.0


def diag_cells(n, fb):
    """Cell updates of tile (K+1, K+1) in block rounds K < nb - 1: with the
    merged look-ahead of small matrices phase 1 of round K+1 applies them,
    and the caller's stream runs the rest of each round's phase 3."""
    nb = (n + fb - 1) // fb
    sizes = [min(fb, n - K * fb) for K in range(nb)]
    return sum(sizes[K] * sizes[K + 1] ** 2 for K in range(nb - 1))


def merged_lookahead(n, fb, batch, sms, sym=False):
    """The library's rule for its merged look-ahead schedule (64-wide tiles,
    fewer rest-of-round tiles than half the SMs)."""
    nb = (n + fb - 1) // fb
    if fb != 64 or nb < 3:
        return False
    rest = 0.5 * (nb - 2) * (nb - 1) if sym else float(nb - 2) ** 2
    return rest * batch < 0.5 * sms


PAIRS_FROM = 48        # block rows from which 128-wide tiles take block rounds in pairs
PAIRS_TILES_64 = 2500  # bulk tiles of a pair (over the batch) from which 64-wide tiles do


def pair_schedule_runs(n, fb, flags=0, sym=False, batch=1):
    """The library's rule for taking block rounds in pairs (look-ahead on;
    forced by BS_PAIRED_ROUNDS): 128-wide tiles from 48 block rows, 64-wide
    ones once a pair's bulk holds 2500 tiles over the batch."""
    nb = (n + fb - 1) // fb
    if nb < 3 or flags & (1 << 7):
        return False
    if flags & (1 << 12):
        return True
    if fb == 128:
        return nb >= PAIRS_FROM
    r = nb - 4
    rest2 = 0 if r <= 0 else (r * (r + 1) // 2 if sym else r * r)
    return rest2 * batch >= PAIRS_TILES_64


def main_stream_phase3(n, fb, flags=0, batch=1, sms=152, pairs=None):
    """Phase-3 launches of one blocked smoothing on the caller's stream
    (general inputs, look-ahead on; the roofline's schedule): (cell updates,
    tile cells passed over).
    A pass over an r x c tile reads and writes it once, whatever the middle
    atoms it applies, so 16 bytes per tile cell (U and L, fp32) are the
    algorithmic DRAM traffic of a pass.
      pairs: per pair (K, K+1) the tiles outside block-rows and -columns
             K .. K+3 take both rounds in one pass, then block-row and
             -column K outside K+1 .. K+3 take round K+1; an odd last round
             runs whole;
      merged (64-wide tiles, few rest tiles): every round but tile (K+1,K+1);
      otherwise: every round but block-row and -column K+1, the last whole.
    `pairs`: take the pair schedule or not (default: the library's rule)."""
    nb = (n + fb - 1) // fb
    size = [min(fb, n - K * fb) for K in range(nb)]
    cells = passes = 0

    def add(tiles, rounds):
        nonlocal cells, passes
        k = sum(size[r] for r in rounds)
        for (i, j) in tiles:
            cells += size[i] * size[j] * k
            passes += size[i] * size[j]

    def others(*excl):
        return [x for x in range(nb) if x not in excl]

    if nb < 2:
        return 0, 0
    if pair_schedule_runs(n, fb, flags, batch=batch) if pairs is None else pairs:
        K = 0
        while K + 1 < nb:
            block = set(range(K, min(K + 4, nb)))
            add([(i, j) for i in range(nb) for j in range(nb)
                 if i not in block and j not in block], (K, K + 1))
            add([(K, j) for j in range(nb) if not (K + 1 <= j <= K + 3)]
                + [(i, K) for i in range(nb) if not (K <= i <= K + 3)], (K + 1,))
            K += 2
        if K == nb - 1:
            add([(i, j) for i in others(K) for j in others(K)], (K,))
    else:
        merged = merged_lookahead(n, fb, batch, sms)
        serial = nb < 3 or flags & (1 << 7)
        for K in range(nb):
            if serial or K == nb - 1:
                skip = ()
            elif merged:
                skip = ((K + 1, K + 1),)
            else:
                skip = None
            if skip is None:
                add([(i, j) for i in others(K, K + 1) for j in others(K, K + 1)], (K,))
            else:
                add([(i, j) for i in others(K) for j in others(K) if (i, j) not in skip], (K,))
    return cells * batch, passes * batch


def next_cells(n, fb):
    """Cell updates of the look-ahead launches of one blocked smoothing: the
    tiles of block row and column K+1 (outside row and column K) in block
    rounds K < nb - 1.  They run on the library's side stream; the rest of
    phase 3 runs on the caller's stream."""
    nb = (n + fb - 1) // fb
    sizes = [min(fb, n - K * fb) for K in range(nb)]
    cells = 0
    for K in range(nb - 1):
        mk, s1 = sizes[K], sizes[K + 1]
        other = n - mk - s1
        cells += mk * s1 * (2 * other + s1)
    return cells


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d.get("hbm_gbs", 6800.0), sm_max_mhz=d.get("sm_max_mhz", 2070.0),
                    source="measured")
    return dict(hbm_gbs=6800.0, sm_max_mhz=2070.0, source="fallback")


KERNEL_SOURCES = ("phase3.cu", "p3_tile.cuh", "pairops.cuh", "bs_tile.cuh", "bs_types.cuh")


def code_only(text):
    """C++ source without its comments, whitespace runs collapsed: what the
    compiler sees, so that the kernel hash ignores edits to comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_hash():
    """Hash of the phase-3 kernel's code (its source file, the device helpers
    and the types it includes; not the host-side declarations of the other
    kernels), comments left out: ties a committed ncu traffic figure to the
    code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blocked_floyd_warshall_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update((f + "\n" + code_only(fh.read())).encode())
    return h.hexdigest()[:16]


def committed_traffic(pass_cells):
    """DRAM bytes of phase-3 launches that pass over `pass_cells` tile cells
    (a pass reads and writes its tile once, whatever the rounds it applies),
    from the committed ncu summary (bytes per tile cell passed x cells), if
    the summary was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "phase3_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    per_pass_cell = d.get("dram_bytes_per_pass_cell")
    if per_pass_cell is None:
        return None
    return per_pass_cell * float(pass_cells)


def committed_capture_rate(alu_peak_ops):
    """The committed capture's launch alone: 6-op rate of its cell updates
    over its ncu duration (one launch, cold caches, nothing beside it) as a
    fraction of the ALU peak, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "phase3_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash() or not d.get("gpu_time_ns"):
        return None
    ops = OPS_PER_CELL * float(d["cells_per_launch"])
    return {"frac": ops / (d["gpu_time_ns"] * 1e-9) / alu_peak_ops,
            "basis": "profiles/phase3_traffic.json: %s, alone under ncu" % d.get("workload", "")}


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = os.path.join("/tmp", "bs_clocks_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        with open(self.out) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, v in zip(self.NAMES, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.out)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_smi_id(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[torch.cuda.current_device()] if vis else torch.cuda.current_device()


# ------------------------------------------------------------------ distributed


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(ms, units, device="cpu"):
    """Whole-job figures over ranks: (max time over ranks, units summed over
    ranks).  Each rank smooths its own replica (the path has no exchange step),
    so the job rate is the summed units over the slowest rank's time.  Without
    an initialised multi-rank process group the local values come back."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(units)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ oracle leg


def oracle_rate(U0, L0, seconds, max_rounds=None):
    """Time the CPU oracle on rounds 0..R-1 of the workload until `seconds`
    elapse; returns (cell-updates/s, rounds, threads)."""
    import oracle
    oracle.build()
    U = U0.copy()
    L = L0.copy()
    n = U.shape[0]
    rounds, t0 = 0, time.perf_counter()
    chunk = 4
    while True:
        k1 = min(n, rounds + chunk)
        oracle.smooth(U, L, k_begin=rounds, k_end=k1, inplace=True)
        rounds = k1
        el = time.perf_counter() - t0
        if el >= seconds or rounds >= n or (max_rounds and rounds >= max_rounds):
            break
    return rounds * float(n) * n / el, rounds, oracle.threads(), el


def oracle_plan(args):
    """The CPU oracle as a reported baseline across the benchmark molecules:
    one thread and all host cores on configs 0-3 (each a bounded sample: whole
    smoothings, or its first rounds, or its first molecules, until about
    --cpu-seconds of work), and with --oracle-full one full all-core run of
    the n = 16384 globule, whose result is checked against the stored digest
    of the oracle (tests/golden/globule16384_oracle.json).  One JSON line each."""
    import oracle
    from workloads import make_config, to_f32
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    all_threads = oracle.threads()
    cases = [(0, "f32"), (1, "f32"), (2, "f32"), (2, "i32"), (3, "f32")]
    for cfg, dt in cases:
        m = make_config(cfg)
        U0, L0 = (to_f32(m["U"]), to_f32(m["L"])) if dt == "f32" else (m["U"], m["L"])
        n, batch = m["n"], m.get("batch", 1)
        for threads in (1, all_threads):
            oracle.set_threads(threads)
            done, t0 = 0.0, time.perf_counter()
            if batch > 1:
                mols = 0
                while mols < batch and time.perf_counter() - t0 < args.cpu_seconds:
                    oracle.smooth(U0[mols], L0[mols])
                    mols += 1
                done = mols * float(n) ** 3
                sample = "%d of %d molecules, whole smoothings" % (mols, batch)
            else:
                U, L = U0.copy(), L0.copy()
                k = 0
                while k < n and time.perf_counter() - t0 < args.cpu_seconds:
                    k1 = min(n, k + 8)
                    oracle.smooth(U, L, k_begin=k, k_end=k1, inplace=True)
                    k = k1
                done = k * float(n) ** 2
                sample = ("whole smoothing" if k == n
                          else "rounds 0..%d of %d" % (k - 1, n))
            el = time.perf_counter() - t0
            print(json.dumps({"oracle": "config %d" % cfg, "dtype": dt, "n": n, "batch": batch,
                              "threads": threads, "host_cores": cores, "seconds": el,
                              "cell_updates_per_s": done / el, "sample": sample}), flush=True)
    oracle.set_threads(all_threads)
    if args.oracle_full:
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from golden.make_oracle_digest import OUT, digest
        m = make_config(4)
        U, L = to_f32(m["U"]), to_f32(m["L"])
        n = m["n"]
        t0 = time.perf_counter()
        oracle.smooth(U, L, inplace=True)
        el = time.perf_counter() - t0
        with open(OUT) as f:
            ref = json.load(f)
        same = (digest(U)["sha256"] == ref["output"]["U"]["sha256"]
                and digest(L)["sha256"] == ref["output"]["L"]["sha256"])
        print(json.dumps({"oracle": "config 4, full", "dtype": "f32", "n": n, "batch": 1,
                          "threads": all_threads, "host_cores": cores, "seconds": el,
                          "cell_updates_per_s": float(n) ** 3 / el,
                          "sample": "whole smoothing",
                          "matches_stored_digest": same}), flush=True)
    return 0


# ------------------------------------------------------------------ main


def bench_config(wl, n, mode, ws):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": wl["desc"], "n": n, "batch": 1, "mode": mode,
            "parallelism": "replicas" if ws > 1 else "single",
            "l2": "inputs larger than L2: each step smooths its own resident "
                  "2 x %d MiB copy" % (n * n * 4 >> 20)}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    from workloads import to_f32
    wl = WORKLOADS[args.workload]
    m = make_workload(args.workload)
    U0, L0 = to_f32(m["U"]), to_f32(m["L"])
    n = m["n"]
    times, rates = [], []
    per_step = args.ref_rounds
    for s in range(args.warmup + args.steps):
        rate, rounds, thr, el = oracle_rate(U0, L0, seconds=1e9, max_rounds=per_step)
        if s >= args.warmup:
            times.append(el)
            rates.append(rate)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * float(np.mean(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(wl, n, "blocked", ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": "each step: rounds 0..%d of the n=%d workload "
                                   "(%d x n^2 cell updates)" % (per_step - 1, n, per_step)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="globule16384")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="only run this many smoothing calls of the workload (no timing, "
                         "no JSON line): a short target for ncu captures")
    ap.add_argument("--mode", choices=["blocked", "perk", "perk2", "upper", "one", "sym"],
                    default="blocked",
                    help="perk: the per-round reference mode, one round per pass (HBM-bound); "
                         "perk2: its two-rounds-per-pass form; both for their HBM roofline "
                         "and captures; upper: bs_smooth_upper (U alone), one: the "
                         "one-launch form, and sym: the symmetric half-work mode, with "
                         "--profile-calls only (the sweep times them)")
    ap.add_argument("--tile", choices=["auto", "64", "128"], default="auto",
                    help="force the tile size of the blocked schedule (captures of one "
                         "kernel form; the default line uses the library's own choice)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU-oracle sample length for cpu_baseline")
    ap.add_argument("--ref-rounds", type=int, default=48,
                    help="oracle rounds per step for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the ALU issue-rate probes")
    ap.add_argument("--no-symmetric", action="store_true",
                    help="skip the extra timing of the symmetric half-work mode")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timing of the other benchmark molecules (configs 0-3)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every benchmark molecule (one JSON line each) instead")
    ap.add_argument("--oracle-plan", action="store_true",
                    help="time the CPU oracle on configs 0-3, one thread and all cores "
                         "(one JSON line each), instead")
    ap.add_argument("--oracle-full", action="store_true",
                    help="with --oracle-plan: also run the full n=16384 oracle once on all "
                         "cores and check it against the stored digest (minutes)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.mode in ("upper", "one", "sym") and args.profile_calls <= 0:
        ap.error("--mode %s is a capture target: use it with --profile-calls" % args.mode)
    if args.workload == "batch256x512" and args.profile_calls <= 0:
        ap.error("the batch workload is a capture target: use it with --profile-calls")

    ws, rank, local = dist_setup()
    if args.oracle_plan:
        return oracle_plan(args) if rank == 0 else 0
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    if args.sweep:
        return sweep(args)

    import torch
    import blocked_floyd_warshall_gb300 as bsm
    from workloads import to_f32

    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    bsm.build()
    bsm.library()

    wl = WORKLOADS[args.workload]
    m = make_workload(args.workload)
    n = m["n"]
    U0, L0 = to_f32(m["U"]), to_f32(m["L"])
    dU0 = torch.from_numpy(U0).cuda()
    dL0 = torch.from_numpy(L0).cuda()
    stream = torch.cuda.current_stream()
    wU, wL = dU0.clone(), dL0.clone()

    flags = PERK_FLAGS.get(args.mode, 0) | (bsm.BS_ONE_LAUNCH if args.mode == "one" else 0) \
        | (bsm.BS_SYMMETRIC if args.mode == "sym" else 0) \
        | {"auto": 0, "64": bsm.BS_TILE_64, "128": bsm.BS_TILE_128}[args.tile]
    if args.profile_calls > 0:
        for _ in range(args.profile_calls):
            wU.copy_(dU0)
            wL.copy_(dL0)
            if args.mode == "upper":
                bsm.bs_smooth_upper(wU)
            elif wU.dim() == 3:
                bsm.bs_smooth_bounds_batched(wU, wL, flags=flags)
            else:
                bsm.bs_smooth_bounds(wU, wL, flags=flags)
        torch.cuda.synchronize()
        print("profile calls done: %d x %s, n=%d" % (args.profile_calls, args.mode, n))
        return 0

    ncopies = min(args.steps, 32)
    copies = [(dU0.clone(), dL0.clone()) for _ in range(ncopies)]
    # warm-up on a scratch copy
    for _ in range(args.warmup):
        wU.copy_(dU0)
        wL.copy_(dL0)
        bsm.bs_smooth_bounds(wU, wL, flags=flags)
    torch.cuda.synchronize()

    # timed region: K steps, each on its own resident copy
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = bsm.bs_launch_count()
    # the per-round mode makes up to 2n launches per call: per-launch profile
    # events would add their own cost to its time, so it is timed without them
    profile = args.mode not in PERK_FLAGS
    with ClockSampler(gpu_smi_id(torch)) as clk:
        if profile:
            bsm.bs_profile_begin()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            U, L = copies[s % ncopies]
            ev[s][0].record(stream)
            bsm.bs_smooth_bounds(U, L, flags=flags)
            ev[s][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        prof = bsm.bs_profile_end() if profile else {
            k: {"ms": 0.0, "launches": 0} for k in bsm.PHASES}
    launches = bsm.bs_launch_count() - launches0
    total_ms = t_start.elapsed_time(t_end)
    cells = float(n) ** 3
    total_ms, units = aggregate(total_ms, args.steps * cells, device="cuda")
    if ws > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    value = units / (total_ms * 1e-3)

    # parity of the timed output: the stored result is the fixed point, so one
    # more smoothing must leave every bit unchanged, and the flags must be zero
    U, L = copies[0]
    U2, L2 = U.clone(), L.clone()
    bsm.bs_smooth_bounds(U2, L2, flags=flags)
    torch.cuda.synchronize()
    fixed_point = bool(torch.equal(U2, U) and torch.equal(L2, L))
    del U2, L2
    assert fixed_point, "timed output is not the smoothing fixed point"
    if wl.get("consistent", True):
        assert bsm.bs_check_feasible(U, L) == 0
    # the feasibility pass (HBM-bound: reads 8 n^2 bytes), timed on its own
    fz = []
    for r in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bsm.bs_check_feasible(U, L)
        b.record(stream)
        torch.cuda.synchronize()
        if r:
            fz.append(a.elapsed_time(b))
    feas_ms = statistics.median(fz)

    peaks = load_peaks()
    fmax = peaks["sm_max_mhz"] * 1e6
    alu_peak_ops = sms * FP32_LANES_PER_SM * fmax            # ALU ops/s
    # phase 3 on the caller's stream (the rest of each block round, and the
    # last round whole): these launches never overlap one another
    p3 = prof["phase3"]
    fb = tile_size(n, flags)
    p3_cells_step = phase_cells(n, fb)[2]
    main_cells_step, main_pass_cells = main_stream_phase3(n, fb, flags, 1, sms)
    p3_ops_step = main_cells_step * OPS_PER_CELL
    p3_s_step = p3["ms"] * 1e-3 / args.steps
    p3_achieved = p3_ops_step / p3_s_step if p3["launches"] else None
    traffic = committed_traffic(main_pass_cells)
    algo_bytes = 16.0 * main_pass_cells
    clocks = clk.summary()
    probes = {} if args.no_probe else {
        name: round(bsm.bs_probe_alu(name), 2) for name in bsm.PROBES}
    mix_cells = mix_ceiling_cells_per_clk(probes.get("fadd2+fmnmx3"))
    mix_peak_cells = sms * mix_cells * fmax

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": bench_config(wl, n, args.mode, ws),
        "fp32_alu_frac": value / ws * OPS_PER_CELL / alu_peak_ops,
        "fp32_alu_peak_basis": "%d SMs x %d lanes x %.0f MHz (%s max SM clock)" % (
            sms, FP32_LANES_PER_SM, peaks["sm_max_mhz"], peaks["source"]),
        "step_ms": {"median": statistics.median(step_ms), "best": min(step_ms)},
        "roofline": {
            "kernel": "k_phase3 (bulk tile update)", "bound": "alu",
            "achieved": p3_achieved / 1e12 if p3_achieved else None,
            "peak": alu_peak_ops / 1e12, "unit": "Tops/s",
            "frac": (p3_achieved / alu_peak_ops) if p3_achieved else None,
            "traffic": traffic,
            "traffic_basis": "DRAM bytes of the same launches in one smoothing step (ncu bytes "
                             "per tile cell passed over, profiles/phase3_traffic.json, x the "
                             "tile cells those launches pass over)",
            "algorithmic_bytes": algo_bytes,
            "traffic_over_algorithmic": (traffic / algo_bytes) if traffic else None,
            "frac_alone_committed_capture": committed_capture_rate(alu_peak_ops),
            "algorithmic_bytes_basis": "16 bytes per tile cell per pass: each output tile of U "
                                       "and L read and written once per pass, a pass applying "
                                       "one block round, or two where rounds go in pairs",
            "schedule": "block rounds in pairs" if pair_schedule_runs(n, fb, flags, batch=1)
                        else "one block round per pass",
            "frac_of_instruction_mix_ceiling": (p3_achieved / OPS_PER_CELL / mix_peak_cells)
                                               if p3_achieved else None,
            "instruction_mix_ceiling_cells_per_clk_per_sm": mix_cells,
            "instruction_mix_ceiling_basis": "3 adds (FP32 pipe) + 3 comparisons (ALU pipe) per "
                                             "cell update, two per add.f32x2 / three-input "
                                             "min-max; issue rate of the two interleaved, "
                                             "measured by the ALU probe in this run",
            "ops_per_step": p3_ops_step,
            "cells_share_of_phase3": main_cells_step / p3_cells_step,
            "ms_per_step": p3_s_step * 1e3,
            "launches_per_step": p3["launches"] / args.steps,
            "achieved_basis": "6 ops x cell updates of the step's phase-3 launches on the caller's "
                              "stream (all but the tiles the look-ahead stream takes) / "
                              "their summed device time, each launch timed with CUDA events on "
                              "that stream; the look-ahead stream's kernels share the GPU with "
                              "them meanwhile, so this understates the kernel alone",
            "share_of_step": p3["ms"] / args.steps / (total_ms / args.steps),
            "peak_basis": "SMs x 128 FP32 lanes x max SM clock, 6 ALU ops per cell update (%s)"
                          % peaks["source"],
        },
        "phases_ms_per_step": {k: prof[k]["ms"] / args.steps for k in bsm.PHASES},
        "gpu_launches": launches,
        "clocks": clocks,
        "feasible": {"ms": feas_ms, "gbs": 8.0 * n * n / (feas_ms * 1e-3) / 1e9,
                     "frac_of_hbm": 8.0 * n * n / (feas_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "basis": "bs_check_feasible on the smoothed matrices: 8 n^2 bytes read / "
                              "event time of the call (launch, counter reset, 8-byte readback)"},
    }
    if args.mode in PERK_FLAGS:
        # per-round mode: every pass reads and writes all of U and L (16 bytes
        # per cell update with one round per pass, 8 with two), HBM-bound; the
        # step is these launches only
        paired = args.mode == "perk2"
        r_gbs = perk_bytes(n, paired) / (total_ms / args.steps * 1e-3) / 1e9
        line["roofline"] = {
            "kernel": ("k_round2 + k_cross2 (per-round mode, two rounds per pass)" if paired
                       else "k_round + k_cross (per-round mode, one round per pass)"),
            "bound": "hbm",
            "achieved": r_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": r_gbs / peaks["hbm_gbs"], "traffic": None,
            "achieved_basis": "16 bytes (read + write of U and L) x n^2 cells per pass (%s) / "
                              "step time (the step is these launches only)"
                              % ("two rounds per pass, a lone last round for n odd" if paired
                                 else "one round per pass"),
            "peak_basis": "STREAM-style copy (%s)" % peaks["source"],
            "launches_per_step": launches / args.steps,
        }

    if not args.no_symmetric:
        line["symmetric"] = symmetric_leg(torch, bsm, dU0, dL0, copies, args, value / ws)
    if probes:
        line["alu_probe_instr_per_clk_per_sm"] = probes
    if not args.no_e2e:
        line["e2e"] = e2e_leg(torch, bsm, U0, L0, args, ws)
    if not args.no_configs and args.mode == "blocked":
        line["other_configs"] = configs_leg(torch, bsm, alu_peak_ops, peaks["hbm_gbs"])
    if rank == 0 and ws >= 1 and not args.no_cpu_baseline and ws == 1:
        rate, rounds, thr, el = oracle_rate(U0, L0, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": thr, "kind": "oracle",
            "host_cores": len(os.sched_getaffinity(0)),
            "sample": "rounds 0..%d of the n=%d workload (%d x n^2 cell updates, %.1f s)"
                      % (rounds - 1, n, rounds, el)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


SCHEDULE_FLAGS = {"auto": 0, "t64": 1 << 5, "t128": 1 << 6,
                  "t64_serial": (1 << 5) | (1 << 7), "t128_serial": (1 << 6) | (1 << 7),
                  "perk": 1 << 2, "perk2": (1 << 2) | (1 << 10), "sym": 1 << 8,
                  "one": 1 << 11, "one_sym": (1 << 11) | (1 << 8),   # one launch per call
                  "pairs": 1 << 12, "pairs64": (1 << 12) | (1 << 5),   # block rounds in pairs, forced
                  "graph": 0,   # "graph": the auto schedule captured once, replayed
                  "upper": 0}   # "upper": bs_smooth_upper, U alone
ALL_SCHEDULES = ("auto", "t64", "t128", "t64_serial", "t128_serial", "sym")
SWEEP = (
    # (config, dtype, schedules, description); config None: random bounds of size n
    (0, "f32", ALL_SCHEDULES + ("graph", "one"), "chain n=256"),
    (1, "f32", ALL_SCHEDULES + ("graph", "one"), "chain n=1000"),
    (("random", 2048), "f32", ALL_SCHEDULES + ("graph", "one"), "random bounds n=2048"),
    (("random", 3000), "f32", ("auto", "t64", "t128", "t128_serial"), "random bounds n=3000"),
    (2, "f32", ALL_SCHEDULES + ("pairs", "pairs64", "perk", "perk2", "upper"), "globule n=4096"),
    (2, "i32", ("auto",), "globule n=4096"),
    (3, "f32", ALL_SCHEDULES + ("pairs64", "one", "one_sym"), "256 chains n=512, batched"),
    (4, "f32", ("auto", "t128_serial", "sym", "upper"), "globule n=16384"),
)


def sweep(args):
    """Device time of one smoothing for every benchmark molecule."""
    import torch
    import blocked_floyd_warshall_gb300 as bsm
    from workloads import make_config, to_f32
    bsm.build()
    props = torch.cuda.get_device_properties(0)
    peaks = load_peaks()
    alu = props.multi_processor_count * FP32_LANES_PER_SM * peaks["sm_max_mhz"] * 1e6
    cache = {}
    for cfg, dt, scheds, desc in SWEEP:
        for algo in scheds:
            if cfg not in cache:
                cache.clear()
                if isinstance(cfg, tuple):
                    from workloads import random_bounds
                    Uq, Lq = random_bounds(cfg[1], 4242, p_known=0.2)
                    cache[cfg] = dict(U=Uq, L=Lq, n=cfg[1])
                else:
                    cache[cfg] = make_config(cfg)
            m = cache[cfg]
            U0, L0 = (to_f32(m["U"]), to_f32(m["L"])) if dt == "f32" else (m["U"], m["L"])
            dU0, dL0 = torch.from_numpy(U0).cuda(), torch.from_numpy(L0).cuda()
            n = m["n"]
            batch = m.get("batch", 1)
            flags = SCHEDULE_FLAGS[algo]
            reps = max(3, min(args.steps, 20)) if n < 16384 else max(3, min(args.steps, 5))
            times = []

            def call(U, L):
                if algo == "upper":
                    bsm.bs_smooth_upper(U, flags=flags)
                elif batch > 1:
                    bsm.bs_smooth_bounds_batched(U, L, flags=flags)
                else:
                    bsm.bs_smooth_bounds(U, L, flags=flags)
            if algo == "graph":
                # one call captured in a CUDA graph, replayed: the launch
                # sequence is submitted at once.  Each replay redoes the full
                # smoothing of the same matrices (the work does not depend
                # on the values).
                U, L = dU0.clone(), dL0.clone()
                call(U, L)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    call(U, L)
                for r in range(args.warmup + reps):
                    torch.cuda.synchronize()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    g.replay()
                    b.record()
                    torch.cuda.synchronize()
                    if r >= args.warmup:
                        times.append(a.elapsed_time(b))
                Uo, Lo = dU0.clone(), dL0.clone()
                call(Uo, Lo)
                assert torch.equal(U, Uo) and torch.equal(L, Lo)
                del g
            for r in range(0 if algo == "graph" else args.warmup + reps):
                U, L = dU0.clone(), dL0.clone()
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                call(U, L)
                b.record()
                torch.cuda.synchronize()
                if r >= args.warmup:
                    times.append(a.elapsed_time(b))
            ms = statistics.median(times)
            cells = batch * float(n) ** 3
            rate = cells / (ms * 1e-3)
            line = {"sweep": desc, "config": cfg, "dtype": dt, "mode": algo, "n": n, "batch": batch,
                    "ms_median": ms, "ms_best": min(times), "cell_updates_per_s": rate,
                    "fp32_alu_frac": rate * OPS_PER_CELL / alu}
            if algo in ("sym", "one_sym"):
                fb = 64 if algo == "one_sym" else tile_size(n, flags, batch)
                executed = batch * float(sum(phase_cells(n, fb, sym=True)))
                line["executed_cell_updates"] = executed
                line["fp32_alu_frac_executed"] = executed / (ms * 1e-3) * OPS_PER_CELL / alu
            if algo == "upper":
                # U alone: an add and a min per cell update
                line["fp32_alu_frac_upper"] = rate * 2 / alu
            if algo in PERK_FLAGS:
                gbs = perk_bytes(n, algo == "perk2") * batch / (ms * 1e-3) / 1e9
                line["hbm_gbs_algorithmic"] = gbs
                line["hbm_frac"] = gbs / peaks["hbm_gbs"]
            print(json.dumps(line), flush=True)
            del dU0, dL0
    return 0


def symmetric_leg(torch, bsm, dU0, dL0, copies, args, general_rate):
    """The same smoothing with BS_SYMMETRIC (tiles on and above the diagonal,
    mirrored): same output, about half the cell updates executed.  Each step
    restores its copy from the resident input outside the timed events."""
    n = dU0.shape[0]
    times = []
    for s in range(args.steps):
        U, L = copies[s % len(copies)]
        U.copy_(dU0)
        L.copy_(dL0)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        bsm.bs_smooth_bounds(U, L, flags=bsm.BS_SYMMETRIC)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    rate = float(n) ** 3 / (ms * 1e-3)
    executed = float(sum(phase_cells(n, tile_size(n, flags=1 << 8), sym=True)))
    return {"ms_per_step": ms, "value": rate, "unit": UNIT + " (n^3 / time, same output)",
            "speedup_vs_general": rate / general_rate,
            "executed_cell_updates": executed,
            "executed_cell_updates_per_s": executed / (ms * 1e-3),
            "note": "inputs are symmetric; only tiles with I <= J are computed and mirrored, "
                    "so about half of the n^3 cell updates are executed"}


def configs_leg(torch, bsm, alu_peak_ops, hbm_gbs):
    """The other benchmark molecules, timed in the same run: device time of
    one call (median of 5, each on a fresh copy restored outside the timed
    events), cell-updates/s and the fraction of the 6-op peak; config 2 also
    in int32 and in the plain per-round mode (HBM-bound, GB/s of its 16 bytes
    per cell update), and config 3 also in the one-launch form."""
    from workloads import make_config, to_f32
    out = {}
    cases = [("chain256", 0, "f32", 0), ("chain1000", 1, "f32", 0),
             ("globule4096", 2, "f32", 0), ("globule4096_i32", 2, "i32", 0),
             ("globule4096_perk", 2, "f32", PERK_FLAGS["perk"]),
             ("batch256x512", 3, "f32", 0),
             ("batch256x512_one_launch", 3, "f32", 1 << 11)]
    cache = {}
    for name, cfg, dt, flags in cases:
        if cfg not in cache:
            cache.clear()
            cache[cfg] = make_config(cfg)
        m = cache[cfg]
        U0, L0 = (to_f32(m["U"]), to_f32(m["L"])) if dt == "f32" else (m["U"], m["L"])
        dU0, dL0 = torch.from_numpy(U0).cuda(), torch.from_numpy(L0).cuda()
        U, L = dU0.clone(), dL0.clone()
        n, batch = m["n"], m.get("batch", 1)
        times = []
        for r in range(3 + 5):
            U.copy_(dU0)
            L.copy_(dL0)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            if batch > 1:
                bsm.bs_smooth_bounds_batched(U, L, flags=flags)
            else:
                bsm.bs_smooth_bounds(U, L, flags=flags)
            b.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        rate = batch * float(n) ** 3 / (ms * 1e-3)
        rec = {"n": n, "batch": batch, "dtype": dt, "ms": ms, "cell_updates_per_s": rate}
        if flags & PERK_FLAGS["perk"]:
            gbs = perk_bytes(n, paired=False) * batch / (ms * 1e-3) / 1e9
            rec.update(hbm_gbs_algorithmic=gbs, hbm_frac=gbs / hbm_gbs)
        else:
            rec["fp32_alu_frac"] = rate * OPS_PER_CELL / alu_peak_ops
        out[name] = rec
        del dU0, dL0, U, L
    return out


def e2e_leg(torch, bsm, U0, L0, args, ws):
    """Same metric through the public call with host buffers.  Every step
    copies its pinned inputs to the device, smooths them and reads both results
    back to pinned host memory.  Steps are pipelined as a caller streaming
    molecules would: two device buffer sets and separate upload, compute and
    download streams, so the upload of step s+1 and the download of step s-1
    overlap the smoothing of step s.  The timed region runs from the first
    upload to the last download."""
    n = U0.shape[0]
    steps = max(2, args.steps)
    hU = [torch.from_numpy(U0).pin_memory() for _ in range(2)]
    hL = [torch.from_numpy(L0).pin_memory() for _ in range(2)]
    oU = [torch.empty_like(hU[0]).pin_memory() for _ in range(2)]
    oL = [torch.empty_like(hL[0]).pin_memory() for _ in range(2)]
    dU = [torch.empty(hU[0].shape, dtype=hU[0].dtype, device="cuda") for _ in range(2)]
    dL = [torch.empty(hL[0].shape, dtype=hL[0].dtype, device="cuda") for _ in range(2)]
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    # the host link alone: one step's upload, timed before the pipeline
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(up)
    dU[0].copy_(hU[0], non_blocking=True)
    dL[0].copy_(hL[0], non_blocking=True)
    b.record(up)
    torch.cuda.synchronize()
    h2d_ms = a.elapsed_time(b)
    loaded = [torch.cuda.Event() for _ in range(2)]
    smoothed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for s in range(steps):
        b = s % 2
        with torch.cuda.stream(up):
            if s >= 2:
                up.wait_event(drained[b])            # buffer b's previous result is out
            dU[b].copy_(hU[b], non_blocking=True)
            dL[b].copy_(hL[b], non_blocking=True)
            loaded[b].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(loaded[b])
            bsm.bs_smooth_bounds(dU[b], dL[b], stream=comp)
            smoothed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(smoothed[b])
            oU[b].copy_(dU[b], non_blocking=True)
            oL[b].copy_(dL[b], non_blocking=True)
            drained[b].record(down)
    t1.record(down)
    torch.cuda.synchronize()
    # the streamed results equal the device-resident ones (sampled rows)
    rows = torch.tensor([0, n // 3, n - 1])
    ref = torch.from_numpy(U0).cuda()
    refL = torch.from_numpy(L0).cuda()
    bsm.bs_smooth_bounds(ref, refL)
    assert torch.equal(oU[0][rows], ref[rows.cuda()].cpu())
    assert torch.equal(oL[(steps - 1) % 2][rows], refL[rows.cuda()].cpu())
    del ref, refL
    ms, units = aggregate(t0.elapsed_time(t1), steps * float(n) ** 3, device="cuda")
    nbytes = 2 * n * n * 4
    return {"value": units / (ms * 1e-3), "unit": UNIT,
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "steps": steps,
            "ms_per_step": ms / steps,
            "h2d_gbs": nbytes / (h2d_ms * 1e-3) / 1e9,
            "exposed": "the first upload and the last download are not overlapped "
                       "(2 x %d bytes over the host link per run)" % nbytes,
            "pipeline": "2 device buffer sets; uploads and downloads on their own streams "
                        "overlap the smoothing of the neighbouring steps"}


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the CSR SpMM engine on one GB300 (or N independent replicas).

A step is one pass of the hot path over the workload: one spmm_run per
(N, reduce) pair the workload lists, each preceded by an L2 flush (a write of
twice the L2 size) so that every timed launch reads its inputs from HBM. The
plan (descriptors, heavy-row tables, workspace) is built before timing, as a
GNN layer reuses it. Device time comes from CUDA events around each run on
the launching stream; value = sum of 2*nnz*N over the timed runs / that time.

Default workload: the largest configuration, a Chung-Lu power-law graph with
M = K = 4,194,304 (degree exponent 2.1, mean 25, capped at 100,000; ids
randomly permuted; about 105M weighted entries), N in {16, 64, 256}, sum,
mean and max + argmax. ``--n`` selects other widths of its sweep
{16, 32, 64, 128, 256}. Beside it the line carries ``per_config``: the sum
runs of the four other workloads (Erdos-Renyi 2k, kNN 1M, R-MAT scale 20,
community 64k), each timed the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

``--impl reference`` times the CPU oracle (the slow, plain fp64 program the
CUDA path is checked against) on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import datetime as _dt
import json
import os
import shutil
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SpMM GFLOP/s (2·nnz·N) and achieved HBM GB/s as % of GB300 peak"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# family's kernels on a workload run, from one ncu capture. The counters belong
# to the kernel build they were taken on: "sources_sha256" is the sha256 of the
# family's sources then, comments and white space left out
# (family_sources_sha256()), and the bench reports the traffic as null once
# they differ.
NCU_TRAFFIC = {
    # the light-row launch k_warprow<4,32,MAX,weighted> (rows of at most 512
    # entries) at full size; the split rows' two launches are not included
    "warprow/chung_lu_4M/N256/max": {"bytes": 34781517056 + 9294084608, "sources_sha256":
                                     "4fe1e81ed6c0338aa67cb3909e45f4eec5a639db4ca1067649b2034bd5cd08a0"},
    "window/knn_1M/N16/sum": {"bytes": 149.09e6, "sources_sha256":
                              "1fe0fed1f8a2523e915205ee6a9478189195e9348ad39b178ca0ae705ed85a50"},
    "window/knn_1M/N16/mean": {"bytes": 148.67e6, "sources_sha256":
                               "1fe0fed1f8a2523e915205ee6a9478189195e9348ad39b178ca0ae705ed85a50"},
    "window/knn_1M/N64/sum": {"bytes": 557.30e6, "sources_sha256":
                              "1fe0fed1f8a2523e915205ee6a9478189195e9348ad39b178ca0ae705ed85a50"},
    "window/knn_1M/N64/mean": {"bytes": 559.95e6, "sources_sha256":
                               "1fe0fed1f8a2523e915205ee6a9478189195e9348ad39b178ca0ae705ed85a50"},
}

_CSRC = "sparse_dense_matrix_gb300/csrc/"
# the sources each family's kernels are built from
FAMILY_SOURCES = {
    "window": (_CSRC + "common.cuh", _CSRC + "tma.cuh", _CSRC + "window.cuh",
               _CSRC + "f_window.cu", _CSRC + "f_window_sum.cu", _CSRC + "f_window_mean.cu",
               _CSRC + "f_window_max.cu", "include/spmm.h"),
    "warprow": (_CSRC + "common.cuh", _CSRC + "f_warprow.cu", "include/spmm.h"),
    "segment": (_CSRC + "common.cuh", _CSRC + "tma.cuh", _CSRC + "segment.cuh",
                _CSRC + "f_segment.cu", _CSRC + "f_segment_sum.cu", _CSRC + "f_segment_max.cu",
                "include/spmm.h"),
    "block": (_CSRC + "common.cuh", _CSRC + "tma.cuh", _CSRC + "f_block.cu", "include/spmm.h"),
    "stream": (_CSRC + "common.cuh", _CSRC + "segment.cuh", _CSRC + "stream.cuh",
               _CSRC + "f_stream.cu", _CSRC + "f_stream_sum.cu", _CSRC + "f_stream_max.cu",
               "include/spmm.h"),
    "gather": (_CSRC + "common.cuh", _CSRC + "tma.cuh", _CSRC + "segment.cuh",
               _CSRC + "gather.cuh", _CSRC + "f_gather.cu", _CSRC + "f_gather_sum.cu",
               _CSRC + "f_gather_max.cu", "include/spmm.h"),
}


def _code_only(text):
    """C/C++/CUDA source without its comments, white space runs collapsed."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                       # string or character literal, kept
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def family_sources_sha256(family):
    h = hashlib.sha256()
    for rel in FAMILY_SOURCES.get(family, ()):
        h.update(rel.encode())
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(key, family):
    """ncu DRAM bytes per launch for a run key, or None (no capture, or the
    family's sources changed since)."""
    ent = NCU_TRAFFIC.get(key)
    if ent is None or family not in FAMILY_SOURCES:
        return None
    return ent["bytes"] if family_sources_sha256(family) == ent["sources_sha256"] else None


FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0    # the ~8 TB/s GB300 HBM3e figure the 60% target is stated against
# widths timed by default where the workload's sweep is longer: its two ends
# and the middle
DEFAULT_N = {5: (16, 64, 256)}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--family", default="auto",
                    choices=["auto", "rowgroup", "warprow", "coltile", "window", "block",
                             "segment", "gather", "stream"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--n", default=None,
                    help="comma-separated feature widths to run (default: all of the workload's)")
    ap.add_argument("--reduce", default=None,
                    help="comma-separated reductions to run (default: all of the workload's)")
    ap.add_argument("--graph-batch", type=int, default=50,
                    help="launches per CUDA graph for the graph-batched figure (0: skip)")
    ap.add_argument("--warm-iters", type=int, default=20,
                    help="back-to-back launches per run for the warm-L2 figure (0: skip)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the sum runs of the other workloads")
    ap.add_argument("--per-config-reps", type=int, default=20)
    return ap.parse_args()


def max_over_ranks(x: float, pg, device=None) -> float:
    """The largest value of x over the ranks (x itself without a process group)."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload(cid, n_sel=None, r_sel=None):
    """The workload's generator spec, its graph and the (N, reduce) runs of one
    step; n_sel / r_sel restrict the runs to a comma-separated subset."""
    import gen
    spec = gen.CONFIGS[cid]
    Ns = DEFAULT_N.get(cid, spec["N"]) if n_sel is None else [int(x) for x in n_sel.split(",")]
    Rs = spec["reduce"] if r_sel is None else r_sel.split(",")
    bad = [n for n in Ns if n not in spec["N"]] + [r for r in Rs if r not in spec["reduce"]]
    if bad:
        raise SystemExit(f"--n/--reduce: {bad} not in {spec['name']} "
                         f"(N {spec['N']}, reduce {spec['reduce']})")
    g = gen.config(cid)
    runs = [(n, r) for n in Ns for r in Rs]
    spec = dict(spec, N=Ns, reduce=Rs)
    return spec, g, runs


def compulsory_bytes(g, N, reduce):
    """rowptr + col + val + B read once + C written (+ argmax for max)."""
    b = 4 * (g.M + 1) + 4 * g.nnz + (4 * g.nnz if g.val is not None else 0)
    b += 4 * g.K * N + 4 * g.M * N
    if reduce == "max":
        b += 4 * g.M * N
    return b


def describe_workload(spec, g, runs):
    return (f"{spec['name']}: M={g.M:,} K={g.K:,} nnz={g.nnz:,} "
            f"{'weighted' if g.val is not None else 'unweighted'}; "
            f"runs per step: " + ", ".join(f"N={n} {r}" for n, r in runs))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        if shutil.which("nvidia-smi") is None:
            return
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="spmm_clocks_", suffix=".csv")
        self.f = os.fdopen(fd, "w")
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
            stderr=subprocess.DEVNULL)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        sm, smax, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            n += 1
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                pass
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n}


def time_oracle(g, B_by_N, runs, rows, budget_s, min_reps=1):
    """Oracle wall time for the given rows over all runs, repeated to fill budget_s."""
    import oracle
    reps, t_total = 0, 0.0
    while True:
        t0 = time.perf_counter()
        for n, r in runs:
            oracle.spmm(g.rowptr, g.col, g.val, B_by_N[n], r, rows=rows)
        t_total += time.perf_counter() - t0
        reps += 1
        if reps >= min_reps and t_total >= budget_s:
            break
        if reps >= min_reps and t_total / reps * (reps + 1) > 3 * budget_s:
            break
    return t_total / reps, reps


def sample_rows(g, frac, seed=0):
    n = max(1, int(round(g.M * frac)))
    if n >= g.M:
        return None, g.nnz
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(g.M, size=n, replace=False)).astype(np.int64)
    deg = np.diff(g.rowptr.astype(np.int64))
    return rows, int(deg[rows].sum())


def cpu_leg(g, B_by_N, runs, budget_s):
    """Size a row sample so that one pass over all runs takes about budget_s / 3."""
    import oracle
    probe_rows, probe_nnz = sample_rows(g, min(1.0, 20000 / max(g.M, 1)), seed=1)
    t_probe, _ = time_oracle(g, B_by_N, runs, probe_rows, 0.0)
    frac = min(1.0, (budget_s / 3) / max(t_probe, 1e-6) * (20000 / max(g.M, 1)))
    rows, nnz_s = sample_rows(g, frac, seed=2)
    t, reps = time_oracle(g, B_by_N, runs, rows, budget_s)
    flops = sum(2.0 * nnz_s * n for n, _ in runs)
    desc = (f"{'all' if rows is None else f'{len(rows):,} random'} rows of {g.M:,} "
            f"({nnz_s:,} entries), every run of the step, {reps} repetition(s)")
    return flops / t / 1e9, t, desc, oracle.threads()


def run_reference(args):
    world, rank, _, pg = dist_init(args)
    if rank != 0:
        return
    spec, g, runs = workload(args.config, args.n, args.reduce)
    import gen
    B_by_N = {n: gen.features(g.K, n, seed=0) for n in spec["N"]}
    # each step: a row sample sized so that W + K steps end within ~2 minutes
    budget_total = args.ref_budget
    per_step = budget_total / max(1, args.steps + args.warmup)
    import oracle
    probe_rows, _ = sample_rows(g, min(1.0, 2000 / max(g.M, 1)), seed=1)
    t_probe, _ = time_oracle(g, B_by_N, runs, probe_rows, 0.0)
    frac = min(1.0, per_step / max(t_probe, 1e-6) * (2000 / max(g.M, 1)))
    rows, nnz_s = sample_rows(g, frac, seed=3)
    for _ in range(args.warmup):
        for n, r in runs:
            oracle.spmm(g.rowptr, g.col, g.val, B_by_N[n], r, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for n, r in runs:
            oracle.spmm(g.rowptr, g.col, g.val, B_by_N[n], r, rows=rows)
    dt = time.perf_counter() - t0
    flops = sum(2.0 * nnz_s * n for n, _ in runs) * args.steps
    value = flops / dt / 1e9
    sample = (f"{'all' if rows is None else f'{len(rows):,} random'} rows of {g.M:,} "
              f"({nnz_s:,} entries) per step, every run of the step")
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe_workload(spec, g, runs)},
        "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def other_configs(sdm, dev, cids, reps, flush_l2, stream, hbm_peak):
    """The sum runs of other workloads, timed like the bench's own runs (L2
    flushed before each launch, CUDA events, median of `reps`)."""
    import torch
    import gen
    out = []
    for cid in cids:
        spec = gen.CONFIGS[cid]
        if "sum" not in spec["reduce"]:
            continue
        g = gen.config(cid)
        rp = torch.from_numpy(g.rowptr).to(dev)
        cl = torch.from_numpy(g.col).to(dev)
        vl = None if g.val is None else torch.from_numpy(g.val).to(dev)
        adj = sdm.SparseAdj(rp, cl, vl, num_cols=g.K)
        for n in spec["N"]:
            Bd = torch.from_numpy(gen.features(g.K, n, seed=0)).to(dev)
            Cd = torch.empty((g.M, n), dtype=torch.float32, device=dev)
            adj.reserve(n, "sum")
            for _ in range(3):
                adj.reduce(Bd, "sum", out=Cd, stream=stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for a, b in evs:
                flush_l2()
                a.record(stream)
                adj.reduce(Bd, "sum", out=Cd, stream=stream)
                b.record(stream)
            torch.cuda.synchronize()
            ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
            by = compulsory_bytes(g, n, "sum")
            out.append({"workload": spec["name"], "N": n, "reduce": "sum",
                        "family": adj.describe(n, "sum")["family_name"], "ms": ms,
                        "gflops": 2.0 * g.nnz * n / (ms / 1e3) / 1e9,
                        "hbm_frac": by / (ms / 1e3) / 1e9 / hbm_peak,
                        "hbm_frac_nominal": by / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS})
            del Bd, Cd
        adj.close()
        del rp, cl, vl
    torch.cuda.synchronize()
    return out


def run_ours(args):
    import torch
    world, rank, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sparse_dense_matrix_gb300 as sdm

    spec, g, runs = workload(args.config, args.n, args.reduce)
    import gen
    Ns = spec["N"]
    B_host = {n: gen.features(g.K, n, seed=0) for n in Ns}
    rowptr = torch.from_numpy(g.rowptr).to(dev)
    col = torch.from_numpy(g.col).to(dev)
    val = None if g.val is None else torch.from_numpy(g.val).to(dev)
    # cold path: plan creation (descriptor pass, heavy-row tables, routing) and
    # the column check / column-spread pass, each timed on its own
    torch.cuda.synchronize()
    t_p0 = time.perf_counter()
    plan = sdm.spmm_plan_create(rowptr.data_ptr(), g.M, g.K)
    torch.cuda.synchronize()
    t_p1 = time.perf_counter()
    sdm.spmm_plan_validate_cols(plan, col.data_ptr())
    t_p2 = time.perf_counter()
    sdm.spmm_plan_destroy(plan)
    adj = sdm.SparseAdj(rowptr, col, val, num_cols=g.K)
    if args.family != "auto":
        adj.set_family(args.family)
    Bd = {n: torch.from_numpy(B_host[n]).to(dev) for n in Ns}
    Cd = {n: torch.empty((g.M, n), dtype=torch.float32, device=dev) for n in Ns}
    Ad = {n: torch.empty((g.M, n), dtype=torch.int32, device=dev) for n in Ns}
    # first call of the first run (includes any workspace allocation) vs steady state
    n1, r1 = runs[0]
    torch.cuda.synchronize()
    t_f0 = time.perf_counter()
    adj.reduce(Bd[n1], r1, out=Cd[n1], argmax=Ad[n1] if r1 == "max" else None)
    torch.cuda.synchronize()
    first_ms = (time.perf_counter() - t_f0) * 1e3
    for n, r in runs:
        adj.reserve(n, r)
    cold = {"plan_create_ms": (t_p1 - t_p0) * 1e3, "validate_cols_ms": (t_p2 - t_p1) * 1e3,
            "first_call_ms": first_ms, "first_call_run": f"N={n1} {r1}",
            "timing": "wall clock, synchronised on both sides"}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one(n, r, on=None):
        sdm.spmm_run(adj.plan, col.data_ptr(), None if val is None else val.data_ptr(),
                     Bd[n].data_ptr(), n, sdm.REDUCE[r], Cd[n].data_ptr(),
                     Ad[n].data_ptr() if r == "max" else None, stream if on is None else on)

    def flush_l2():
        # overwrite L2, then hold the stream ~50 us so that the host has enqueued
        # the start event and the launch before the GPU reaches them
        flush.fill_(1.0)
        torch.cuda._sleep(100_000)

    for _ in range(args.warmup):
        for n, r in runs:
            flush_l2()
            one(n, r)
    torch.cuda.synchronize()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in runs] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    launches0 = sdm.spmm_launch_count()
    t0 = time.time()
    for s in range(args.steps):
        for k, (n, r) in enumerate(runs):
            flush_l2()
            ev[s][k][0].record(stream)
            one(n, r)
            ev[s][k][1].record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    t1 = time.time()
    launches = sdm.spmm_launch_count() - launches0
    # nvidia-smi samples every 100 ms: when the timed steps took less than a
    # second, the same steps run on (untimed, same work) with the sampler still
    # going until one second has passed, so that the clock record covers them
    t_clk = t1
    extra = 0
    while t_clk - t0 < 1.0:
        for n, r in runs:
            flush_l2()
            one(n, r)
        torch.cuda.synchronize()
        extra += 1
        t_clk = time.time()
    sdm.spmm_plan_sync(adj.plan)
    clk = clocks.stop(t0, t_clk)
    clk["region_s"] = t_clk - t0
    clk["region"] = (f"the {args.steps} timed steps" +
                     (f" and {extra} more untimed steps of the same work" if extra else ""))

    # Warm-L2 figure, outside the timed region and not part of value: each run
    # launched back to back without the flush, so B, col and C stay in L2 as far
    # as they fit.
    warm_ms = [None] * len(runs)
    if args.warm_iters > 0:
        wev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.warm_iters)] for _ in runs]
        for k, (n, r) in enumerate(runs):
            one(n, r)
            for a, b in wev[k]:
                a.record(stream)
                one(n, r)
                b.record(stream)
        torch.cuda.synchronize()
        warm_ms = [float(np.median([a.elapsed_time(b) for a, b in wev[k]]))
                   for k in range(len(runs))]

    # CUDA-graph figure, also outside the timed region and not part of value:
    # G launches of each run captured back to back in one graph and replayed,
    # so a small problem is timed without the per-launch CPU and launch gaps
    # (warm L2). For a workload of well under a megabyte (the 2k-row graph)
    # this is the figure that the launch overhead otherwise hides.
    graph_ms = [None] * len(runs)
    graph_nb = [None] * len(runs)
    graph_note = None
    mean_run_ms = np.array([[a.elapsed_time(b) for a, b in ev[s_]] for s_ in range(args.steps)]).mean(axis=0)
    if args.graph_batch > 0:
        try:
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            for k, (n, r) in enumerate(runs):
                # about 5 ms of launches per graph (at most --graph-batch)
                nb = int(max(1, min(args.graph_batch, round(5.0 / max(mean_run_ms[k], 1e-3)))))
                cg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(cg, stream=gs, capture_error_mode="relaxed"):
                    for _ in range(nb):
                        one(n, r, gs)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(gs):
                    cg.replay()
                    e0.record(gs)
                    cg.replay()
                    e1.record(gs)
                torch.cuda.synchronize()
                graph_ms[k] = e0.elapsed_time(e1) / nb
                graph_nb[k] = nb
                del cg
        except Exception as exc:     # capture unsupported here: report why, keep the line
            graph_ms = [None] * len(runs)
            graph_note = f"not measured: {type(exc).__name__}: {exc}"[:200]
        torch.cuda.synchronize()

    per_run_ms = np.array([[a.elapsed_time(b) for a, b in ev[s]] for s in range(args.steps)])
    dev_ms = float(per_run_ms.sum())
    if pg is not None:
        dev_ms = max_over_ranks(dev_ms, pg, dev)
    flops_step = sum(2.0 * g.nnz * n for n, _ in runs)
    value = flops_step * args.steps * world / (dev_ms / 1e3) / 1e9

    hbm_peak, peak_kind = peaks()
    # dominant kernel: the run with the largest median device time
    med_ms = np.median(per_run_ms, axis=0)
    kdom = int(np.argmax(med_ms))
    n_dom, r_dom = runs[kdom]
    info = adj.describe(n_dom, r_dom)
    bytes_dom = compulsory_bytes(g, n_dom, r_dom)
    achieved = bytes_dom / (med_ms[kdom] / 1e3) / 1e9
    key = f"{info['family_name']}/{spec['name']}/N{n_dom}/{r_dom}"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                "nominal_peak": NOMINAL_HBM_GBS, "duration": "median of the run's steps",
                "traffic": ncu_traffic(key, info["family_name"]),
                "traffic_scope": "dram__bytes_read.sum + dram__bytes_write.sum of the run's "
                                 "main launch (for WARPROW the light rows; its split-row "
                                 "launches are not included), one ncu capture",
                "kernel": key, "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": bytes_dom,
                "launches_per_run": info["launches"]}
    per_run = []
    for k, (n, r) in enumerate(runs):
        b = compulsory_bytes(g, n, r)
        per_run.append({"N": n, "reduce": r, "family": adj.describe(n, r)["family_name"],
                        "ms": float(np.median(per_run_ms[:, k])),
                        "ms_p10": float(np.percentile(per_run_ms[:, k], 10)),
                        "ms_p90": float(np.percentile(per_run_ms[:, k], 90)),
                        "warm_l2_ms": warm_ms[k],
                        "graph_batched_ms": graph_ms[k],
                        "graph_launches": graph_nb[k],
                        "gflops": 2.0 * g.nnz * n / (np.median(per_run_ms[:, k]) / 1e3) / 1e9,
                        "hbm_frac": b / (np.median(per_run_ms[:, k]) / 1e3) / 1e9 / hbm_peak,
                        "hbm_frac_nominal": b / (np.median(per_run_ms[:, k]) / 1e3) / 1e9
                        / NOMINAL_HBM_GBS})

    # End to end through the public API with pinned host buffers: every step
    # copies each feature matrix in once (one per N) and every result out; the
    # copies run on their own streams and overlap the other runs' kernels.
    e2e = None
    if not args.no_e2e:
        Bh = {n: torch.from_numpy(B_host[n]).pin_memory() for n in Ns}
        Ch = [torch.empty((g.M, n), dtype=torch.float32).pin_memory() for n, _ in runs]
        Ah = [torch.empty((g.M, n), dtype=torch.int32).pin_memory() if r == "max" else None
              for n, r in runs]
        Cr = [torch.empty((g.M, n), dtype=torch.float32, device=dev) for n, _ in runs]
        Ar = [torch.empty((g.M, n), dtype=torch.int32, device=dev) if r == "max" else None
              for n, r in runs]
        h2d = sum(g.K * n * 4 for n in Ns)
        d2h = sum(g.M * n * 4 * (2 if r == "max" else 1) for n, r in runs)
        e2e_steps = max(3, min(args.steps, 50))
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        # two sets of device buffers: step k + 1 uploads and computes while step
        # k's results are still being copied out (the link, ~200 GB/s each way,
        # bounds this leg)
        Bset = [Bd, {n: torch.empty_like(Bd[n]) for n in Ns}]
        Cset = [Cr, [torch.empty_like(c) for c in Cr]]
        Aset = [Ar, [None if a_ is None else torch.empty_like(a_) for a_ in Ar]]
        kern_done = [None, None]          # per set: the step's kernels are done
        out_done = [[None] * len(runs), [None] * len(runs)]   # per set and run: copied out
        it = [0]

        def e2e_step():
            b = it[0] % 2
            it[0] += 1
            ready = {}
            with torch.cuda.stream(s_in):
                if kern_done[b] is not None:
                    s_in.wait_event(kern_done[b])      # the buffers' previous readers
                for n in Ns:
                    Bset[b][n].copy_(Bh[n], non_blocking=True)
                    ready[n] = torch.cuda.Event()
                    ready[n].record(s_in)
            for k, (n, r) in enumerate(runs):
                stream.wait_event(ready[n])
                if out_done[b][k] is not None:
                    stream.wait_event(out_done[b][k])  # the previous copy-out of this buffer
                adj.reduce(Bset[b][n], r, out=Cset[b][k], argmax=Aset[b][k], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    Ch[k].copy_(Cset[b][k], non_blocking=True)
                    if Aset[b][k] is not None:
                        Ah[k].copy_(Aset[b][k], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_out)
                    out_done[b][k] = ev
            kd = torch.cuda.Event()
            kd.record(stream)
            kern_done[b] = kd

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        t_e0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t_e0) * 1e3
        e2e = {"value": flops_step * e2e_steps * world / (e2e_ms / 1e3) / 1e9, "unit": "GFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
               "timing": "wall clock, synchronised on both sides; two buffer sets, so copies "
                         "in, kernels and copies out of consecutive steps overlap"}

    # Reuse break-even: the plan-free entry point (spmm_run_noalloc, which
    # finds the split rows on every call) against the planned call; the plan
    # and its column check pay for themselves after break_even_calls calls.
    try:
        Cn = torch.empty_like(Cd[n1])
        An = torch.empty_like(Ad[n1]) if r1 == "max" else None

        def noalloc():
            sdm.spmm_run_noalloc(rowptr.data_ptr(), col.data_ptr(),
                                 None if val is None else val.data_ptr(), Bd[n1].data_ptr(),
                                 g.M, g.K, n1, sdm.REDUCE[r1], Cn.data_ptr(),
                                 None if An is None else An.data_ptr(), stream)
        noalloc()
        ts_ = []
        for _ in range(5):
            flush_l2()
            torch.cuda.synchronize()
            t_a = time.perf_counter()
            noalloc()
            torch.cuda.synchronize()
            ts_.append((time.perf_counter() - t_a) * 1e3)
        ts_p = []
        for _ in range(5):
            flush_l2()
            torch.cuda.synchronize()
            t_a = time.perf_counter()
            one(n1, r1)
            torch.cuda.synchronize()
            ts_p.append((time.perf_counter() - t_a) * 1e3)
        na_ms, pl_ms = float(np.median(ts_)), float(np.median(ts_p))
        gain = na_ms - pl_ms
        plan_cost = cold["plan_create_ms"] + cold["validate_cols_ms"]
        cold.update({"noalloc_call_ms": na_ms, "planned_call_ms": pl_ms,
                     "break_even_calls": (plan_cost / gain) if gain > 0 else None,
                     "break_even": f"(plan_create_ms + validate_cols_ms) / (noalloc_call_ms - "
                                   f"planned_call_ms) for N={n1} {r1}, both calls wall clock "
                                   "after an L2 flush; null when the plan-free call is not "
                                   "slower"})
        del Cn, An
    except Exception as exc:
        cold["break_even"] = f"not measured: {type(exc).__name__}: {exc}"[:200]

    per_config = None
    if not args.no_per_config:
        per_config = other_configs(sdm, dev, [c for c in (1, 2, 3, 4) if c != args.config],
                                   args.per_config_reps, flush_l2, stream, hbm_peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, t, desc, cores = cpu_leg(g, B_host, runs, budget_s=15.0)
        cpu = {"value": v, "unit": "GFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dev_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": describe_workload(spec, g, runs),
                       "l2": "flushed (write of 2x L2) before every timed launch",
                       "timing": "CUDA events around each spmm_run on the launching stream; "
                                 "per_run ms is the median over steps, with p10 and p90",
                       "warm_l2": "per_run warm_l2_ms: back-to-back launches without the "
                                  "flush, after the timed region; not part of value",
                       "graph_batched": graph_note or (
                           "per_run graph_batched_ms: per-launch time of graph_launches "
                           "launches (about 5 ms of work, at most "
                           f"{args.graph_batch}) captured in one CUDA graph (warm L2, no "
                           "launch gaps), after the timed region; not part of value"),
                       "per_run": per_run,
                       "per_config": "per_config: the sum runs of the other workloads, each "
                                     "timed as the runs above (median of "
                                     f"{args.per_config_reps}); not part of value"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "per_config": per_config,
            "gpu_launches": int(launches), "clocks": clk, "cold_path": cold,
            "hbm_gbs_compulsory": sum(compulsory_bytes(g, n, r) for n, r in runs) * args.steps
            / (dev_ms / 1e3) / 1e9,
        }
        print(json.dumps(out))
    adj.close()
    if pg is not None:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

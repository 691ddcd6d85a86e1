#!/usr/bin/env python3
"""Benchmark: PageRank power iteration on GB300, whole hot path per step.

One step = pr_graph_create from an out-edge CSR already resident in HBM (GPU
transpose, degree classes) + pr_run to L1 < tol (every update on the device in
one CUDA-graph launch). Default workload: RMAT scale 24, edge factor 16,
a/b/c/d = .57/.19/.19/.05, seed 4 (deduplicated, no self-loops), d = 0.85, fp32,
tol 1e-6, at most 200 updates.

value = edges traversed per second over the whole step, in GTEPS:
m * updates / step time, the one-time transpose included. The line also
carries the iteration-only rate (m / time per update), the time to converge,
the roofline of the dominant kernel (the fused update), the end-to-end figure
through the C ABI with host buffers, and the oracle timed on the host cores.

Multi-GPU: replicas only (one independent solve per GPU, no collective on the
data path); value = all ranks' edges / the slowest rank's time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "PageRank GTEPS/iteration and time-to-converge; % of HBM roofline"
UNIT = "GTEPS"
GATHER_PROBE = 1 << 27   # gathers per pass of the gather-rate measurement
GRAPH_DESC = {
    "rmat24": "RMAT scale 24, edge factor 16, a/b/c/d=.57/.19/.19/.05, seed 4, dedup, no self-loops",
    "rmat22": "RMAT scale 22, edge factor 16, a/b/c/d=.57/.19/.19/.05, seed 3, dedup, no self-loops",
    "rmat18": "RMAT scale 18, edge factor 16, a/b/c/d=.57/.19/.19/.05, seed 2, dedup, no self-loops",
    "er24": "Erdos-Renyi n=2^24, 10% dangling, out-degree 16 distinct uniform targets, seed 5",
    "citation30k": "citation-like n=30000, seed 1, 7.9% dangling, out-degree ~k^-2.1 on [3,500], "
                   "preferential attachment to earlier vertices",
}
L2_BYTES = 126 * 1024 * 1024


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="rmat24", choices=sorted(GRAPH_DESC))
    p.add_argument("--dtype", choices=["f32", "f64"], default="f32")
    p.add_argument("--tol", type=float, default=1e-6)
    p.add_argument("--max-iter", type=int, default=200)
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-updates", type=int, default=2,
                   help="updates in the oracle's CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-library", action="store_true",
                   help="skip the library-composed comparator (torch sort + cuSPARSE SpMV)")
    return p.parse_args(argv)


# ------------------------------------------------------------ small pieces --

def bytes_model(n: int, m: int) -> dict:
    """Algorithmic bytes of one update.

    b_spmv: row_ptr 4(n+1) + col_idx 4m + one 4-byte gather per edge 4m + y 4n
            (the per-edge gather convention that reproduces the Day 40 page's
            printed per-iteration byte counts).
    b_floor: the same with each gathered value counted once (4n instead of 4m).
    """
    return {"b_spmv": 4 * (n + 1) + 8 * m + 4 * n, "b_floor": 4 * (n + 1) + 4 * m + 8 * n}


def build_bytes(n: int, m: int) -> int:
    """Algorithmic bytes of the one-time transpose, as the counting sort of the
    Day 40 page ("One iteration, three shapes of work") moves them: the
    in-degree histogram reads col_idx (4m), the exclusive scan reads the counts
    and writes in_ptr (8n), the scatter reads row_ptr and col_idx and writes
    in_col (8n + 8m)."""
    return 12 * m + 16 * n


def day40_bytes(n: int, nnz: int) -> dict:
    """Per-iteration bytes of the Day 40 page's two implementations (4-byte
    values, 1-byte dangling mask): hand-written 8 nnz + 33 n + 4; the library
    path adds the materialised gather (8 nnz) and masked vector (8 n)."""
    hand = 8 * nnz + 33 * n + 4
    return {"hand": hand, "library": hand + 8 * nnz + 8 * n}


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return 6800.0, "fallback"


def code_digest(text: str) -> str:
    """sha256 (first 16 hex digits) of C/CUDA source with its comments, blank
    lines and trailing spaces removed, so that editing a comment does not
    orphan a profile taken on the same code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()[:16]


def kernel_source_digest() -> str:
    """Code digest of the update kernel's device code: iterate.cu up to its host
    side (which starts at make_args), and the header it includes."""
    csrc = os.path.join(ROOT, "pagerank_power_iteration_gb300", "csrc")
    it = open(os.path.join(csrc, "iterate.cu")).read()
    cut = it.find("IterArgs<T> make_args(pr_graph *g)")
    device = it[:cut] if cut >= 0 else it
    return code_digest(device + open(os.path.join(csrc, "pr_internal.cuh")).read())


def profiled_traffic(workload: str):
    """DRAM bytes per update of k_iterate from the committed ncu record
    profiles/k_iterate_<workload>.json, if it was taken on the current kernel
    source; else None. Returns (bytes per update, the record)."""
    path = os.path.join(ROOT, "profiles", f"k_iterate_{workload}.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_digest") != kernel_source_digest():
        return None, None
    return float(rec["dram_bytes_per_update"]), rec


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, uuid: str | None):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        target = uuid if uuid else str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", target], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        loaded = [r for r in rows if (num(r[2]) or 0) > 20] or rows
        sm = [num(r[0]) for r in loaded if num(r[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(loaded[0][1]), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded)}


def host_info():
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        model = m.group(1).strip() if m else None
    except Exception:
        pass
    return {"cpu_model": model, "host_cores": os.cpu_count()}


def aggregate(dist, device, slowest_ms: float, edges: float):
    """Whole-job figures across ranks: the slowest rank's time (MAX) and the
    edges all ranks traversed (SUM). Identity without a process group."""
    if dist is None:
        return slowest_ms, edges
    import torch
    t = torch.tensor([slowest_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    e = torch.tensor([float(edges)], dtype=torch.float64, device=device)
    dist.all_reduce(e, op=dist.ReduceOp.SUM)
    return float(t.item()), float(e.item())


# ------------------------------------------------------------- CPU legs ---

def prefix_sample(rp, ci, max_edges):
    """Out-edges of the first sources up to max_edges edges, over all n vertices
    (the remaining vertices keep no out-edge): a prefix of the workload's edge
    stream."""
    if max_edges >= len(ci):
        return rp, ci
    cut = int(np.searchsorted(rp, max_edges, side="right") - 1)
    rs = rp.copy()
    rs[cut + 1:] = rp[cut]
    return rs, ci[: rp[cut]]


def time_oracle(rp, ci, d, updates):
    import oracle
    t0 = time.perf_counter()
    out = oracle.pagerank(rp, ci, d, tol=0.0, max_iter=updates)
    dt = time.perf_counter() - t0
    return dt, out


# --------------------------------------------------------------- our arm ---

def run_ours(args, rank, world, local_rank, dist):
    import torch
    import graphgen as gg
    import pagerank_power_iteration_gb300 as prg
    from pagerank_power_iteration_gb300 import build as prbuild

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    prbuild.build()
    dev = torch.device("cuda", local_rank)
    threads = max(1, (os.cpu_count() or 1) // world)
    t0 = time.perf_counter()
    rp, ci = gg.workload(args.workload, threads=threads)
    gen_s = time.perf_counter() - t0
    n, m = len(rp) - 1, len(ci)
    dcode = prg.PR_F32 if args.dtype == "f32" else prg.PR_F64
    tdt = torch.float32 if args.dtype == "f32" else torch.float64
    d = 0.85

    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    rp_d = torch.from_numpy(rp).to(dev)
    ci_d = torch.from_numpy(ci).to(dev)
    out = torch.empty(n, dtype=tdt, device=dev)

    def step():
        g = prg.pr_graph_create(n, m, rp_d.data_ptr(), ci_d.data_ptr() if m else None, sp)
        try:
            st, it, l1 = prg.pr_run(g, d, args.tol, args.max_iter, dcode, out.data_ptr(), None, sp)
            return it, l1, prg.pr_graph_last_run(g), prg.pr_graph_get_info(g)
        finally:
            prg.pr_graph_destroy(g)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (
        str(uuid) if uuid else None)
    sampler = ClockSampler(local_rank, uuid)
    time.sleep(0.3)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    recs = []
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    w0 = time.perf_counter()
    first = torch.cuda.Event(enable_timing=True)
    last = torch.cuda.Event(enable_timing=True)
    first.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        recs.append(step())
        ev[k][1].record(stream)
    last.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - w0
    clocks = sampler.stop()

    iters = [r[0] for r in recs]
    total_ms, edges_all = aggregate(dist, dev, first.elapsed_time(last),
                                    float(sum(m * it for it in iters)))
    value = edges_all / (total_ms * 1e-3) / 1e9

    stats = [r[2] for r in recs]
    info = recs[-1][3]
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    run_ms = [s["total_ms"] for s in stats]
    per_update_ms = statistics.mean(s["loop_ms"] / max(s["iterations"], 1) for s in stats)
    transpose_ms = statistics.mean(sm - rm for sm, rm in zip(step_ms, run_ms))
    bm = bytes_model(n, m)
    peak, peak_kind = measured_peak_hbm()
    achieved = bm["b_spmv"] / (per_update_ms * 1e-3) / 1e9
    launches = sum(info["build_launches"] + s["launches"] for s in stats)
    build_ms = statistics.mean(r[3]["build_ms"] for r in recs)
    traffic, traffic_rec = profiled_traffic(args.workload)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded generator, host-built CSR copied to HBM before timing)",
        "config": {
            "workload": args.workload, "graph": GRAPH_DESC[args.workload], "n": n, "m": m,
            "d": d, "tol": args.tol, "max_iter": args.max_iter,
            "updates_per_step": iters[-1],
            "step": "pr_graph_create from the device-resident out-CSR (GPU transpose + degree "
                    "classes) + pr_run to L1 < tol; value = m * updates / step time",
            "l2": f"inputs larger than L2 (col_idx {4 * m / 1e9:.2f} GB vs L2 126 MB); no flush",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "iteration_gteps": round(m / (per_update_ms * 1e-3) / 1e9, 3),
        "ms_per_update": round(per_update_ms, 5),
        "time_to_converge_ms": round(statistics.median(run_ms), 4),
        "transpose_ms": round(transpose_ms, 4),
        "gpu_launches": launches,
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "traffic_source": (f"profiles/k_iterate_{args.workload}.json: ncu dram__bytes_read.sum + "
                               f"dram__bytes_write.sum over {traffic_rec['updates']} updates of "
                               f"{traffic_rec['workload']}, per update" if traffic_rec else
                               "null: no ncu record taken on the current kernel source"),
            "kernel": "k_iterate (fused gather SpMV + combine + L1/D reductions, one launch per update)",
            "bytes_per_launch": bm["b_spmv"], "bytes_model": "4(n+1) + 8m + 4n (row_ptr, col_idx, "
            "per-edge gather, y)", "peak_source": f"{peak_kind} hbm_gbs",
            "frac_of_8tbs": round(achieved / 8000.0, 4),
            "frac_floor_bytes": round(bm["b_floor"] / (per_update_ms * 1e-3) / 1e9 / peak, 4),
        },
        "build_roofline": {
            "bound": "hbm", "achieved": round(build_bytes(n, m) / (build_ms * 1e-3) / 1e9, 1),
            "peak": peak, "unit": "GB/s",
            "frac": round(build_bytes(n, m) / (build_ms * 1e-3) / 1e9 / peak, 4),
            "kernel": "pr_graph_create (degrees, edge sources, LSD radix passes by destination, "
                      "in-degree scan, class-major work layout)",
            "bytes_per_build": build_bytes(n, m),
            "bytes_model": "12m + 16n (counting sort: histogram 4m, scan 8n, scatter 8m + 8n)",
            "ms": round(build_ms, 4),
            "ms_source": "pr_graph_info.build_ms: CUDA events on the build's stream, mean over the timed steps",
            "peak_source": f"{peak_kind} hbm_gbs",
        },
        "clocks": clocks,
        "host_wall_s": round(wall, 3), "generate_s": round(gen_s, 2),
    }

    # the bound that holds the update: gathers not served from shared memory,
    # against the random-gather rate of this GPU measured here
    hot = int(info["edges_hot_f32" if args.dtype == "f32" else "edges_hot_f64"])
    l2_gathers = m - hot
    g_peak = prg.pr_measure_gather_rate(n, dcode, GATHER_PROBE, sp, prg.PR_GATHER_LOAD)
    g_ach = l2_gathers / (per_update_ms * 1e-3)
    line["gather_roofline"] = {
        "bound": "l2 random gather", "achieved": round(g_ach / 1e9, 2),
        "peak": round(g_peak / 1e9, 2), "unit": "G gathers/s",
        "frac": round(g_ach / g_peak, 4),
        "l2_gathers_per_update": l2_gathers, "smem_gathers_per_update": hot,
        "peak_source": f"pr_measure_gather_rate: {GATHER_PROBE} uniform random gathers from an "
                       f"{n}-element {args.dtype} state (the run's working set), measured in this run",
    }

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, rp, ci, n, m, dev, tdt, d, dist)
    if rank == 0 and not args.no_library:
        line["library_comparator"] = run_library(rp, ci, d, args.tol, args.max_iter, tdt, dev,
                                                 ours=out, ours_updates=iters[-1])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_multicore"] = time_cpu_parallel(rp, ci, d, args.cpu_updates)
        dt, _ = time_oracle(rp, ci, d, args.cpu_updates)
        line["cpu_baseline"] = {
            "value": round(m * args.cpu_updates / dt / 1e9, 5), "unit": UNIT, "cores": 1,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"full {args.workload} graph: the oracle's counting-sort transpose + "
                      f"{args.cpu_updates} fixed fp64 updates, single thread",
            **host_info(),
        }
    return line


def time_cpu_parallel(rp, ci, d, updates):
    """The multi-core CPU baseline (OpenMP pull, fp64, all host cores) on the full
    workload: its parallel transpose plus a fixed number of updates."""
    import cpu_parallel
    cpu_parallel.build()
    m = len(ci)
    r = cpu_parallel.pagerank(rp, ci, d, tol=0.0, max_iter=updates)
    return {"value": round(m * r["iters"] / r["t_loop"] / 1e9, 4), "unit": UNIT, "cores": r["threads"],
            "kind": "openmp pull over the in-edge CSR, fp64", "transpose_s": round(r["t_transpose"], 3),
            "loop_s": round(r["t_loop"], 3),
            "step_gteps": round(m * r["iters"] / (r["t_transpose"] + r["t_loop"]) / 1e9, 4),
            "sample": f"full graph: the parallel transpose + {r['iters']} fixed fp64 updates"}


def library_pagerank(rp, ci, d, tol, max_iter, tdt, dev, fixed=None):
    """The same method composed from library calls, timed beside ours: the
    transpose as a library sort of (destination, source) keys, each update as
    a cuSPARSE CSR SpMV (torch.mv on a sparse CSR tensor) over x/outdeg plus
    torch elementwise ops and reductions for the dangling mass, the combine
    and the L1 distance. The loop checks L1 on the host after every update,
    as the library composition of Day 40 does; `fixed` runs exactly that many
    updates with no check. Returns (x, updates, transpose_ms, loop_ms)."""
    import torch
    n, m = len(rp) - 1, len(ci)
    outdeg = torch.from_numpy(np.diff(rp)).to(dev)
    start, mid, end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize(dev)
    start.record()
    dst = torch.from_numpy(ci).to(dev).long()
    src = torch.repeat_interleave(torch.arange(n, device=dev), outdeg)
    key, _ = torch.sort(dst * n + src)
    crow = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    crow[1:] = torch.cumsum(torch.bincount(dst, minlength=n), 0)
    a = torch.sparse_csr_tensor(crow, key % n, torch.ones(m, dtype=tdt, device=dev), size=(n, n))
    del key, src, dst
    mid.record()
    dang = (outdeg == 0).to(tdt)
    inv = torch.where(outdeg > 0, 1.0 / outdeg.clamp(min=1).to(tdt), torch.zeros((), dtype=tdt, device=dev))
    x = torch.full((n,), 1.0 / n, dtype=tdt, device=dev)
    updates = 0
    while updates < (fixed or max_iter):
        y = torch.mv(a, x * inv)
        dm = torch.dot(x, dang)
        xn = (1.0 - d) / n + d * (y + dm / n)
        l1 = torch.sum(torch.abs(xn - x))
        x = xn
        updates += 1
        if fixed is None and tol > 0 and float(l1) < tol:
            break
    end.record()
    torch.cuda.synchronize(dev)
    return x, updates, start.elapsed_time(mid), mid.elapsed_time(end)


def run_library(rp, ci, d, tol, max_iter, tdt, dev, ours=None, ours_updates=None):
    """Library-composed comparator: a warm-up call, then the best of two timed calls."""
    import torch
    m = len(ci)
    library_pagerank(rp, ci, d, tol, max_iter, tdt, dev, fixed=2)
    runs = [library_pagerank(rp, ci, d, tol, max_iter, tdt, dev) for _ in range(2)]
    x, ups = runs[-1][0], runs[-1][1]
    t_ms, loop_ms = min(r[2] for r in runs), min(r[3] for r in runs)
    res = {"impl": "torch.sort transpose + cuSPARSE CSR SpMV (torch.mv) + torch elementwise and "
                   "reductions; L1 read on the host after every update",
           "updates": ups, "transpose_ms": round(t_ms, 3), "time_to_converge_ms": round(loop_ms, 3),
           "ms_per_update": round(loop_ms / max(ups, 1), 5),
           "iteration_gteps": round(m * ups / (loop_ms * 1e-3) / 1e9, 3),
           "step_gteps": round(m * ups / ((t_ms + loop_ms) * 1e-3) / 1e9, 3)}
    if ours is not None and ours_updates == ups:
        xo = ours.to(x.dtype)
        res["max_rel_diff_vs_ours"] = float(torch.max(torch.abs(x - xo) / torch.clamp(torch.abs(xo), min=1e-30)))
    return res


def run_e2e(args, rp, ci, n, m, dev, tdt, d, dist):
    """Same metric through the public API with pinned host buffers: the H2D copy
    of the CSR and the D2H copy of the ranks are inside every step."""
    import torch
    import pagerank_power_iteration_gb300 as prg
    rp_h = torch.from_numpy(rp).pin_memory()
    ci_h = torch.from_numpy(ci).pin_memory()
    out_h = torch.empty(n, dtype=tdt).pin_memory()
    k = max(1, args.e2e_steps)
    torch.cuda.synchronize(dev)
    # as many warm-up steps as the device-timed leg: the first steps through the
    # host path grow the library's memory pool by the staging buffers of the CSR
    for _ in range(max(3, args.warmup)):
        g = prg.Graph(rp_h, ci_h)
        g.run(d, args.tol, args.max_iter, dtype=tdt, out=out_h)
        g.close()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    edges = 0
    step_ms, create_ms = [], []
    t0 = time.perf_counter()
    for _ in range(k):
        ts = time.perf_counter()
        g = prg.Graph(rp_h, ci_h)   # returns once the build (and its H2D copy) is done
        tc = time.perf_counter()
        _, it, _, _ = g.run(d, args.tol, args.max_iter, dtype=tdt, out=out_h)   # synchronises
        g.close()
        torch.cuda.synchronize(dev)   # the step ends when its frees have landed too
        te = time.perf_counter()
        step_ms.append((te - ts) * 1e3)
        create_ms.append((tc - ts) * 1e3)
        edges += m * it
    torch.cuda.synchronize(dev)
    ms, edges = aggregate(dist, dev, (time.perf_counter() - t0) * 1e3, float(edges))
    dt = ms * 1e-3
    elt = torch.finfo(tdt).bits // 8
    return {"value": round(edges / dt / 1e9, 3), "unit": UNIT,
            "h2d_bytes_per_step": 8 * (n + 1) + 4 * m, "d2h_bytes_per_step": elt * n,
            "steps": k, "ms_per_step": round(dt / k * 1e3, 3),
            "ms_per_step_median": round(sorted(step_ms)[len(step_ms) // 2], 3),
            "step_ms_min_max": [round(min(step_ms), 3), round(max(step_ms), 3)],
            "step_ms": [round(x, 3) for x in step_ms],
            "create_ms": [round(x, 3) for x in create_ms],   # of step_ms: Graph() from host memory
            "warmup": max(3, args.warmup),
            "api": "Graph(pinned host CSR) + Graph.run(out=pinned host tensor)"}


# ---------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is one oracle call
    (counting-sort transpose + one fp64 update) on a prefix sample of the
    workload's edge stream, sized so that warmup + steps stay within ~2 minutes."""
    import graphgen as gg
    import oracle
    oracle.build()
    rp, ci = gg.workload(args.workload)
    n, m = len(rp) - 1, len(ci)
    total_steps = max(1, args.steps + args.warmup)
    # calibrate: cost per edge of one call on a small prefix
    probe_rp, probe_ci = prefix_sample(rp, ci, min(m, 4_000_000))
    dt, _ = time_oracle(probe_rp, probe_ci, 0.85, 1)
    per_edge = dt / max(len(probe_ci), 1)
    budget = 100.0 / total_steps
    sample_edges = int(min(m, max(1_000_000, budget / max(per_edge, 1e-12))))
    srp, sci = prefix_sample(rp, ci, sample_edges)
    ms = len(sci)
    for _ in range(args.warmup):
        time_oracle(srp, sci, 0.85, 1)
    times = []
    for _ in range(args.steps):
        t, _ = time_oracle(srp, sci, 0.85, 1)
        times.append(t)
    total = sum(times)
    value = ms * len(times) / total / 1e9
    sample = (f"{args.workload} (n={n}, m={m}): first {ms} edges of the out-CSR over all n vertices; "
              "per step the oracle's counting-sort transpose + 1 fp64 update, single thread")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / len(times) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "graph": GRAPH_DESC[args.workload], "n": n, "m": m,
                   "d": 0.85, "sample_edges": ms},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, **host_info()},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main ---

def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE",
              file=sys.stderr)

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        tdist.init_process_group(backend=backend)
        dist = tdist
    try:
        line = run_ours(args, rank, world, local_rank, dist)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if dist is not None:
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

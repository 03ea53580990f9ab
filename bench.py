#!/usr/bin/env python
"""Benchmark of the 3D Gaussian Splatting training step on GB300.

Workload: 3,000,000 Gaussians in 256 clusters, a batch of 4 cameras at
1920x1080 on a 30 m ring, SH degree 3, L1 loss, dense Adam over the 59
parameters (the 1080p / 3M-Gaussian configuration the headline metric is
quoted on).  Synthetic, seeded inputs (no dataset).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` = train iterations/s over the whole
job; the fwd+bwd compositing rate (Mpix/s) and Gaussians/s are extra keys.
Multi-GPU runs are independent replicas (the step has no exchange on one
GPU), so value = N x iterations / max-over-ranks time ("scaling": "weak").
--impl reference times the CPU oracle (the plain reference implementation of
the method) on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "ring_3m_4x1080p"
METRIC = "train iters/s and fwd+bwd Mpix/s at 1080p/3M Gaussians; % HBM roofline"
UNIT = "iters/s"

# Algorithmic work per unit: the flops and bytes each kernel's roofline counts.
# Compositing, the method's count (the roofline's `frac`): 14 FP32 operations
# (+1 exp) per tested pair of the forward -- every list entry a pixel passes
# before it stops -- and 45 (+1 exp, +1 reciprocal) per pair the backward
# evaluates -- every list entry below the pixel's last contributor.
FWD_FLOP_PAIR = 14
BWD_FLOP_PAIR = 45
# The arithmetic the method needs on those pairs (`frac_useful`): the exponent
# and alpha test of every tested or evaluated pair, and the compositing and
# gradient arithmetic only of the pairs that pass the 1/255 test.
FWD_FLOP_TESTED = 13     # per tested pair: dx, dy, power, alpha (+1 exp)
FWD_FLOP_INCLUDED = 9    # per composited pair: transmittance, weight, colour
BWD_FLOP_EVAL = 13       # per pair visited below the last contributor (+1 exp)
BWD_FLOP_INCLUDED = 44   # per contributing pair: gradients of colour, alpha, geometry
PROJ_READ = 236          # B per Gaussian: 59 fp32 parameters
SPLAT_BYTES = 48         # B per visible (view, Gaussian) row
CULLED_BYTES = 4         # B per culled row (its tile count)
ADAM_BYTES = 59 * 28     # B per Gaussian: read p, g, m, v; write p, m, v
LOSS_BYTES = 36          # B per pixel: image, target read, gradient written (3 channels)
PROJ_BWD_BYTES = 472     # B per Gaussian: parameters read, gradient written
PROJ_BWD_ROW = 60        # B per visible row: 36 gradient + 24 conic/colour
PROJ_BWD_COUNT = 4       # B per row: its tile count, read to find the visible rows
ZERO_ROW = 4             # B per row: its tile count, read to find the visible rows
ZERO_VISIBLE = 48        # B per visible row: its gradient record zeroed
# binning: every row's tile count (4 B) is read; a visible row's record
# (mean, radius, depth: 32 B) read and its sort element and rectangle written
# (16 B), 4 depth passes (16 B each), its sorted element and rectangle read at
# emission (16 B) and its (depth, id) word written there in depth order (8 B);
# an intersection written at emission (8 B), 16 B per tile pass (read +
# write), in the last one its row's (depth, id) word read and 4 B more written
# (ids; the tile ranges are marked by that pass)
BIN_ROW = 4
BIN_VISIBLE = 32 + 24 + 4 * 16 + 16
BIN_ISECT = 8 + 8 + 4

FP32_LANES_PER_SM = 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prune", type=int, default=None, metavar="K",
                    help="prune once to a per-tile working set of K entries before timing")
    ap.add_argument("--prune-tau", type=float, default=2.0,
                    help="quality floor of the pruning (> 1: none)")
    ap.add_argument("--morton", action="store_true",
                    help="rename the Gaussians in Morton order of their means before timing")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls only (default: the step captured once in a CUDA graph "
                         "and replayed is the headline; eager calls give the per-kernel breakdown)")
    ap.add_argument("--separate", action="store_true",
                    help="composite with three calls (forward, L1 loss, backward) instead of the "
                         "fused one")
    ap.add_argument("--gaussians", type=int, default=None,
                    help="override the Gaussian count (smaller profiling cases)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank, local_ms, world):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time.  Returns (max ms, units per second)."""
    ms = max_over_ranks(local_ms, world)
    return ms, world * units_per_rank / (ms / 1e3)


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# DRAM bytes (read + write) per call of each timed kernel (for bin_and_sort,
# the sum over its launches), from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum, one pass per launch) of this workload at full size.
# They describe the sources whose SHA-256 are given; for any other source
# the figure is unknown (null).
_RASTER = "gaussian_splatting_differentiable_gs_gb300/csrc/raster.cu"
_PROJECT = "gaussian_splatting_differentiable_gs_gb300/csrc/project.cu"
_BINNING = "gaussian_splatting_differentiable_gs_gb300/csrc/binning.cu"
_ORDER = "gaussian_splatting_differentiable_gs_gb300/csrc/tile_order.cu"
_ADAM = "gaussian_splatting_differentiable_gs_gb300/csrc/adam_loss.cu"
TRAFFIC_WORKLOAD = "ring_3m_4x1080p"
TRAFFIC = {
    # the compositing kernel (the gradient records zeroed before by zero_grads)
    "rasterize_fused": {"sources": {_RASTER: "e6aee4fd328c363750bcb3fa35f70b693788a9d836b1c236da5a7a9441d292dc"},
                        "bytes": 5381000000},
    "zero_grads": {"sources": {_RASTER: "e6aee4fd328c363750bcb3fa35f70b693788a9d836b1c236da5a7a9441d292dc"},
                   "bytes": 534500000},
    "project": {"sources": {_PROJECT: "49e8c0396a45093103dff381a567b2674796aeb8f2d23798e4a195e35670eadb"},
                "bytes": 1256300000},
    "project_bwd": {"sources": {_PROJECT: "49e8c0396a45093103dff381a567b2674796aeb8f2d23798e4a195e35670eadb"},
                    "bytes": 2630000000},
    "adam": {"sources": {_ADAM: "7461d48d4dc14b809b9e6d40c07a06c27730c9e24d506df79ddfc7376091fad1"},
             "bytes": 4895300000},
    # compaction, six radix passes, emission and the tile order (the three small
    # scan and check kernels, under 1 MB together, are not counted)
    "bin_and_sort": {"sources": {_BINNING: "d5f6be1b280038b299141b8d98160fe8282b6ec0d762d72c7fab9c088c3bad13",
                                 _ORDER: "4b863354671176f4c937a4a4dac807b3f8f894266513fd909e3ad5a0edd3317a"},
                     "bytes": 3244500000},
}


def traffic_of(kernel, workload, variant):
    t = TRAFFIC.get(kernel)
    if t is None or workload != TRAFFIC_WORKLOAD or variant:
        return None
    import hashlib
    for src, digest in t["sources"].items():
        try:
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return t["bytes"]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2070.0)), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 2070.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload


SAMPLE_EVERY = 8  # the sampled oracle step: 1/8 of the Gaussians, every 8th non-empty tile


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_lists(cfg, threads, cache):
    """The oracle's own projection and sorted lists of the whole scene (set-up
    of the sampled step, untimed)."""
    import numpy as np

    import oracle
    if "full" not in cache:
        params, cams = cfg["params"], cfg["cams"]
        n, V = params.shape[1], len(cams)
        W, H = cams[0]["width"], cams[0]["height"]
        pr = oracle.project(params.astype(np.float64), cams, threads=threads)
        _, vals, ranges = oracle.bin_and_sort(n, V, pr["mean2d"].astype(np.float32), pr["radius"],
                                              pr["depth"].astype(np.float32), W, H,
                                              threads=threads)
        cache["full"] = (pr, vals, ranges)
    return cache["full"]


def oracle_step(cfg, threads, every, cache, offset=0):
    """One training step of the CPU oracle on `threads` POSIX threads.

    every = 1: the whole step (projection, binning, compositing forward, L1
    loss, compositing backward, projection backward, Adam).  every = k > 1:
    the sampled step -- projection, binning, projection backward and Adam on
    a contiguous 1/k of the Gaussians (their cost is linear in the count,
    scaled by k), compositing forward and backward on every k-th non-empty
    tile of the whole scene's lists taken in list-length order (so the
    sample spans the lengths, which set a tile's cost; scaled by the number
    of non-empty tiles over the sample), the loss on the full batch.
    Returns (seconds of a full step, seconds spent, per-stage seconds, text)."""
    import numpy as np

    import oracle
    params, cams = cfg["params"], cfg["cams"]
    n, V = params.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    t = {}
    if every == 1:
        p64 = params.astype(np.float64)
        t0 = time.perf_counter()
        pr = oracle.project(p64, cams, threads=threads)
        t["project"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        _, vals, ranges = oracle.bin_and_sort(n, V, pr["mean2d"].astype(np.float32), pr["radius"],
                                              pr["depth"].astype(np.float32), W, H,
                                              threads=threads)
        t["bin"] = time.perf_counter() - t0
        sel, sub, pr_sub, lin, tile_scale = None, p64, pr, 1.0, 1.0
    else:
        pr, vals, ranges = oracle_lists(cfg, threads, cache)
        m = max(1, n // every)
        a = (offset * m) % max(1, n - m + 1)
        sub = np.ascontiguousarray(params[:, a:a + m].astype(np.float64))
        t0 = time.perf_counter()
        spr = oracle.project(sub, cams, threads=threads)
        t["project"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.bin_and_sort(m, V, spr["mean2d"].astype(np.float32), spr["radius"],
                            spr["depth"].astype(np.float32), W, H, threads=threads)
        t["bin"] = time.perf_counter() - t0
        lens = ranges[:, 1] - ranges[:, 0]
        nonempty = np.nonzero(lens > 0)[0]
        by_len = nonempty[np.argsort(lens[nonempty], kind="stable")]
        sel = np.sort(by_len[offset % every::every])
        lin = n / m
        tile_scale = nonempty.size / max(1, sel.size)
    t0 = time.perf_counter()
    fw = oracle.raster_fwd(n, V, W, H, pr, vals, ranges, tile_sel=sel, threads=threads)
    t["raster_fwd"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    loss, g_img = oracle.loss_l1(fw["image"], cfg["target"])
    t["loss"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    g2 = oracle.raster_bwd(n, V, W, H, pr, vals, ranges, g_img, tile_sel=sel, threads=threads)
    t["raster_bwd"] = time.perf_counter() - t0
    if every != 1:
        g2 = {k: np.ascontiguousarray(v.reshape(V, n, -1)[:, a:a + m].reshape(V * m, -1).squeeze())
              for k, v in g2.items()}
    t0 = time.perf_counter()
    grad, _ = oracle.project_bwd(sub, cams, g2, threads=threads)
    t["project_bwd"] = time.perf_counter() - t0
    mm, vv = np.zeros_like(sub), np.zeros_like(sub)
    t0 = time.perf_counter()
    oracle.adam(sub, grad, mm, vv, 1, cfg["lr"], threads=threads)
    t["adam"] = time.perf_counter() - t0
    full = ((t["project"] + t["bin"] + t["project_bwd"] + t["adam"]) * lin +
            (t["raster_fwd"] + t["raster_bwd"]) * tile_scale + t["loss"])
    if every == 1:
        text = "full oracle step (all stages over the whole workload); %d threads" % threads
    else:
        text = ("sampled oracle step: projection, binning, projection backward and Adam on "
                "%d of %d Gaussians (x%.0f), compositing fwd+bwd on every %dth of %d non-empty "
                "tiles in list-length order (%d tiles, x%.2f), L1 loss on the full batch; "
                "%d threads" % (m, n, lin, every, nonempty.size, sel.size, tile_scale, threads))
    return full, sum(t.values()), t, text


# full oracle steps on all cores for the workloads whose step fits in about
# half a minute on the host (3M Gaussians x 4 views takes ~15-30 s)
FULL_ORACLE_STEP = {"tiny_2k_256", "small_200k_1024x768", "ring_3m_4x1080p"}


def cpu_baseline(cfg, workload):
    """The oracle timed on the host's cores: the whole step on all cores
    where it fits (value), and the sampled step on all cores and on one
    thread (extra keys).  Too large workloads (the oracle's lists of 20M x 4K
    need ~80 GB of host memory) are not timed."""
    if workload not in FULL_ORACLE_STEP:
        return None
    cores = host_cores()
    cache = {}
    full, wall, stages, text = oracle_step(cfg, cores, 1, cache)
    out = {"value": 1.0 / full, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": text,
           "step_s": round(full, 3), "stages_s": {k: round(v, 3) for k, v in stages.items()}}
    if workload == WORKLOAD:
        s_full, s_wall, _, s_text = oracle_step(cfg, cores, SAMPLE_EVERY, cache)
        o_full, o_wall, _, o_text = oracle_step(cfg, 1, SAMPLE_EVERY, cache)
        out["sampled_all_cores"] = {"value": 1.0 / s_full, "step_s": round(s_full, 3),
                                    "wall_s": round(s_wall, 2), "sample": s_text}
        out["one_thread"] = {"value": 1.0 / o_full, "step_s": round(o_full, 3),
                             "wall_s": round(o_wall, 2), "sample": o_text}
    return out


def reference_arm(args, rank, world):
    if rank != 0:
        return
    import scenes
    cfg = scenes.make(args.workload, n_override=args.gaussians)
    cores = host_cores()
    cache = {}
    every = 1 if args.workload in ("tiny_2k_256", "small_200k_1024x768") else SAMPLE_EVERY
    fulls = []
    text = ""
    for i in range(args.warmup + args.steps):
        full, _, _, text = oracle_step(cfg, cores, every, cache, offset=i)
        if i >= args.warmup:
            fulls.append(full)
    sec = sum(fulls) / len(fulls)
    value = 1.0 / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": text, "value": value,
                             "unit": UNIT},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------


def our_arm(args, rank, world, local):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    import scenes

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = scenes.make(args.workload, n_override=args.gaussians)
    cams = cfg["cams"]
    V = len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    n = cfg["params"].shape[1]
    params0 = torch.tensor(cfg["params"], device=dev)
    target_host = torch.from_numpy(cfg["target"]).pin_memory()
    target = target_host.to(dev)
    fused = not args.separate
    step = gs.TrainStep(params0.clone(), cams, target, lr=cfg["lr"], sparse=cfg["sparse_adam"],
                        fused=fused)
    stream = torch.cuda.current_stream()
    tile_passes = (gs.gs_key_bits(V, W, H) - 32 + 7) // 8
    # project; binning: compaction, capacity check, 2 digit scans, 4 depth passes, emission,
    # tile passes, ranges; tile order; (zeroing, fused | fwd, loss, zeroing, bwd); project_bwd;
    # adam.  The emission is one kernel, or two (a row scan and the balanced chunks) when rows
    # average 8 tiles or more against the buffers and one tile pass finishes the lists (with
    # more, the first tile pass makes the chunks itself)
    kernels_per_step = (15 if fused else 17) + tile_passes

    def emission_extra():
        return 1 if (step.capacity >= 8 * V * n and tile_passes == 1) else 0

    prune_info = None
    if args.prune is not None:
        def over_capacity(st):
            nc = st.n_contrib
            tx, ty = (W + 15) // 16, (H + 15) // 16
            pad = torch.zeros((V, ty * 16, tx * 16), dtype=torch.int32, device=dev)
            pad[:, :H, :W] = nc
            L = pad.view(V, ty, 16, tx, 16).amax(dim=(2, 4))
            return int((L > args.prune).sum().item()), int((L > 0).sum().item())
        step.step()
        torch.cuda.synchronize()
        over0, busy0 = over_capacity(step)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        pruned = step.prune_to_capacity(args.prune, args.prune_tau)
        p1.record(stream)
        torch.cuda.synchronize()
        kept = pruned[0].shape[1]
        step = gs.TrainStep(pruned[0].contiguous(), cams, target, lr=cfg["lr"],
                            sparse=cfg["sparse_adam"], fused=fused)
        step.step()
        torch.cuda.synchronize()
        over1, busy1 = over_capacity(step)
        prune_info = {"capacity": args.prune, "tau": args.prune_tau, "ms": round(p0.elapsed_time(p1), 3),
                      "gaussians_before": n, "gaussians_after": kept,
                      "tiles_over_capacity_before": over0, "tiles_over_capacity_after": over1,
                      "nonempty_tiles": busy0}
        del pruned
        n = kept

    reorder_ms = None
    if args.morton:
        step.reorder_morton()  # first call: workspace sizing, module load
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        step.reorder_morton()
        r1.record(stream)
        torch.cuda.synchronize()
        reorder_ms = r0.elapsed_time(r1)

    # warm-up (sizes the intersection buffers)
    for _ in range(max(args.warmup, 3)):
        step.step()
    torch.cuda.synchronize()

    # work counts of this step (instrumented forward, outside the timed region)
    counts = torch.zeros(2, dtype=torch.int64, device=dev)
    step.project()
    step.bin_and_sort()
    step.rasterize_fwd(counts=counts)
    torch.cuda.synchronize()
    tested, included = [int(x) for x in counts.cpu()]
    bwd_eval = int(step.n_contrib.to(torch.int64).sum().item())
    visible_rows = int((step.tile_counts > 0).sum().item())
    I = step.n_isect

    if fused:
        # the step's order; the replayed step runs the zeroing on a second
        # stream while the lists are built
        names = ["project", "zero_grads", "bin_and_sort", "rasterize_fused", "project_bwd", "adam"]
        calls = [step.project, step.zero_grads, step.bin_and_sort,
                 lambda: step.rasterize_fused(accumulate=True), step.project_bwd, step.adam]
    else:
        names = ["project", "bin_and_sort", "rasterize_fwd", "loss_l1", "rasterize_bwd",
                 "project_bwd", "adam"]
        calls = [step.project, step.bin_and_sort, step.rasterize_fwd, step.loss_l1,
                 step.rasterize_bwd, step.project_bwd, step.adam]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
          for _ in range(args.steps)]

    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    barrier(world)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        for i, fn in enumerate(calls):
            fn()
            ev[k][i + 1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms, value = aggregate(args.steps, t_start.elapsed_time(t_end), world)
    per_kernel = {nm: sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)) / args.steps
                  for i, nm in enumerate(names)}
    eager_ms_step = total_ms / args.steps
    graph = not args.no_graph
    if graph:
        # the whole step captured once and replayed: one launch per step
        step.capture()
        for _ in range(3):
            step.step()
        torch.cuda.synchronize()
        barrier(world)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            step.step()
        g1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        if step.check() != gs.GS_OK:
            raise RuntimeError("a replayed step outgrew the intersection buffers")
        total_ms, value = aggregate(args.steps, g0.elapsed_time(g1), world)
        kernels_per_step += 1  # the device step counter
    kernels_per_step += emission_extra()
    clock_info = clocks.stop()
    ms_step = total_ms / args.steps

    # end to end through the public API: pinned host target in, loss out.  Each
    # step's images are copied from pinned host memory on a copy stream into
    # one of two staging buffers while the previous step runs (as a loader
    # would prefetch); the step waits for its buffer and moves it into place.
    copy_stream = torch.cuda.Stream(device=dev)
    stage = [torch.empty_like(step.target) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def prefetch(k):
        with torch.cuda.stream(copy_stream):
            if k >= 2:
                copy_stream.wait_event(freed[k % 2])
            stage[k % 2].copy_(target_host, non_blocking=True)
            copied[k % 2].record(copy_stream)

    torch.cuda.synchronize()
    barrier(world)
    w0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # each step's loss goes to pinned host memory behind an event and is read
    # after the next step has been launched, so the GPU never waits for the host
    loss_host = torch.empty((2, 1), dtype=torch.float32).pin_memory()
    loss_ready = [torch.cuda.Event() for _ in range(2)]
    e0.record(stream)
    copy_stream.wait_event(e0)
    losses = []
    prefetch(0)
    for k in range(args.steps):
        if k + 1 < args.steps:
            prefetch(k + 1)
        stream.wait_event(copied[k % 2])
        step.target.copy_(stage[k % 2], non_blocking=True)
        freed[k % 2].record(stream)
        step.step()
        loss_host[k % 2].copy_(step.loss.reshape(1), non_blocking=True)
        loss_ready[k % 2].record(stream)
        if k >= 1:
            loss_ready[(k - 1) % 2].synchronize()
            losses.append(float(loss_host[(k - 1) % 2, 0]))
    loss_ready[(args.steps - 1) % 2].synchronize()
    losses.append(float(loss_host[(args.steps - 1) % 2, 0]))
    e1.record(stream)
    torch.cuda.synchronize()
    if graph and step.check() != gs.GS_OK:
        raise RuntimeError("a replayed step outgrew the intersection buffers")
    e2e_ms, e2e_value = aggregate(args.steps, e0.elapsed_time(e1), world)
    e2e_wall = time.perf_counter() - w0

    # roofline accounting
    hbm_peak, sm_max, peak_kind = peaks()
    sm_mhz = clock_info["sm_mhz"] if clock_info else sm_max
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    fp32_peak_tflops = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    fwd_flops = FWD_FLOP_PAIR * tested
    bwd_flops = BWD_FLOP_PAIR * bwd_eval
    useful = {"rasterize_fwd": FWD_FLOP_TESTED * tested + FWD_FLOP_INCLUDED * included,
              "rasterize_bwd": BWD_FLOP_EVAL * bwd_eval + BWD_FLOP_INCLUDED * included}
    useful["rasterize_fused"] = useful["rasterize_fwd"] + useful["rasterize_bwd"]
    rows = V * n
    adam_cols = int(step.visible.sum().item()) if cfg["sparse_adam"] else n
    kern = {
        "rasterize_fwd": ("alu", fwd_flops / 1e12, "TFLOP/s", fp32_peak_tflops),
        "rasterize_bwd": ("alu", bwd_flops / 1e12, "TFLOP/s", fp32_peak_tflops),
        "project": ("hbm", (PROJ_READ * n + SPLAT_BYTES * visible_rows +
                            CULLED_BYTES * (rows - visible_rows)) / 1e9, "GB/s", hbm_peak),
        "bin_and_sort": ("hbm", (BIN_ROW * rows + BIN_VISIBLE * visible_rows +
                                 (BIN_ISECT + 16 * tile_passes) * I) / 1e9, "GB/s", hbm_peak),
        "loss_l1": ("hbm", LOSS_BYTES * V * W * H / 1e9, "GB/s", hbm_peak),
        "project_bwd": ("hbm", (PROJ_BWD_BYTES * n + PROJ_BWD_ROW * visible_rows +
                                PROJ_BWD_COUNT * rows) / 1e9, "GB/s", hbm_peak),
        "adam": ("hbm", ADAM_BYTES * adam_cols / 1e9, "GB/s", hbm_peak),
    }
    if fused:
        # one kernel does the forward, the loss and the backward
        kern["rasterize_fused"] = ("alu", (fwd_flops + bwd_flops) / 1e12, "TFLOP/s",
                                   fp32_peak_tflops)
        kern["zero_grads"] = ("hbm", (ZERO_ROW * rows + ZERO_VISIBLE * visible_rows) / 1e9,
                              "GB/s", hbm_peak)
        for nm in ("rasterize_fwd", "rasterize_bwd", "loss_l1"):
            del kern[nm]
    # the recorded DRAM bytes describe the default run of the workload only
    variant = bool(args.gaussians or args.prune is not None or args.morton)
    kernels = {}
    for nm, (bound, work, unit, peak) in kern.items():
        ach = work / (per_kernel[nm] / 1e3)
        kernels[nm] = {"ms": round(per_kernel[nm], 4), "bound": bound, "achieved": round(ach, 3),
                       "peak": round(peak, 2), "unit": unit, "frac": round(ach / peak, 4),
                       "traffic": traffic_of(nm, args.workload, variant)}
        if nm in useful:
            u = useful[nm] / 1e12 / (per_kernel[nm] / 1e3)
            kernels[nm]["achieved_useful"] = round(u, 3)
            kernels[nm]["frac_useful"] = round(u / peak, 4)
    dom = max(kern, key=lambda k: per_kernel[k])
    d = kernels[dom]
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"],
                "traffic": traffic_of(dom, args.workload, variant),
                "peak_source": (peak_kind + " HBM copy") if d["bound"] == "hbm" else
                ("FP32 lanes x 2 x median SM clock %.0f MHz, %d SMs" % (sm_mhz, sms))}
    if "frac_useful" in d:
        roofline["frac_useful"] = d["frac_useful"]
        roofline["work"] = ("%d flop per tested pair + %d per backward pair (frac); useful: "
                            "%d per tested + %d per composited pair forward, %d per evaluated + "
                            "%d per contributing pair backward (frac_useful)" %
                            (FWD_FLOP_PAIR, BWD_FLOP_PAIR, FWD_FLOP_TESTED, FWD_FLOP_INCLUDED,
                             BWD_FLOP_EVAL, BWD_FLOP_INCLUDED))
    raster_ms = (per_kernel["rasterize_fused"] if fused else
                 per_kernel["rasterize_fwd"] + per_kernel["loss_l1"] + per_kernel["rasterize_bwd"])
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "gaussians": n, "views": V, "width": W,
                       "height": H, "intersections": I, "l2": "inputs larger than L2 "
                       "(708 MB parameters, 2.1 GB with Adam state)", "adam": "sparse" if
                       cfg["sparse_adam"] else "dense", "compositing": "fused" if fused else
                       "separate", "gaussian_order": "morton" if args.morton else "as generated",
                       "pruned_to_capacity": args.prune,
                       "launch": "CUDA graph replay" if graph else "eager calls"},
            "mpix_per_s": round(V * W * H / (raster_ms / 1e3) / 1e6, 2),
            "gaussians_per_s": round(n * V / (ms_step / 1e3), 1),
            "gpu_launches": kernels_per_step * args.steps,
            "e2e": {"value": round(e2e_value, 4), "unit": UNIT,
                    "h2d_bytes_per_step": int(target_host.numel() * 4), "d2h_bytes_per_step": 4,
                    "wall_s": round(e2e_wall, 3)},
            "roofline": roofline, "kernels": kernels,
            "morton_reorder_ms": None if reorder_ms is None else round(reorder_ms, 3),
            "eager_ms_per_step": round(eager_ms_step, 4),
            "prune": prune_info,
            "work": {"pairs_tested_fwd": tested, "pairs_included": included,
                     "pairs_bwd": bwd_eval, "visible_rows": visible_rows,
                     "adam_columns": adam_cols},
            "loss_first_last": [round(losses[0], 6), round(losses[-1], 6)],
            "clocks": clock_info}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not variant:
        cb = cpu_baseline(cfg, args.workload)
        if cb is not None:
            line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        our_arm(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

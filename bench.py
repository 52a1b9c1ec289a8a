#!/usr/bin/env python3
"""Benchmark: cone-beam forward projection + matched backprojection (Siddon) on one B300.

Workload: 256^3 float32 ellipsoid phantom, 360-view circular cone orbit (sid 500, sdd 1000),
384 x 384 detector at 1.2, voxel spacing 1.0.  One step = one ct_project + one ct_backproject
(the whole hot path; geometry staging happens once, before timing).

Metric: ray-voxel updates per second of the pair, 2 U / (t_FP + t_BP), where U is the number of
ray-voxel segments one pass walks (counted on the host in float64 from the geometry).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 it is launched under torchrun, one rank per GPU; each rank runs an independent replica
of the workload (the path needs no exchange for replicas) and rank 0 prints one JSON line.
`--impl reference` times the float64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fan_beam_projector_siddon_b300 import workloads as W  # noqa: E402

METRIC = "cone FP+BP ray-voxel updates/s at 256^3x360 views"
UNIT = "updates/s"
CONFIG_ID = 3


# ----------------------------------------------------------------------------------------------
# units of work
# ----------------------------------------------------------------------------------------------

def _count_view(w: W.Workload, k: int) -> int:
    """Ray-voxel segments of view k (see count_updates)."""
    nz, ny, nx = w.vol_shape
    s = w.voxel_spacing
    dims = 2 if w.is_2d else 3
    ncell = np.array([nx, ny, nz], dtype=np.float64)[:dims]
    half = 0.5 * ncell * s
    uu = (np.arange(w.n_u) - (w.n_u - 1) / 2.0) * w.du
    vv = (np.arange(w.n_v) - (w.n_v - 1) / 2.0) * w.dv if not w.is_2d else np.zeros(1)
    parallel = w.beam in (W.PARALLEL2D, W.PARALLEL3D)
    r = w.views[k]
    if w.is_2d:
        first, ctr, du = r[0:2], r[2:4], r[4:6]
        dv = np.zeros(2)
    else:
        first, ctr, du, dv = r[0:3], r[3:6], r[6:9], r[9:12]
    pix = ctr + uu[:, None, None] * du + vv[None, :, None] * dv      # (U, V, dims)
    if parallel:
        e = pix
        d = np.broadcast_to(first, pix.shape)
        amin = np.full(pix.shape[:2], -np.inf)
        amax = np.full(pix.shape[:2], np.inf)
    else:
        e = np.broadcast_to(first, pix.shape)
        d = pix - first
        amin = np.zeros(pix.shape[:2])
        amax = np.ones(pix.shape[:2])
    ok = np.ones(pix.shape[:2], dtype=bool)
    with np.errstate(divide="ignore", invalid="ignore"):
        for a in range(dims):
            da, ea = d[..., a], e[..., a]
            nzd = da != 0
            t1 = np.where(nzd, (-half[a] - ea) / np.where(nzd, da, 1), -np.inf)
            t2 = np.where(nzd, (half[a] - ea) / np.where(nzd, da, 1), np.inf)
            amin = np.maximum(amin, np.minimum(t1, t2))
            amax = np.minimum(amax, np.maximum(t1, t2))
            ok &= nzd | ((ea >= -half[a]) & (ea < half[a]))
    hit = ok & (amax > amin)
    segs = np.where(hit, 1, 0).astype(np.int64)
    for a in range(dims):
        ci = (e[..., a] + np.where(hit, amin, 0) * d[..., a] + half[a]) / s
        co = (e[..., a] + np.where(hit, amax, 0) * d[..., a] + half[a]) / s
        lo, hi = np.minimum(ci, co), np.maximum(ci, co)
        first_plane = np.maximum(np.floor(lo) + 1, 1)
        last_plane = np.minimum(np.ceil(hi) - 1, ncell[a] - 1)
        segs += np.where(hit, np.maximum(0, last_plane - first_plane + 1), 0).astype(np.int64)
    return int(segs.sum())


def count_updates(w: W.Workload, views=None, threads: int | None = None) -> int:
    """Ray-voxel segments walked by one pass: per ray that meets the box, 1 + the number of
    interior cell planes it crosses (float64, vectorised per view, views on a thread pool).
    Independent of both the CUDA path and the oracle."""
    import concurrent.futures as cf
    view_ids = list(range(w.n_views) if views is None else views)
    threads = threads or min(16, os.cpu_count() or 1)
    if threads <= 1 or len(view_ids) < 4:
        return sum(_count_view(w, k) for k in view_ids)
    with cf.ThreadPoolExecutor(threads) as ex:
        return sum(ex.map(lambda k: _count_view(w, k), view_ids))


# ----------------------------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ----------------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------------------------

def oracle_sample_rate(w: W.Workload, x: np.ndarray, n_views: int, threads: int):
    """Oracle FP+BP over n_views evenly spaced views; returns (updates/s, seconds, updates)."""
    import oracle
    ids = np.linspace(0, w.n_views, n_views, endpoint=False).astype(int)
    sub = w.subset(ids)
    go = oracle.Geometry.from_workload(sub)
    u = count_updates(sub)
    y = W.random_sinogram(sub, 7)
    t0 = time.perf_counter()
    go.project(x, threads=threads)
    go.backproject(y, threads=threads)
    dt = time.perf_counter() - t0
    return 2 * u / dt, dt, 2 * u


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = W.config(CONFIG_ID)
    x = w.phantom()
    cores = os.cpu_count() or 1
    n_views = sample_views(w, args.sample_views)
    rates, times = [], []
    for _ in range(args.warmup):
        oracle_sample_rate(w, x, max(1, n_views // 4), cores)
    for _ in range(args.steps):
        r, dt, _ = oracle_sample_rate(w, x, n_views, cores)
        rates.append(r)
        times.append(dt)
    value = statistics.median(rates)
    sample = (f"FP+BP of {n_views} evenly spaced views of {w.n_views} per step "
              f"(float64 oracle, thread pool over views)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "volume": list(w.vol_shape), "views": w.n_views,
                   "detector": [w.n_u, w.n_v], "sample_views": n_views},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

def max_over_ranks(value: float, world: int) -> float:
    """Largest `value` over all ranks of the default process group (NCCL or gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sample_views(w: W.Workload, requested: int | None) -> int:
    """Views per oracle step: one per host core (bounded), so a step is seconds of CPU work."""
    cores = os.cpu_count() or 1
    n = requested if requested else cores
    return int(max(1, min(w.n_views, n)))


def profiled_traffic(kernel: str, source: str = "siddon_kernels.cu"):
    """DRAM bytes per launch of `kernel` from its committed ncu summary, or None when the kernel
    source changed since that capture (the summary records the source's sha256 prefix)."""
    import hashlib
    import glob
    src = os.path.join(ROOT, "fan_beam_projector_siddon_b300", "csrc", source)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for path in glob.glob(os.path.join(ROOT, "profiles", f"{kernel}_cone256_360v.md")):
        text = open(path).read()
        m_sha = re.search(r"sha256 \(first 16 hex digits of `csrc/" + re.escape(source) +
                          r"`\): ([0-9a-f]{16})", text)
        m_tr = re.search(r"traffic_bytes_per_launch: (\d+)", text)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return int(m_tr.group(1)), os.path.relpath(path, ROOT)
    return None, None


def profiled_sol(kernel: str, source: str = "siddon_kernels.cu"):
    """ncu speed-of-light figures of `kernel` from its committed summary (percent of ncu's own
    peaks: memory SOL = max over L1/L2/DRAM, L2 and DRAM throughput), or None when the kernel
    source changed since the capture."""
    traffic, path = profiled_traffic(kernel, source)
    if path is None:
        return None
    text = open(os.path.join(ROOT, path)).read()
    out = {"source": path}
    for key, label in (("memory_sol_pct", "memory throughput (ncu SOL"),
                       ("l1tex_pct", "L1TEX throughput"), ("l2_pct", "L2 throughput"),
                       ("dram_pct", "DRAM throughput"), ("issue_pct", "issue slots busy")):
        m = re.search(r"\| " + re.escape(label) + r"[^|]*\| ([0-9.]+) %", text)
        out[key] = float(m.group(1)) if m else None
    m = re.search(r"\| duration \(sum over captured launches, serialised\) \| ([0-9.]+) ms", text)
    out["ms"] = float(m.group(1)) if m else None
    m = re.search(r"\| L2 sector bandwidth \| ([0-9.]+) GB/s = ([0-9.]+) % of the L2 sector peak "
                  r"\(([0-9.]+) GB/s\)", text)
    out["l2_sector_gbs"] = float(m.group(1)) if m else None
    out["l2_sector_peak_gbs"] = float(m.group(3)) if m else None
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def measured_sm_max_mhz():
    """The SM clock limit recorded beside the measured peaks, or None."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            v = json.load(f).get("sm_max_mhz")
        return float(v) if v else None
    return None


def sirt_leg(ct, torch, n_iters: int = 10):
    """SIRT on the dual-axis tilt-series workload (512^3, 280 parallel3d views, 512x512 detector),
    the configuration the pages quote SIRT timings on: n_iters iterations from zero, timed with
    CUDA events; the one-off C = 1/(A^T 1) initialisation is timed separately."""
    w = W.config(5)
    g = ct.Geometry.from_workload(w)
    x_true = torch.from_numpy(w.phantom()).cuda()
    y = g.project(x_true)
    ws = g.new_workspace(sirt=True)
    x = torch.zeros_like(x_true)
    stream = torch.cuda.current_stream()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    e0.record(stream)
    g.sirt(x, y, 0, ws, initialised=False)
    e1.record(stream)
    g.sirt(x, y, n_iters, ws, initialised=True)
    e2.record(stream)
    torch.cuda.synchronize()
    init_ms, run_ms = e0.elapsed_time(e1), e1.elapsed_time(e2)
    U5 = count_updates(w)
    rel = float((x - x_true).norm() / x_true.norm())
    sirt = {"workload": w.name, "iterations": n_iters, "ms_per_iteration": run_ms / n_iters,
            "init_ms": init_ms, "updates_per_pass": U5,
            "updates_per_s": 2 * U5 * n_iters / (run_ms * 1e-3),
            "rel_error_vs_phantom": rel,
            "note": "iteration = residual projection + backprojection + update; "
                    "the pages' RTX 8000 figure for this workload is ~2.2 s per iteration"}
    del ws
    wc = g.new_workspace(cgls=True)
    x.zero_()
    torch.cuda.synchronize()
    e0.record(stream)
    g.cgls(x, y, 0, wc, initialised=False)
    e1.record(stream)
    g.cgls(x, y, n_iters, wc, initialised=True)
    e2.record(stream)
    torch.cuda.synchronize()
    cgls = {"workload": w.name, "iterations": n_iters,
            "ms_per_iteration": e1.elapsed_time(e2) / n_iters, "init_ms": e0.elapsed_time(e1),
            "rel_error_vs_phantom": float((x - x_true).norm() / x_true.norm()),
            "note": "iteration = projection (+|q|^2) + fused residual backprojection + |s|^2 "
                    "+ update, scalars on the device"}
    del wc, x, y, x_true
    torch.cuda.empty_cache()
    return sirt, cgls


def batch_leg(ct, torch, w, U, nb: int = 4, reps: int = 3):
    """The metric workload with nb volumes at once (leading batch dimension): one walk per ray
    serves all nb volumes.  Updates counted as nb x U per direction."""
    g = ct.Geometry.from_workload(w)
    vols = torch.rand((nb,) + tuple(w.volume_shape), device="cuda")
    sinos = torch.empty((nb,) + tuple(w.sino_shape), device="cuda")
    backs = torch.empty_like(vols)
    need = ct.ct_batch_workspace_bytes(g.handle, nb)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fps, bps = [], []
    for k in range(reps + 1):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        g.project(vols, out=sinos, workspace=ws)
        e[1].record(stream)
        g.backproject(sinos, out=backs, workspace=ws)
        e[2].record(stream)
        torch.cuda.synchronize()
        if k:
            fps.append(e[0].elapsed_time(e[1]))
            bps.append(e[1].elapsed_time(e[2]))
    fp, bp = statistics.median(fps), statistics.median(bps)
    del vols, sinos, backs, ws, flush
    torch.cuda.empty_cache()
    return {"batch": nb, "fp_ms": fp, "bp_ms": bp,
            "fp_updates_per_s": nb * U / (fp * 1e-3), "bp_updates_per_s": nb * U / (bp * 1e-3),
            "pair_updates_per_s": 2 * nb * U / ((fp + bp) * 1e-3)}


FDK_FLOPS_PER_VOXEL_VIEW = 38   # projection 23, distance weight 2, bilinear 11, accumulate 2
FDK_L1_BYTES_PER_VOXEL_VIEW = 16  # the four bilinear taps of the filtered sinogram (L1-served)
FP32_LANES_PER_SM = 128


# The cone workload's walk kernels (its detector columns share their outer-axis lines, and the
# 256^3 volume fits in L2, so the forward projection reads one crossing list per line).
FP_KERNEL, BP_KERNEL = "line_project_kernel", "backproject_kernel"


def ncu_sol():
    """Figures COPIED from the committed ncu summaries under profiles/ (hand-kept notes of
    earlier captures of the same kernel source; not measured in this run): per walk kernel the
    ncu memory SOL, L1TEX, L2 and DRAM throughput percentages, and the pair's L2-only and
    memory-SOL fractions weighted by the captured durations.  None when a summary is missing or
    its recorded source hash differs from the current kernel source."""
    fp, bp = profiled_sol(FP_KERNEL), profiled_sol(BP_KERNEL)
    if not fp or not bp or None in (fp["ms"], bp["ms"], fp["memory_sol_pct"],
                                    bp["memory_sol_pct"], fp["l2_pct"], bp["l2_pct"]):
        return None
    tot = fp["ms"] + bp["ms"]
    return {"source": "copied from committed profiles/*.md (not measured in this run)",
            FP_KERNEL: fp, BP_KERNEL: bp,
            "pair_l2_throughput_pct": (fp["l2_pct"] * fp["ms"] + bp["l2_pct"] * bp["ms"]) / tot,
            "pair_memory_sol_pct":
                (fp["memory_sol_pct"] * fp["ms"] + bp["memory_sol_pct"] * bp["ms"]) / tot,
            "note": "percent of ncu's own peaks; memory SOL is the max over L1TEX/L2/DRAM, "
                    "the L2-only figure is lts__throughput"}


def fdk_leg(ct, torch, w, peaks, sm_mhz, reps: int = 5, cpu_baseline: bool = True):
    """Filtered backprojection (FDK, Ram-Lak window) of the metric workload's geometry and its
    transpose, CUDA events around each C-ABI call, L2 flushed before each.  Rate in voxel-view
    updates per second.  Roofline: the gather kernel, which dominates the call, is bound by
    L1TEX throughput (its bilinear reads of the filtered sinogram hit L1), so the call's
    16 B of bilinear taps per voxel-view are set against the measured L1 read rate; the float32
    ALU fraction (38 flops per voxel-view against SMs x 128 lanes x 2 flops x the SM clock
    sampled in this run) is reported beside it."""
    g = ct.Geometry.from_workload(w)
    sino = torch.from_numpy(W.random_sinogram(w, 11)).cuda()
    vol = torch.empty(g.volume_shape, device="cuda")
    ws = torch.empty(ct.ct_fbp_workspace_bytes(g.handle), dtype=torch.uint8, device="cuda")
    ws_t = torch.empty(ct.ct_fbp_transpose_workspace_bytes(g.handle), dtype=torch.uint8,
                       device="cuda")
    out_t = torch.empty_like(sino)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fw, tr = [], []
    for k in range(reps + 2):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.zero_()
        e[0].record(stream)
        g.fbp(sino, out=vol, workspace=ws)
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        g.fbp_transpose(vol, out=out_t, workspace=ws_t)
        e[3].record(stream)
        torch.cuda.synchronize()
        if k >= 2:
            fw.append(e[0].elapsed_time(e[1]))
            tr.append(e[2].elapsed_time(e[3]))
    fms, tms = statistics.median(fw), statistics.median(tr)
    vv = w.n_voxels * w.n_views
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    alu_peak = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12 if sm_mhz else float("nan")
    alu = FDK_FLOPS_PER_VOXEL_VIEW * vv / (fms * 1e-3) / 1e12
    l1 = FDK_L1_BYTES_PER_VOXEL_VIEW * vv / (fms * 1e-3) / 1e9
    out = {"workload": w.name, "window": "ram-lak", "fdk_ms": fms, "transpose_ms": tms,
           "voxel_views": vv, "voxel_views_per_s": vv / (fms * 1e-3),
           "transpose_voxel_views_per_s": vv / (tms * 1e-3),
           "roofline": {"bound": "l1", "kernel": "ct_fbp (the gather dominates it)",
                        "achieved": l1, "peak": peaks["l1_read_gbs"], "unit": "GB/s",
                        "frac": l1 / peaks["l1_read_gbs"],
                        "peak_source": "measured in this run: L1-hitting 16-B read probe",
                        "bytes_model": "16 B of bilinear taps per voxel-view",
                        "alu": {"achieved_tflops": alu, "peak_tflops": alu_peak,
                                "frac": alu / alu_peak,
                                "peak_source": f"{sms} SMs x 128 fp32 lanes x 2 x {sm_mhz} MHz "
                                               "(median SM clock sampled in this run)",
                                "flops_model": "38 flops per voxel-view"}}}
    traffic, src = profiled_traffic("fdk_gather_kernel", "fbp_kernels.cu")
    out["roofline"]["traffic"] = traffic
    out["roofline"]["traffic_source"] = src
    out["roofline"]["ncu_from_committed_profiles"] = profiled_sol("fdk_gather_kernel",
                                                                  "fbp_kernels.cu")
    del sino, vol, ws, ws_t, out_t, flush
    torch.cuda.empty_cache()
    if cpu_baseline:
        from oracle import fbp as F
        n_views, n_vox = 16, 4096
        idx_views = np.linspace(0, w.n_views - 1, n_views).round().astype(int)
        rng = np.random.default_rng(12)
        vox = np.stack([rng.integers(0, s, n_vox) for s in w.vol_shape], axis=1)
        sino_h = W.random_sinogram(w, 11)[idx_views].astype(np.float64)
        t0 = time.perf_counter()
        F.fbp(w.beam, w.views[idx_views], w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
              sino_h, voxels=vox)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": n_views * n_vox / dt, "unit": "voxel-views/s",
                               "cores": 1, "kind": "oracle",
                               "sample": f"{n_vox} voxels x {n_views} views (filtering of the "
                                         f"{n_views} views included), {dt:.1f} s"}
    return out


def context_leg(ct, torch):
    """The pages' performance-table workload shape (512^3 volume, circular cone, 360 views,
    1024x768 detector at pitch 1.25; sid/sdd are not printed and are read as 1000/1500): one
    forward projection, one backprojection, one CGLS iteration, CUDA events."""
    views = W.circular_cone(360, 1000.0, 1500.0)
    w = W.Workload("cone-512^3-360v-1024x768", W.CONE, views, (512, 512, 512), 1.0, 1024, 768,
                   1.25, 1.25, 0, None)
    g = ct.Geometry.from_workload(w)
    x = torch.rand(w.volume_shape, device="cuda")
    sino = torch.empty(w.sino_shape, device="cuda")
    back = torch.empty(w.volume_shape, device="cuda")
    ws = g.new_workspace()
    stream = torch.cuda.current_stream()

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    fp = timed(lambda: g.project(x, out=sino, workspace=ws))
    bp = timed(lambda: g.backproject(sino, out=back, workspace=ws))
    del ws
    wc = g.new_workspace(cgls=True)
    xc = torch.zeros_like(x)
    g.cgls(xc, sino, 0, wc, initialised=False)
    it = timed(lambda: g.cgls(xc, sino, 1, wc, initialised=True))
    del wc, xc, x, sino, back
    torch.cuda.empty_cache()
    return {"workload": w.name, "fp_ms": fp, "bp_ms": bp, "cgls_iteration_ms": it,
            "pages_a100_ms": {"fp": 566.79, "bp": 1060.77, "cgls_iteration": 1753.73},
            "note": "context only: the pages' figures are diffct on one A100 with unstated "
                    "sid/sdd; not the same measurement"}


L2_PROBE_BYTES = 64 << 20   # fits the 126 MB L2 (about the cone workload's volume)


def l2_peaks(ct, torch, reps: int = 5):
    """Measured on-chip rates on this GPU with the library's probe kernels (CUDA events on the
    launching stream, best of `reps` after a warm-up; the 64 MiB buffer stays in L2):
    16-byte L1-bypassing reads, 16-byte L1-hitting reads (every block re-reading 16 KB), and
    red.global.add.f32 with 8 and 4 updates per 32-byte sector (warp lanes 1 and 2 floats
    apart)."""
    n = L2_PROBE_BYTES // 4
    buf = torch.zeros(n, dtype=torch.float32, device="cuda")
    sink = torch.zeros(1, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def best(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e-3)
        return min(ts)

    passes_r = 40
    t = best(lambda: ct.ct_probe_l2_read(buf.data_ptr(), n, passes_r, sink.data_ptr(), sp))
    read_gbs = 16 * (n // 4) * passes_r / t / 1e9
    out = {"read_gbs": read_gbs, "buffer_bytes": L2_PROBE_BYTES,
           "how": "ct_probe_l2_read / ct_probe_l2_reduce on a 64 MiB L2-resident buffer, CUDA "
                  "events, best of %d" % reps}
    n1, passes_1 = 4096, 4000         # 16 KB per block, re-read: L1 hits after the first pass
    t = best(lambda: ct.ct_probe_l1_read(buf.data_ptr(), n1, passes_1, sink.data_ptr(), sp))
    blocks = 4 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out["l1_read_gbs"] = blocks * 16 * (n1 // 4) * passes_1 / t / 1e9
    passes_a = 8
    for stride in (1, 2):
        t = best(lambda: ct.ct_probe_l2_reduce(buf.data_ptr(), n, passes_a, stride, sp))
        upd = 32 * (n // (32 * stride)) * passes_a / t
        out[f"red_stride{stride}_updates_per_s"] = upd
        out[f"red_stride{stride}_gbs"] = 4 * upd / 1e9
    del buf, sink
    torch.cuda.empty_cache()
    return out


def walk_roofline(U, fp_ms, bp_ms, peaks):
    """Each walk's algorithmic L2 fraction: 4 B per ray-voxel update over its CUDA-event time,
    against the measured L2 rate of its access pattern (gathers: the read probe; reductions: the
    red.global.add.f32 probe with full sectors)."""
    fp_gbs = 4.0 * U / (fp_ms * 1e-3) / 1e9
    bp_gbs = 4.0 * U / (bp_ms * 1e-3) / 1e9
    return {"fp": {"achieved_gbs": fp_gbs, "peak_gbs": peaks["read_gbs"],
                   "frac": fp_gbs / peaks["read_gbs"]},
            "bp": {"achieved_gbs": bp_gbs, "peak_gbs": peaks["red_stride1_gbs"],
                   "frac": bp_gbs / peaks["red_stride1_gbs"],
                   "frac_vs_4_per_sector": bp_gbs / peaks["red_stride2_gbs"]}}


def workload_leg(ct, torch, n: int, peaks, cpu_baseline: bool, reps: int = 3,
                 views: int | None = None):
    """FP and BP of workload n through the C ABI (CUDA events on the launching stream, L2 flushed
    before each call, median of `reps` after one warm-up), views/s, ray-voxel updates/s, the
    algorithmic L2 fractions, and the float64 oracle on the host cores over evenly spaced views
    (the whole workload when it has at most 16 views' worth of work, else extrapolated).
    `views` restricts the workload to that many evenly spaced views (for profiling captures)."""
    w = W.config(n)
    if views:
        w = w.subset(np.linspace(0, w.n_views, views, endpoint=False).astype(int))
    x_host = w.phantom()
    U = count_updates(w)
    g = ct.Geometry.from_workload(w)
    vol = torch.from_numpy(x_host).cuda()
    meas = torch.from_numpy(W.random_sinogram(w, 3)).cuda()
    sino = torch.empty(w.sino_shape, dtype=torch.float32, device="cuda")
    back = torch.empty(w.volume_shape, dtype=torch.float32, device="cuda")
    ws = g.new_workspace()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fps, bps = [], []
    for k in range(reps + 1):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.zero_()
        e[0].record(stream)
        g.project(vol, out=sino, workspace=ws)
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        g.backproject(meas, out=back, workspace=ws)
        e[3].record(stream)
        torch.cuda.synchronize()
        if k:
            fps.append(e[0].elapsed_time(e[1]))
            bps.append(e[2].elapsed_time(e[3]))
    fp, bp = statistics.median(fps), statistics.median(bps)
    shared_lines = int(g.info.shared_lines)
    del vol, meas, sino, back, ws, flush
    torch.cuda.empty_cache()
    out = {"workload": w.name, "volume": list(w.vol_shape), "views": w.n_views,
           "detector": [w.n_u, w.n_v], "shared_lines": shared_lines, "updates_per_pass": U,
           "fp_ms": fp, "bp_ms": bp,
           "views_per_s": {"fp": w.n_views / (fp * 1e-3), "bp": w.n_views / (bp * 1e-3)},
           "fp_updates_per_s": U / (fp * 1e-3), "bp_updates_per_s": U / (bp * 1e-3),
           "pair_updates_per_s": 2 * U / ((fp + bp) * 1e-3),
           "l2_roofline": walk_roofline(U, fp, bp, peaks),
           "volume_bytes": 4 * w.n_voxels,
           "volume_fits_l2": 4 * w.n_voxels <= L2_PROBE_BYTES * 2}
    if cpu_baseline:
        cores = os.cpu_count() or 1
        n_views = w.n_views if 2 * U <= 4e9 else min(w.n_views, 16)
        r, dt, nu = oracle_sample_rate(w, x_host, n_views, cores)
        whole = n_views == w.n_views
        out["cpu_baseline"] = {
            "value": r, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"FP+BP of all {w.n_views} views ({nu} updates, {dt:.1f} s)" if whole else
                       f"FP+BP of {n_views} evenly spaced views of {w.n_views} ({nu} updates, "
                       f"{dt:.1f} s); whole-workload time extrapolated linearly: "
                       f"{dt * 2 * U / nu:.0f} s"),
            "extrapolated": not whole}
    return out


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from fan_beam_projector_siddon_b300 import build as ct_build
    if rank == 0 or not os.path.exists(ct_build.LIB):
        ct_build.build()
    if world > 1:
        dist.barrier()
    import fan_beam_projector_siddon_b300 as ct

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    if args.workload is not None:
        # one workload's FP/BP leg alone (profiling and spot checks); not the benchmark line
        if rank == 0:
            peaks = l2_peaks(ct, torch)
            print(json.dumps(workload_leg(ct, torch, args.workload, peaks,
                                          cpu_baseline=not args.no_cpu_baseline,
                                          reps=max(1, args.steps), views=args.views)),
                  flush=True)
        return 0
    w = W.config(CONFIG_ID)
    x_host = w.phantom()
    U = count_updates(w)
    g = ct.Geometry.from_workload(w)
    vol = torch.from_numpy(x_host).cuda()
    sino = torch.empty(w.sino_shape, dtype=torch.float32, device="cuda")
    # backprojection input: a dense "measured" sinogram (no exact zeros, so every counted
    # ray-voxel update is performed; the kernel skips rays whose value is exactly 0)
    meas_host = W.random_sinogram(w, 3)
    meas = torch.from_numpy(meas_host).cuda()
    back = torch.empty(w.volume_shape, dtype=torch.float32, device="cuda")
    ws = g.new_workspace()
    wsb = 0 if ws is None else ws.numel()
    wsp = None if ws is None else ws.data_ptr()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # > 126 MB L2

    def fp():
        ct.ct_project(g.handle, vol.data_ptr(), sino.data_ptr(), wsp, wsb, sp)

    def bp():
        ct.ct_backproject(g.handle, meas.data_ptr(), back.data_ptr(), wsp, wsb, sp)

    for _ in range(args.warmup):
        flush.zero_()
        fp()
        bp()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            fp()
            ev[k][1].record(stream)
            bp()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    fp_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bp_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = [a + b for a, b in zip(fp_ms, bp_ms)]
    mean_step = sum(step_ms) / len(step_ms)
    mean_step = max_over_ranks(mean_step, world)
    value = world * 2 * U / (mean_step * 1e-3)

    # ---- end to end through the C ABI: pinned host in, host out, copies inside the region ----
    # A user of the library would overlap the copies with compute, as a pipeline does: two sets
    # of device buffers alternate between steps, the next step's volume and measured sinogram go
    # up on one copy stream while this step's kernels run, and the results come down on another
    # (the two directions use separate copy engines).  Each copy waits only for the kernel that
    # last used its buffer.
    vol_h = torch.from_numpy(x_host).pin_memory()
    meas_h = torch.from_numpy(meas_host).pin_memory()
    sino_h = torch.empty(w.sino_shape, dtype=torch.float32).pin_memory()
    back_h = torch.empty(w.volume_shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(2, min(args.steps, 5))
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    sets = []
    for j in range(2):
        bufs = {"vol": vol if j == 0 else torch.empty_like(vol),
                "meas": meas if j == 0 else torch.empty_like(meas),
                "sino": sino if j == 0 else torch.empty_like(sino),
                "back": back if j == 0 else torch.empty_like(back),
                "done_fp": ev(), "done_bp": ev(), "sino_dl": ev(), "back_dl": ev()}
        for k in ("done_fp", "done_bp", "sino_dl", "back_dl"):
            bufs[k].record(stream)
        sets.append(bufs)

    def e2e_step(k):
        b = sets[k % 2]
        vol_up, meas_up = ev(), ev()
        with torch.cuda.stream(up_s):
            up_s.wait_event(b["done_fp"])               # this set's volume no longer read
            b["vol"].copy_(vol_h, non_blocking=True)
            vol_up.record(up_s)
            up_s.wait_event(b["done_bp"])               # this set's sinogram no longer read
            b["meas"].copy_(meas_h, non_blocking=True)
            meas_up.record(up_s)
        stream.wait_event(vol_up)
        stream.wait_event(b["sino_dl"])                 # this set's last projection downloaded
        ct.ct_project(g.handle, b["vol"].data_ptr(), b["sino"].data_ptr(), wsp, wsb, sp)
        b["done_fp"].record(stream)
        stream.wait_event(meas_up)
        stream.wait_event(b["back_dl"])
        ct.ct_backproject(g.handle, b["meas"].data_ptr(), b["back"].data_ptr(), wsp, wsb, sp)
        b["done_bp"].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(b["done_fp"])
            sino_h.copy_(b["sino"], non_blocking=True)
            b["sino_dl"].record(down_s)
            down_s.wait_event(b["done_bp"])
            back_h.copy_(b["back"], non_blocking=True)
            b["back_dl"].record(down_s)

    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    h2d = vol_h.numel() * 4 + meas_h.numel() * 4
    d2h = sino_h.numel() * 4 + back_h.numel() * 4
    del sets

    if rank != 0:
        return 0
    # ---- roofline of the dominant kernel: L2, measured on this GPU ---------------------------
    peaks = l2_peaks(ct, torch)
    hbm_peak, hbm_kind = load_peaks()
    fp_avg, bp_avg = sum(fp_ms) / len(fp_ms), sum(bp_ms) / len(bp_ms)
    walks = walk_roofline(U, fp_avg, bp_avg, peaks)
    dom = "bp" if bp_avg >= fp_avg else "fp"
    kname = BP_KERNEL if dom == "bp" else FP_KERNEL
    traffic, traffic_src = profiled_traffic(kname)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "volume": list(w.vol_shape), "views": w.n_views,
                   "detector": [w.n_u, w.n_v], "updates_per_pass": U,
                   "l2": "flushed before each step (256 MiB write outside the timed events)",
                   "parallelism": f"replicas x{world}",
                   "shared_lines": int(g.info.shared_lines)},
        "fp_ms": statistics.mean(fp_ms), "bp_ms": statistics.mean(bp_ms),
        "fp_updates_per_s": U / (fp_avg * 1e-3), "bp_updates_per_s": U / (bp_avg * 1e-3),
        "views_per_s": {"fp": w.n_views / (fp_avg * 1e-3), "bp": w.n_views / (bp_avg * 1e-3)},
        "roofline": {"bound": "l2", "kernel": "ct_backproject" if dom == "bp" else "ct_project",
                     "achieved": walks[dom]["achieved_gbs"], "peak": walks[dom]["peak_gbs"],
                     "unit": "GB/s", "frac": walks[dom]["frac"], "traffic": traffic,
                     "traffic_source": traffic_src,
                     "peak_source": "measured in this run: " + (
                         "red.global.add.f32 probe, 8 updates per 32-B sector" if dom == "bp"
                         else "L1-bypassing 16-B read probe") + " (l2_peaks)",
                     "bytes_model": "4 B per ray-voxel update (the L2-served gathers or "
                                    "reductions); traffic = DRAM bytes per launch from the "
                                    "committed ncu summary, null when its source is stale",
                     "walks": walks},
        "l2_peaks": peaks,
        "hbm_peak": {"gbs": hbm_peak, "source": hbm_kind + " (MEASURED_PEAKS.json copy)"},
        "e2e": {"value": world * 2 * U / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "timing": "host wall clock around the steps; two device buffer sets alternate, "
                          "uploads and downloads on their own streams overlap the kernels"},
        "ncu_from_committed_profiles": ncu_sol(),
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    line["batch4"] = batch_leg(ct, torch, w, U)
    if not args.no_workloads and args.workload is None:
        line["workloads"] = {f"config{n}": workload_leg(ct, torch, n, peaks,
                                                        cpu_baseline=not args.no_cpu_baseline)
                             for n in (1, 2, 4, 5)}
    if not args.no_fdk:
        line["fdk"] = fdk_leg(ct, torch, w, peaks, clocks["sm_mhz"] or clocks["sm_max_mhz"] or
                              measured_sm_max_mhz(),
                              cpu_baseline=world == 1 and not args.no_cpu_baseline)
    if not args.no_sirt:
        line["sirt"], line["cgls"] = sirt_leg(ct, torch)
    if args.context:
        line["context_pages_table"] = context_leg(ct, torch)
    if world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        n_views = sample_views(w, args.sample_views)
        r, dt, nu = oracle_sample_rate(w, x_host, n_views, cores)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"FP+BP of {n_views} evenly spaced views of "
                                          f"{w.n_views} ({nu} updates, {dt:.1f} s)"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sirt", action="store_true", help="skip the SIRT/CGLS leg")
    ap.add_argument("--no-fdk", action="store_true", help="skip the FBP/FDK leg")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the FP/BP legs of the other four workloads")
    ap.add_argument("--workload", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="time only this workload's FP/BP leg (--steps reps) and print it")
    ap.add_argument("--views", type=int, default=None,
                    help="with --workload: that many evenly spaced views of it")
    ap.add_argument("--context", action="store_true",
                    help="also time the pages' performance-table workload shape")
    ap.add_argument("--sample-views", type=int, default=None,
                    help="views per oracle step (default: one per host core)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

"""Host-side parts of the benchmark: work counting, max-over-ranks with two gloo ranks, and the
reference (oracle) arm's JSON line and rank behaviour.  No GPU."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_count_updates_matches_oracle_segments(n):
    """1 + crossings per ray equals the oracle's positive-length segment count, except where a
    ray crosses two planes at the same point (a zero-length segment the oracle merges)."""
    w = W.small_config(n)
    _, segs = oracle.Geometry.from_workload(w).ray_lengths()
    counted = bench.count_updates(w)
    assert counted >= int(segs.sum())
    assert counted - int(segs.sum()) <= 1e-3 * counted


def test_count_updates_jittered_workload_is_exact():
    """With per-view jitter no ray meets two planes at one point: the counts agree exactly."""
    w = W.small_config(4)
    _, segs = oracle.Geometry.from_workload(w).ray_lengths()
    assert bench.count_updates(w) == int(segs.sum())


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0", "--sample-views", "2"],
                          capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_json_line():
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "updates/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["metric"] == bench.METRIC
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_non_zero_rank_exits_quietly():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_profile_figures_parse_or_are_withheld():
    """Traffic and ncu speed-of-light figures come from the committed profiles only while the
    kernel source matches the capture; otherwise they are None (never stale numbers)."""
    import bench
    for kern, src in ((bench.FP_KERNEL, "siddon_kernels.cu"),
                      (bench.BP_KERNEL, "siddon_kernels.cu"),
                      ("fdk_gather_kernel", "fbp_kernels.cu")):
        traffic, path = bench.profiled_traffic(kern, src)
        sol = bench.profiled_sol(kern, src)
        if path is None:
            assert traffic is None and sol is None
            continue
        assert traffic > 0
        assert 0 < sol["memory_sol_pct"] <= 100 and 0 < sol["issue_pct"] <= 100
        assert sol["ms"] > 0
    pair = bench.ncu_sol()
    if pair is not None:
        fp, bp = pair[bench.FP_KERNEL], pair[bench.BP_KERNEL]
        lo = min(fp["memory_sol_pct"], bp["memory_sol_pct"])
        hi = max(fp["memory_sol_pct"], bp["memory_sol_pct"])
        assert lo <= pair["pair_memory_sol_pct"] <= hi


def test_l2_figures_of_the_walk_profiles():
    """The L2 sector bandwidth parsed from the committed walk summaries agrees with the row's
    own percentage of the L2 sector peak, and the pair's L2-only fraction lies between the two
    kernels' figures."""
    import re
    import bench
    pair = bench.ncu_sol()
    if pair is None:
        pytest.skip("walk summaries do not match the current kernel source")
    assert "not measured in this run" in pair["source"]
    for name in (bench.FP_KERNEL, bench.BP_KERNEL):
        d = pair[name]
        text = open(os.path.join(bench.ROOT, d["source"])).read()
        pct = float(re.search(r"= ([0-9.]+) % of the L2 sector peak", text).group(1))
        assert 0 < d["l2_sector_gbs"] < d["l2_sector_peak_gbs"]
        assert abs(100 * d["l2_sector_gbs"] / d["l2_sector_peak_gbs"] - pct) < 0.1
    lo = min(pair[bench.FP_KERNEL]["l2_pct"], pair[bench.BP_KERNEL]["l2_pct"])
    hi = max(pair[bench.FP_KERNEL]["l2_pct"], pair[bench.BP_KERNEL]["l2_pct"])
    assert lo <= pair["pair_l2_throughput_pct"] <= hi


def test_walk_roofline_fractions():
    """The algorithmic L2 fraction of a walk is 4 B per update over its time against the
    measured rate of its access pattern, and halves when the time doubles."""
    import bench
    U = 18315651008
    peaks = {"read_gbs": 20000.0, "red_stride1_gbs": 8000.0, "red_stride2_gbs": 5000.0}
    a = bench.walk_roofline(U, 16.3, 17.5, peaks)
    b = bench.walk_roofline(U, 32.6, 35.0, peaks)
    assert abs(a["fp"]["achieved_gbs"] - 4 * U / 16.3e-3 / 1e9) < 1e-6
    for k in ("fp", "bp"):
        assert 0 < a[k]["frac"] < 1
        assert abs(2 * b[k]["frac"] - a[k]["frac"]) < 1e-12
    assert a["bp"]["frac_vs_4_per_sector"] > a["bp"]["frac"]

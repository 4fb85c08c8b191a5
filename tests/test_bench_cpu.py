"""bench.py host logic on the CPU: the multi-rank timing reduction with two
gloo ranks, the weak-scaling throughput formula, and the reference arm (the
fp64 oracle timed on the host cores)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 100.0 + 25.0 * rank            # each rank timed a different region
    dist.barrier()
    slowest = bench.slowest_rank_ms(elapsed, dist, "cpu")
    out.put((rank, slowest, bench.job_tflops(world, 10, 2.0e12, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 125.0
        # 2 ranks x 10 steps x 2 TFLOP in 0.125 s
        assert abs(value - 2 * 10 * 2.0 / 0.125) < 1e-9


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(3.5, None, "cpu") == 3.5
    assert abs(bench.job_tflops(1, 4, 1e12, 1000.0) - 4.0) < 1e-12


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["full_config_s_extrapolated"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_cpu_baseline_extrapolates_from_full_length_rows():
    r = bench.oracle_sample(0.0, block=64)
    assert r["sampled_rows"] == 64 and r["full_config_rows"] == 2 * 32 * 8192
    assert abs(r["full_config_s_extrapolated"] - r["measured_sample_s"] * 2 * 32 * 8192 / 64) < 1e-9
    f, b = bench.step_flops(bench.WORKLOAD)
    assert abs(r["value"] - (f + b) / r["full_config_s_extrapolated"] / 1e12) < 1e-12


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_kernel_work_and_flop_convention():
    w = bench.WORKLOAD
    f, b = bench.step_flops(w)
    assert f == 4.0 * 2 * 32 * 8192 ** 2 * 128 * 0.5 and b == 2.5 * f
    work = bench.kernel_work(w)
    assert work["fwd"] == ("tensor", f)
    assert work["bwd_dkdv"][1] + work["bwd_dq"][1] == 2.5 * f


def test_window_pair_count_matches_brute_force():
    import numpy as np
    for n, w in [(1, 1), (10, 1), (10, 3), (10, 10), (10, 25), (300, 128), (1000, 999)]:
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        assert bench.window_pairs(n, w) == int(((i - j >= 0) & (i - j < w)).sum())
    # the benchmark's window is three quarters of the causal pairs
    assert abs(bench.window_pairs(8192, 4096) / (8192 * 8193 / 2) - 0.75) < 1e-3

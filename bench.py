#!/usr/bin/env python3
"""Exact-attention benchmark on GB300: forward + backward TFLOP/s.

One step = one forward (attn_fwd) and one backward (attn_bwd: preprocessing,
dK/dV, dQ) pass over the causal GPT-style workload B=2, H=32, N=8192, d=128
with seeded synthetic bf16 inputs resident in HBM.  FLOPs follow the
published convention: 4*B*H*N^2*d for the forward, 2.5x that for the
backward, halved under a causal mask.

Printed (rank 0): one JSON line with the headline value, per-kernel roofline of
the dominant kernel (durations from CUDA events the library records around its
own launches, on the launching stream), the chunked partial-forward + LSE-merge
rows measured in the same run, an end-to-end number through the public API
with host buffers, the fp64 CPU oracle timed on a bounded sample, and the SM
clocks sampled during the timed region.

``--impl reference`` times the fp64 CPU oracle itself (the only reference this
method has: the pages hold no runnable implementation) on a bounded sample of
the same workload.  Multi-GPU (torchrun, one rank per GPU): every rank runs its
own independent batch (weak scaling, no collective on the data path); the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s (bf16, causal-adjusted) and % of GB300 dense BF16 peak"
WORKLOAD = dict(name="gpt_causal", B=2, Hq=32, Hkv=32, N=8192, d=128, mask="causal")
CHUNKED = dict(name="chunked_gqa", B=1, Hq=32, Hkv=8, N=32768, d=128, chunks=8)
WINDOW = dict(name="gpt_sliding_window", B=2, Hq=32, Hkv=32, N=8192, d=128, window=4096)
DECODE = dict(name="decode_gqa", B=8, Hq=32, Hkv=8, Nq=1, Nk=32768, d=128)
VARLEN = dict(name="varlen_causal", B=16, Hq=32, Hkv=32, d=128, min_len=512, max_len=8192)
FP8 = dict(name="gpt_causal_fp8", B=2, Hq=32, Hkv=32, N=8192, d=128)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "fwd": ["fwd.cu", "ptx.cuh", "schedule.h", "internal.h"],
    "partial_fwd": ["fwd.cu", "ptx.cuh", "schedule.h", "internal.h"],
    "bwd_dkdv": ["bwd.cu", "ptx.cuh", "internal.h"],
    "bwd_dq": ["bwd.cu", "ptx.cuh", "internal.h"],
    "bwd_preprocess": ["merge.cu", "ptx.cuh", "internal.h"],
    "merge": ["merge.cu", "ptx.cuh", "internal.h"],
    "fwd_fp8": ["fwd_fp8.cu", "ptx.cuh", "schedule.h", "internal.h"],
    "decode": ["fwd.cu", "ptx.cuh", "schedule.h", "internal.h"],   # the forward kernel in decode mode
}


def fwd_flops(B, H, N, d, causal):
    return 4.0 * B * H * N * N * d * (0.5 if causal else 1.0)


def step_flops(w):
    f = fwd_flops(w["B"], w["Hq"], w["N"], w["d"], w["mask"] == "causal")
    return f, 2.5 * f


def kernel_work(w):
    """Algorithmic work per launch of each kernel of one step: counted GEMM
    FLOPs (one N x N x d product = 2*B*H*N^2*d, halved under the causal mask)
    for the tensor-bound kernels, bytes read once plus written once for the
    HBM-bound preprocessing kernel."""
    B, H, N, d = w["B"], w["Hq"], w["N"], w["d"]
    cf = 0.5 if w["mask"] == "causal" else 1.0
    gemm = 2.0 * B * H * N * N * d * cf          # one N x N x d product over all heads
    Np = -(-N // 128) * 128
    return {
        "fwd": ("tensor", 2 * gemm),                 # S = QK^T, O = PV
        "bwd_dkdv": ("tensor", 4 * gemm),            # S^T, dP^T, dV, dK
        "bwd_dq": ("tensor", 1 * gemm),              # dQ (S and dP are recomputed, not counted)
        "bwd_preprocess": ("hbm", 2 * B * H * N * d * 2 + 4 * B * H * N + 2 * 4 * B * H * Np),
    }


def executed_gemms(kernel, d):
    """N x N x d products each kernel runs per step, counted or not: the dQ
    kernel recomputes S and dP next to its dQ product, and the dK/dV
    kernel's S^T and dP^T products each have one more K = 16 step (the
    per-query statistics), so the backward runs 7 + 32/d products for the five
    the metric's 2.5x convention credits."""
    return {"fwd": 2, "bwd_dkdv": 4 + 2 * 16 / d, "bwd_dq": 3}.get(kernel)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_text(src):
    """A source file's code with its comments and blank lines removed, so that
    editing a comment does not mark the ncu summaries of its kernels stale
    (string literals in these sources hold no comment markers)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def source_hash(kernel):
    """Hash of the code (comments excluded) a kernel is compiled from; an ncu
    summary whose recorded hash differs was taken on other code."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "io_aware_exact_attn_gb300", "csrc", f)) as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def profile_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    for path in glob.glob(os.path.join(ROOT, "profiles", f"{kernel}_{workload}*.txt")):
        text = open(path).read()
        m_hash = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
        m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if m_hash and m_bytes and m_hash.group(1) == source_hash(kernel):
            return float(m_bytes.group(1))
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id is not None:
                cmd += ["-i", str(self.gpu_id)]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


def slowest_rank_ms(elapsed_ms, dist, device):
    """Every rank's timed region ends at a barrier; the job's time is the slowest rank's."""
    if dist is None:
        return float(elapsed_ms)
    import torch
    t = torch.tensor([float(elapsed_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, steps, flops_per_rank_step, elapsed_ms):
    """Whole-job throughput: every rank processes its own batch (weak scaling)."""
    return world * steps * flops_per_rank_step / (elapsed_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ oracle leg

def oracle_sample(seconds, rank=0, block=256):
    """Time the fp64 oracle (forward and backward, as it stands) on full-length
    rows of the workload: blocks of `block` query rows drawn uniformly from the
    N = 8192 positions of one head (each row against all of its visible keys,
    so the causal cost averages as in the full workload), block after block
    for about `seconds` seconds (at least one block).  The full configuration's
    time is extrapolated from the rows per second."""
    import numpy as np
    import oracle
    from oracle import attention as oa
    from io_aware_exact_attn_gb300 import inputs
    w = WORKLOAD
    N, d = w["N"], w["d"]
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = inputs.make_qkvdo(1, 1, 1, N, N, d, seed=inputs.SEED + 100 * rank)
    q, k, v, do = (inputs.to_f64(t)[0, 0] for t in (q, k, v, do))
    mask = oracle.MaskSpec("causal")
    rng = np.random.default_rng(inputs.SEED + 17)
    t0 = time.perf_counter()
    rows_done = 0
    while True:
        r = np.sort(rng.choice(N, block, replace=False))
        vis = oracle.visible(r, N, mask)
        oa.head_forward(q[r], k, v, scale, vis)
        oa.head_backward(q[r], k, v, do[r], scale, vis)
        rows_done += block
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    total_rows = w["B"] * w["Hq"] * N
    f, b = step_flops(w)
    full_s = el * total_rows / rows_done
    return dict(value=(f + b) / full_s / 1e12, unit="TFLOP/s", cores=os.cpu_count(), kind="oracle",
                sample=f"{rows_done} full-length query rows ({rows_done // block} blocks of {block} rows drawn "
                       f"uniformly from N={N}) of one head of the causal d={d} workload, fp64 NumPy forward and "
                       f"backward with full score rows, {el:.1f} s measured; BLAS threads = default "
                       f"(all {os.cpu_count()} host cores)",
                measured_sample_s=el, sampled_rows=rows_done, full_config_rows=total_rows,
                full_config_s_extrapolated=full_s, seconds=el)


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle  # noqa: F401
    for _ in range(args.warmup):
        oracle_sample(0.0)
    times = []
    rows = 0
    for _ in range(args.steps):
        r = oracle_sample(0.0)
        times.append(r["seconds"])
        rows += r["sampled_rows"]
        total_rows = r["full_config_rows"]
    total = sum(times)
    f, b = step_flops(WORKLOAD)
    value = (f + b) * rows / total_rows / total / 1e12
    cpu = dict(value=value, unit="TFLOP/s", cores=os.cpu_count(), kind="oracle",
               sample=f"each step: 256 full-length query rows drawn uniformly from one head of the causal "
                      f"d={WORKLOAD['d']} N={WORKLOAD['N']} workload, fp64 NumPy oracle forward and backward on "
                      f"the host cores",
               full_config_s_extrapolated=total * total_rows / rows)
    line = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
                ms_per_step=1e3 * total / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=workload_desc(WORKLOAD), sample="256 full-length query rows per step"),
                cpu_baseline=cpu, e2e=dict(value=value, unit="TFLOP/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def workload_desc(w):
    return (f"{w['name']}: B={w['B']} Hq={w['Hq']} Hkv={w['Hkv']} N={w['N']} d={w['d']} {w['mask']}, "
            f"bf16 N(0,1) inputs, scale 1/sqrt(d)")


# ------------------------------------------------------------------ GPU leg

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extras", action="store_true", help="skip the e2e, chunked and CPU legs")
    ap.add_argument("--profile-pass", action="store_true",
                    help="one untimed step and one E4M3 forward only (for profiler captures); prints nothing")
    ap.add_argument("--profile-workload", default=None,
                    choices=["gpt", "gpt_noncausal", "block_sparse", "bert_large", "decode", "varlen", "chunked_bwd",
                             "fp8"],
                    help="one untimed forward + backward of the named workload only (for profiler captures; the "
                         "ragged batch is cut to 8 sequences); prints nothing")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.warmup < 3 and not args.profile_pass:
        raise SystemExit("--warmup must be at least 3")

    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from io_aware_exact_attn_gb300 import api, inputs

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    if args.profile_workload:
        profile_workload(args.profile_workload, api, inputs, torch)
        torch.cuda.synchronize()
        assert api.get_status() == 0
        return 0

    w = WORKLOAD
    causal = w["mask"] == "causal"
    q, k, v, do = (t.cuda() for t in inputs.make_qkvdo(w["B"], w["Hq"], w["Hkv"], w["N"], w["N"], w["d"],
                                                       seed=inputs.SEED + 100 * rank))
    o = torch.empty_like(q)
    lse = torch.empty(w["B"], w["Hq"], w["N"], device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(api.bwd_workspace_bytes(w["B"], w["Hq"], w["Hkv"], w["N"], w["d"]), device="cuda",
                     dtype=torch.uint8)

    def step():
        api.attn_fwd(q, k, v, causal=causal, out=o, lse=lse)
        api.attn_bwd(q, k, v, o, lse, do, causal=causal, workspace=ws, dq=dq, dk=dk, dv=dv)

    if args.profile_pass:
        step()
        # and one E4M3 forward on the same shape (the fp8_fwd leg's workload)
        f = FP8
        q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(f["B"], f["Hq"], f["Hkv"], f["N"], f["d"])
        api.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, causal=True)
        # and one pass of the chunked workload (36 partial forwards, 8 merges)
        chunked_setup(api, inputs, torch, rank)[-1]()
        torch.cuda.synchronize()
        return 0

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.get_status() == 0

    props = torch.cuda.get_device_properties(local)
    gpu_id = None
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        gpu_id = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    api.trace_enable(8 * args.steps + 64)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = t0.elapsed_time(t1)
    api.trace_disable()
    clocks = sampler.stop()
    recs, n_launch = api.trace_read(8 * args.steps + 64)
    status = api.get_status()
    elapsed_ms = slowest_rank_ms(elapsed_ms, dist, "cuda")

    f_fwd, f_bwd = step_flops(w)
    ms_step = elapsed_ms / args.steps
    value = job_tflops(world, args.steps, f_fwd + f_bwd, elapsed_ms)
    peaks, peak_src = load_peaks()
    peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    peak_burst = peaks["bf16_tflops"]

    # per-kernel durations (CUDA events on the launching stream, inside the timed region)
    per = {}
    for name, ms in recs:
        per.setdefault(name, []).append(ms)
    work = kernel_work(w)
    kernels = {}
    for name, lst in per.items():
        avg = sum(lst) / len(lst)
        kind, amount = work.get(name, ("?", 0.0))
        entry = dict(launches=len(lst), avg_ms=avg, share=sum(lst) / sum(sum(x) for x in per.values()))
        if kind == "tensor":
            entry["tflops"] = amount / (avg * 1e-3) / 1e12
            gem = 2.0 * w["B"] * w["Hq"] * w["N"] * w["N"] * w["d"] * (0.5 if w["mask"] == "causal" else 1.0)
            entry["tflops_executed"] = executed_gemms(name, w["d"]) * gem / (avg * 1e-3) / 1e12
        elif kind == "hbm":
            entry["gbs"] = amount / (avg * 1e-3) / 1e9
        kernels[name] = entry
    dom = max(kernels, key=lambda n: kernels[n]["share"])
    kind, amount = work[dom]
    if kind == "tensor":
        # the timed region lasts well under the seconds-long loop the sustained
        # peak was measured over, so the burst peak is the denominator
        ach = kernels[dom]["tflops"]
        roof = dict(bound="tensor", achieved=ach, peak=peak_burst, unit="TFLOP/s", frac=ach / peak_burst,
                    traffic=profile_traffic(dom, w["name"]), kernel=dom,
                    peak_source=f"{peak_src} bf16_tflops (burst: timed region of {elapsed_ms / 1e3:.2f} s)",
                    frac_of_sustained_peak=ach / peak_sus)
    else:
        ach = kernels[dom]["gbs"]
        roof = dict(bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s", frac=ach / peaks["hbm_gbs"],
                    traffic=profile_traffic(dom, w["name"]), kernel=dom, peak_source=f"{peak_src} hbm_gbs")
    fwd_ms = kernels.get("fwd", {}).get("avg_ms", float("nan"))
    bwd_ms = sum(kernels.get(n, {}).get("avg_ms", 0.0) for n in ("bwd_preprocess", "bwd_dkdv", "bwd_dq"))
    split = dict(fwd_tflops=f_fwd / (fwd_ms * 1e-3) / 1e12, bwd_tflops=f_bwd / (bwd_ms * 1e-3) / 1e12)
    split["fwd_frac_of_burst_peak"] = split["fwd_tflops"] / peak_burst
    split["bwd_frac_of_burst_peak"] = split["bwd_tflops"] / peak_burst

    # parity spot check on the bench's own outputs (sampled rows vs the oracle)
    rows = np.array([0, 1, 127, 128, 4095, 8191])
    f64 = inputs.to_f64
    qh, kh, vh, doh = (f64(t[:1, :2]) for t in (q, k, v, do))
    o_ref, l_ref = oracle.attention_forward(qh, kh, vh, 1 / math.sqrt(w["d"]), oracle.MaskSpec("causal"),
                                            heads=[(0, 0), (0, 1)], rows=rows)
    o_err = float(np.abs(f64(o[0, :2, rows]) - o_ref).max())
    l_err = float(np.abs(f64(lse[0, :2, rows]) - l_ref).max())
    dq_ref = oracle.attention_backward_dq_rows(qh, kh, vh, doh, 1 / math.sqrt(w["d"]), 0, 1, rows,
                                               oracle.MaskSpec("causal"))
    dq_err = float(np.abs(f64(dq[0, 1, rows]) - dq_ref).max() / np.abs(dq_ref).max())
    parity = dict(rows_checked=int(2 * rows.size), o_max_abs=o_err, lse_max_abs=l_err, dq_rel=dq_err,
                  ok=bool(o_err <= 1e-2 and l_err <= 2e-3 and dq_err <= 3e-2 and status == 0))

    out = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
               ms_per_step=ms_step, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
               data="synthetic",
               config=dict(workload=workload_desc(w), B=w["B"], Hq=w["Hq"], Hkv=w["Hkv"], N=w["N"], d=w["d"],
                           mask=w["mask"], per_rank="one independent batch per GPU",
                           l2="inputs larger than L2 (Q, K, V, O, dO are 134 MB each; L2 is 129 MB), no flush"),
               roofline=roof, kernels=kernels, split=split, gpu_launches=n_launch, parity=parity,
               pct_of_burst_peak=value / world / peak_burst)
    if clocks is not None:
        out["clocks"] = clocks

    if not args.no_extras:
        out["e2e"] = e2e_leg(api, inputs, torch, w, causal, rank)
        out["chunked_gqa"] = chunked_leg(api, inputs, torch, peaks, rank)
        out["noncausal"] = noncausal_leg(api, inputs, torch, peaks, rank, kernels)
        out["sliding_window"] = window_leg(api, inputs, torch, peaks, rank)
        out["decode"] = decode_leg(api, inputs, torch, peaks, rank)
        out["varlen"] = varlen_leg(api, inputs, torch, peaks, rank)
        out["fp8_fwd"] = fp8_leg(api, inputs, torch, peaks, rank)
        out["configs"] = configs_leg(api, inputs, torch, peaks, rank)
        if rank == 0:
            out["cpu_baseline"] = {k_: v_ for k_, v_ in oracle_sample(args.cpu_seconds).items()
                                   if k_ not in ("seconds",)}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


def profile_workload(name, api, inputs, torch):
    """One untimed pass of a workload, for a profiler to capture: launches in
    the order forward, then backward (preprocess, dK/dV, dQ)."""
    if name in ("gpt", "gpt_noncausal", "block_sparse", "bert_large"):
        w = inputs.WORKLOADS["gpt_causal" if name == "gpt" else name]
        q, k, v, do = (t.cuda() for t in w.tensors())
        bm_np = w.block_mask()
        bm = None if bm_np is None else torch.as_tensor(bm_np, dtype=torch.uint8).cuda()
        causal = w.mask == "causal"
        o, lse = api.attn_fwd(q, k, v, causal=causal, block_mask=bm)
        api.attn_bwd(q, k, v, o, lse, do, causal=causal, block_mask=bm)
    elif name == "decode":
        c = DECODE
        g = torch.Generator().manual_seed(inputs.SEED + 9)
        q = torch.randn(c["B"], c["Hq"], c["Nq"], c["d"], generator=g).to(torch.bfloat16).cuda()
        k = torch.randn(c["B"], c["Hkv"], c["Nk"], c["d"], generator=g).to(torch.bfloat16).cuda()
        v = torch.randn(c["B"], c["Hkv"], c["Nk"], c["d"], generator=g).to(torch.bfloat16).cuda()
        api.attn_decode(q, k, v)
    elif name == "varlen":
        import numpy as np
        c = VARLEN
        lens = varlen_lengths(inputs.SEED + 11)[:8]
        total = sum(lens)
        g = torch.Generator().manual_seed(inputs.SEED + 12)
        q, k, v, do = (torch.randn(total, h, c["d"], generator=g).to(torch.bfloat16).cuda()
                       for h in (c["Hq"], c["Hkv"], c["Hkv"], c["Hq"]))
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
        o, lse = api.attn_varlen_fwd(q, k, v, cu, max(lens), causal=True)
        api.attn_varlen_bwd(q, k, v, o, lse, do, cu, max(lens), causal=True)
    elif name == "fp8":
        f = FP8
        q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(f["B"], f["Hq"], f["Hkv"], f["N"], f["d"])
        api.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, causal=True)
    elif name == "chunked_bwd":
        c = CHUNKED
        q, k, v, o, lse, run = chunked_setup(api, inputs, torch, 0)
        run()
        g = torch.Generator().manual_seed(inputs.SEED + 4)
        do = torch.randn(c["B"], c["Hq"], c["N"], c["d"], generator=g).to(torch.bfloat16).cuda()
        api.chunked_bwd(q, k, v, o, lse, do, c["chunks"])


def e2e_leg(api, inputs, torch, w, causal, rank, steps=30, chunks_per_batch=2):
    """Same metric through the public API with pinned HOST buffers: every step copies
    Q, K, V, dO to the device and O, LSE, dQ, dK, dV back.  The step is cut into
    (batch, head-block) chunks that are independent problems; each chunk's copies
    in, forward + backward, and copies out run on three streams, so one chunk's
    transfers overlap another's kernels.  The same step run as one chunk on one
    stream is reported beside it."""
    B, Hq, Hkv, N, d = w["B"], w["Hq"], w["Hkv"], w["N"], w["d"]
    hq, hk, hv, hdo = (t.pin_memory() for t in inputs.make_qkvdo(B, Hq, Hkv, N, N, d,
                                                                  seed=inputs.SEED + 100 * rank + 7))
    outs = [torch.empty(B, Hq, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hq, N, dtype=torch.float32).pin_memory(),
            torch.empty(B, Hq, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16).pin_memory()]
    dev_in = [torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (hq, hk, hv, hdo)]
    dev_out = [torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in outs]
    g = Hq // Hkv
    kvc = Hkv // chunks_per_batch if Hkv % chunks_per_batch == 0 else Hkv   # kv heads per chunk
    pieces = [(b, h0) for b in range(B) for h0 in range(0, Hkv, kvc)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_done = [torch.cuda.Event() for _ in pieces]   # a chunk's kernels finished (its inputs are free)
    ev_in = [torch.cuda.Event() for _ in pieces]
    ev_out = [torch.cuda.Event() for _ in pieces]    # a chunk's results copied out (its outputs are free)

    def sl(b, h0, per):   # the chunk's [1, heads, ...] view: q-side tensors per = g, kv-side per = 1
        return (slice(b, b + 1), slice(h0 * per, (h0 + kvc) * per))

    def pipelined(first):
        for c, (b, h0) in enumerate(pieces):
            with torch.cuda.stream(s_in):
                if not first:
                    s_in.wait_event(ev_done[c])
                for i, (dst, src) in enumerate(zip(dev_in, (hq, hk, hv, hdo))):
                    idx = sl(b, h0, g if i in (0, 3) else 1)
                    dst[idx].copy_(src[idx], non_blocking=True)
                ev_in[c].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[c])
                if not first:
                    s_cmp.wait_event(ev_out[c])
                qi, ki, vi, doi = (t[sl(b, h0, g if i in (0, 3) else 1)] for i, t in enumerate(dev_in))
                o_, l_, dq_, dk_, dv_ = (t[sl(b, h0, g if i < 3 else 1)] for i, t in enumerate(dev_out))
                api.attn_fwd(qi, ki, vi, causal=causal, out=o_, lse=l_)
                api.attn_bwd(qi, ki, vi, o_, l_, doi, causal=causal, dq=dq_, dk=dk_, dv=dv_)
                ev_done[c].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[c])
                for i, (dst, src) in enumerate(zip(outs, dev_out)):
                    idx = sl(b, h0, g if i < 3 else 1)
                    dst[idx].copy_(src[idx], non_blocking=True)
                ev_out[c].record(s_out)

    def sequential():
        q, k, v, do = (t.to("cuda", non_blocking=True) for t in (hq, hk, hv, hdo))
        o, lse = api.attn_fwd(q, k, v, causal=causal)
        dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=causal)
        for dst, src in zip(outs, (o, lse, dq, dk, dv)):
            dst.copy_(src, non_blocking=True)

    def timed(fn):
        for i in range(2):
            fn(i == 0) if fn is pipelined else fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn(False) if fn is pipelined else fn()
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    el = timed(pipelined)
    piped = [t.clone() for t in outs]
    el_seq = timed(sequential)
    # both schedules compute every (batch, head) problem with the same kernels
    same = max(float((a.float() - b_.float()).abs().max()) for a, b_ in zip(piped, outs))
    f_fwd, f_bwd = step_flops(w)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in outs)
    return dict(value=steps * (f_fwd + f_bwd) / el / 1e12, unit="TFLOP/s", h2d_bytes_per_step=h2d,
                d2h_bytes_per_step=d2h, steps=steps, ms_per_step=1e3 * el / steps, chunks=len(pieces),
                one_chunk_one_stream_ms_per_step=1e3 * el_seq / steps, chunked_vs_one_chunk_max_abs=same)


def chunked_setup(api, inputs, torch, rank):
    """Inputs, partial buffers and one pass of the chunked causal GQA workload
    (B=1, Hq=32, Hkv=8, N=32768, d=128, 8 chunks): the 36 partial forwards in
    load-balanced order, then one LSE merge per query chunk."""
    c = CHUNKED
    B, Hq, Hkv, N, d, nc = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["chunks"]
    L = N // nc
    q, k, v, _ = (t.cuda() for t in inputs.make_qkvdo(B, Hq, Hkv, N, N, d, seed=inputs.SEED + 100 * rank + 3))
    sched = api.build_chunk_schedule(nc)
    parts = {p: (torch.empty(B, Hq, L, d, device="cuda"), torch.empty(B, Hq, L, device="cuda")) for p in sched}
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, N, device="cuda")

    def run():
        for qc, kc in sched:
            api.attn_partial_fwd(q[:, :, qc * L:(qc + 1) * L], k[:, :, kc * L:(kc + 1) * L],
                                 v[:, :, kc * L:(kc + 1) * L], qc * L, kc * L, causal=True,
                                 o_part=parts[(qc, kc)][0], lse_part=parts[(qc, kc)][1])
        for qc in range(nc):
            api.attn_merge_lse([parts[(qc, kc)][0] for kc in range(qc + 1)],
                               [parts[(qc, kc)][1] for kc in range(qc + 1)],
                               out=o[:, :, qc * L:(qc + 1) * L], lse_out=lse[:, :, qc * L:(qc + 1) * L])

    return q, k, v, o, lse, run


def chunked_leg(api, inputs, torch, peaks, rank, reps=3):
    """The chunked causal GQA workload: partial forwards and merges timed from
    the library's launch trace, and the merged result against monolithic attn_fwd."""
    c = CHUNKED
    B, Hq, Hkv, N, d, nc = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["chunks"]
    L = N // nc
    q, k, v, o, lse, run = chunked_setup(api, inputs, torch, rank)
    run()
    torch.cuda.synchronize()
    api.trace_enable(64 * reps)
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    api.trace_disable()
    recs, _ = api.trace_read(64 * reps)
    part_ms = sum(ms for n, ms in recs if n == "partial_fwd") / reps
    merge_ms = sum(ms for n, ms in recs if n == "merge") / reps
    flops = fwd_flops(B, Hq, N, d, True)
    merge_bytes = sum((qc + 1) * (B * Hq * L * (d * 4 + 4)) for qc in range(nc)) + B * Hq * N * (d * 2 + 4)
    # monolithic causal forward on the same tensors, and agreement with the chunked result
    o_m, l_m = api.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    agree = dict(o_max_abs=float((o.float() - o_m.float()).abs().max()),
                 lse_max_abs=float((lse - l_m).abs().max()))
    gbs = merge_bytes / (merge_ms * 1e-3) / 1e9
    # DRAM bytes of the last query chunk's merge (8 parts) from the committed ncu
    # summary, beside that launch's algorithmic bytes
    last_alg = nc * (B * Hq * L * (d * 4 + 4)) + B * Hq * L * (d * 2 + 4)
    del o_m, l_m
    bwd = chunked_bwd_leg(api, inputs, torch, peaks, rank, q, k, v, o, lse)
    return dict(workload=f"B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} causal, {nc} chunks, {nc * (nc + 1) // 2} pairs",
                backward=bwd,
                partial_fwd_ms=part_ms, partial_fwd_tflops=flops / (part_ms * 1e-3) / 1e12,
                merge_ms=merge_ms, merge_bytes=merge_bytes, merge_gbs=gbs, merge_frac_of_hbm=gbs / peaks["hbm_gbs"],
                merge_roofline=dict(bound="hbm", achieved=gbs, peak=peaks["hbm_gbs"], unit="GB/s",
                                    frac=gbs / peaks["hbm_gbs"], peak_source="measured hbm_gbs",
                                    traffic_last_merge=profile_traffic("merge", "chunked_gqa"),
                                    algorithmic_bytes_last_merge=last_alg),
                chunked_vs_monolithic=agree)


def chunked_bwd_leg(api, inputs, torch, peaks, rank, q, k, v, o, lse, reps=3):
    """Backward of the chunked causal GQA workload, the chunked way: one
    preprocess per query chunk on the merged O and LSE, then the 36 pair
    backwards in the load-balanced order adding into float32 dQ, dK, dV, on one
    stream and dealt to two and three streams.  Timed with CUDA events around
    the whole backward (the side streams join the timing stream); FLOPs 2.5x
    the causal forward convention.  Compared with the monolithic attn_bwd."""
    c = CHUNKED
    B, Hq, Hkv, N, d, nc = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["chunks"]
    g = torch.Generator().manual_seed(inputs.SEED + 100 * rank + 4)
    do = torch.randn(B, Hq, N, d, generator=g).to(torch.bfloat16).cuda()
    dq = torch.zeros(B, Hq, N, d, device="cuda")
    dk = torch.zeros(B, Hkv, N, d, device="cuda")
    dv = torch.zeros(B, Hkv, N, d, device="cuda")
    flops = 2.5 * fwd_flops(B, Hq, N, d, True)
    res = {}
    for ns in (1, 2, 3):
        def run():
            for t in (dq, dk, dv):
                t.zero_()
            api.chunked_bwd(q, k, v, o, lse, do, nc, n_streams=ns, dq=dq, dk=dk, dv=dv)
        run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[ns] = ms
    zero_ms = (B * Hq * N * d * 4 + 2 * B * Hkv * N * d * 4) / (peaks["hbm_gbs"] * 1e9) * 1e3
    best = min(res, key=res.get)
    for t in (dq, dk, dv):
        t.zero_()
    api.chunked_bwd(q, k, v, o, lse, do, nc, n_streams=best, dq=dq, dk=dk, dv=dv)
    dq_m, dk_m, dv_m = api.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    agree = {n: float((a - b.float()).abs().max() / b.float().abs().max())
             for n, a, b in (("dq_rel", dq, dq_m), ("dk_rel", dk, dk_m), ("dv_rel", dv, dv_m))}
    # the monolithic backward on the same tensors, for comparison
    ws = torch.empty(api.bwd_workspace_bytes(B, Hq, Hkv, N, d), device="cuda", dtype=torch.uint8)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        api.attn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws, dq=dq_m, dk=dk_m, dv=dv_m)
    e1.record()
    torch.cuda.synchronize()
    mono_ms = e0.elapsed_time(e1) / reps
    return dict(what="8 preprocesses + 36 attn_partial_bwd pairs (float32 accumulation), zeroing included",
                ms_by_streams={str(n): m for n, m in res.items()},
                tflops_by_streams={str(n): flops / (m * 1e-3) / 1e12 for n, m in res.items()},
                best_streams=best, tflops=flops / (res[best] * 1e-3) / 1e12,
                frac_of_burst_peak=flops / (res[best] * 1e-3) / 1e12 / peaks["bf16_tflops"],
                zeroing_ms_at_hbm_peak=zero_ms,
                monolithic_attn_bwd_ms=mono_ms, monolithic_attn_bwd_tflops=flops / (mono_ms * 1e-3) / 1e12,
                chunked_vs_monolithic=agree)


def noncausal_leg(api, inputs, torch, peaks, rank, causal_kernels, reps=5):
    """The GPT shape without a mask (B=2, H=32, N=8192, d=128): forward and
    backward kernel times from the launch trace, and the causal step's time as
    a fraction of this one (causal tile skipping should bring it near 1/2)."""
    w = WORKLOAD
    B, Hq, Hkv, N, d = w["B"], w["Hq"], w["Hkv"], w["N"], w["d"]
    q, k, v, do = (t.cuda() for t in inputs.make_qkvdo(B, Hq, Hkv, N, N, d, seed=inputs.SEED + 100 * rank + 13))
    ws = torch.empty(api.bwd_workspace_bytes(B, Hq, Hkv, N, d), device="cuda", dtype=torch.uint8)

    def run():
        o, lse = api.attn_fwd(q, k, v)
        api.attn_bwd(q, k, v, o, lse, do, workspace=ws)

    run()
    torch.cuda.synchronize()
    api.trace_enable(16 * reps)
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    api.trace_disable()
    recs, _ = api.trace_read(16 * reps)
    fwd_ms = sum(ms for n, ms in recs if n == "fwd") / reps
    bwd_ms = sum(ms for n, ms in recs if n.startswith("bwd_")) / reps
    f_fwd = fwd_flops(B, Hq, N, d, False)
    c_fwd = causal_kernels.get("fwd", {}).get("avg_ms", float("nan"))
    c_bwd = sum(causal_kernels.get(n, {}).get("avg_ms", 0.0) for n in ("bwd_preprocess", "bwd_dkdv", "bwd_dq"))
    return dict(workload=f"B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} no mask", fwd_ms=fwd_ms, bwd_ms=bwd_ms,
                fwd_tflops=f_fwd / (fwd_ms * 1e-3) / 1e12, bwd_tflops=2.5 * f_fwd / (bwd_ms * 1e-3) / 1e12,
                step_tflops=3.5 * f_fwd / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                causal_over_noncausal_time=dict(fwd=c_fwd / fwd_ms, bwd=c_bwd / bwd_ms,
                                                step=(c_fwd + c_bwd) / (fwd_ms + bwd_ms)))


def window_pairs(N, w):
    """Visible (query, key) pairs of a sliding window of width w over N positions:
    row i sees min(i + 1, w) keys."""
    w = min(w, N)
    return w * (w + 1) // 2 + (N - w) * w


def configs_leg(api, inputs, torch, peaks, rank, reps=10):
    """The BERT-large-shaped (B=8, H=16, N=512, d=64, non-causal) and the
    block-sparse (B=1, H=16, N=16384, d=64, 128 x 128 blocks, diagonal plus
    1/8 of the rest) workloads: forward and backward kernel times from the
    library's launch trace, FLOPs by the metric's convention (4 B H N^2 d for
    the forward, 2.5x for the backward, times the kept-block fraction)."""
    res = {}
    for name in ("bert_large", "block_sparse"):
        w = inputs.WORKLOADS[name]
        q, k, v, do = (t.cuda() for t in w.tensors(seed=inputs.SEED + 100 * rank + 9))
        bm_np = w.block_mask()
        bm = None if bm_np is None else torch.as_tensor(bm_np, dtype=torch.uint8).cuda()
        ws = torch.empty(api.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d), device="cuda", dtype=torch.uint8)
        kept = 1.0 if bm_np is None else float(bm_np.mean())

        def run():
            o, lse = api.attn_fwd(q, k, v, block_mask=bm)
            api.attn_bwd(q, k, v, o, lse, do, block_mask=bm, workspace=ws)

        run()
        torch.cuda.synchronize()
        api.trace_enable(16 * reps)
        for _ in range(reps):
            run()
        torch.cuda.synchronize()
        api.trace_disable()
        recs, _ = api.trace_read(16 * reps)
        fwd_ms = sum(ms for n, ms in recs if n == "fwd") / reps
        bwd_ms = sum(ms for n, ms in recs if n.startswith("bwd_")) / reps
        f_fwd = 4.0 * w.B * w.Hq * w.N * w.N * w.d * kept
        res[name] = dict(workload=f"B={w.B} H={w.Hq} N={w.N} d={w.d} {w.mask}" +
                         ("" if bm_np is None else f" (kept block fraction {kept:.4f})"),
                         fwd_ms=fwd_ms, bwd_ms=bwd_ms, fwd_tflops=f_fwd / (fwd_ms * 1e-3) / 1e12,
                         bwd_tflops=2.5 * f_fwd / (bwd_ms * 1e-3) / 1e12,
                         step_tflops=3.5 * f_fwd / ((fwd_ms + bwd_ms) * 1e-3) / 1e12)
    return res


def window_leg(api, inputs, torch, peaks, rank, reps=5):
    """Sliding-window (local causal) attention at the GPT shape: B=2, H=32,
    N=8192, d=128, each query sees itself and the 4095 positions before it.
    FLOPs count the visible pairs: fwd 4*d per pair and head, bwd 2.5x that."""
    c = WINDOW
    B, Hq, Hkv, N, d, wnd = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["window"]
    q, k, v, do = (t.cuda() for t in inputs.make_qkvdo(B, Hq, Hkv, N, N, d, seed=inputs.SEED + 100 * rank + 5))
    ws = torch.empty(api.bwd_workspace_bytes(B, Hq, Hkv, N, d), device="cuda", dtype=torch.uint8)

    def run():
        o, lse = api.attn_fwd(q, k, v, window=wnd)
        api.attn_bwd(q, k, v, o, lse, do, window=wnd, workspace=ws)

    run()
    torch.cuda.synchronize()
    api.trace_enable(16 * reps)
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    api.trace_disable()
    recs, _ = api.trace_read(16 * reps)
    fwd_ms = sum(ms for n, ms in recs if n == "fwd") / reps
    bwd_ms = sum(ms for n, ms in recs if n.startswith("bwd_")) / reps
    f_fwd = 4.0 * B * Hq * d * window_pairs(N, wnd)
    return dict(workload=f"B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} sliding window {wnd}",
                visible_fraction_of_causal=window_pairs(N, wnd) / (N * (N + 1) / 2),
                fwd_ms=fwd_ms, bwd_ms=bwd_ms, fwd_tflops=f_fwd / (fwd_ms * 1e-3) / 1e12,
                bwd_tflops=2.5 * f_fwd / (bwd_ms * 1e-3) / 1e12,
                step_tflops=3.5 * f_fwd / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                fwd_frac_of_burst_peak=f_fwd / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"])


def decode_leg(api, inputs, torch, peaks, rank, reps=20, splits=(0, 8, 16, 24)):
    """Split-KV decoding: one new token per sequence (B=8, Hq=32, Hkv=8, d=128)
    against a full 32768-position cache.  HBM-bound: the algorithmic bytes are
    the cache read once (K and V), the queries read and the outputs written."""
    c = DECODE
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    gen = torch.Generator().manual_seed(inputs.SEED + 100 * rank + 9)
    q = torch.randn(B, Hq, Nq, d, generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn(B, Hkv, Nk, d, generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, Nk, d, generator=gen).to(torch.bfloat16).cuda()
    algo_bytes = 2 * B * Hkv * Nk * d * 2 + B * Hq * Nq * (d * 2 * 2 + 4)
    res = {}
    for ns in splits:
        ws = torch.empty(api.decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, ns), device="cuda", dtype=torch.uint8)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, Nq, device="cuda")
        for _ in range(3):
            api.attn_decode(q, k, v, n_splits=ns, out=o, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        api.trace_enable(4 * reps)
        for _ in range(reps):
            api.attn_decode(q, k, v, n_splits=ns, out=o, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        api.trace_disable()
        recs, _ = api.trace_read(4 * reps)
        dec_ms = sum(ms for n, ms in recs if n == "decode") / reps
        mrg_ms = sum(ms for n, ms in recs if n == "merge") / reps
        res[ns] = (dec_ms, mrg_ms)
    auto = api.decode_splits(B, Hkv, Nk)
    dec_ms, mrg_ms = res[0]
    gbs = algo_bytes / ((dec_ms + mrg_ms) * 1e-3) / 1e9
    return dict(workload=f"B={B} Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal, {auto} splits (automatic)",
                algorithmic_bytes=algo_bytes, decode_ms=dec_ms, merge_ms=mrg_ms, gbs=gbs,
                frac_of_hbm=gbs / peaks["hbm_gbs"],
                by_splits={str(ns if ns else auto): dict(decode_ms=a, merge_ms=b,
                                                         gbs=algo_bytes / ((a + b) * 1e-3) / 1e9)
                           for ns, (a, b) in res.items()})


def varlen_lengths(seed):
    """Seeded ragged lengths: uniform in [min_len, max_len] (the longest forced to max_len)."""
    import numpy as np
    c = VARLEN
    rng = np.random.default_rng(seed)
    lens = rng.integers(c["min_len"], c["max_len"] + 1, c["B"])
    lens[0] = c["max_len"]
    return [int(x) for x in lens]


def varlen_leg(api, inputs, torch, peaks, rank, reps=10):
    """Causal forward and backward over 16 packed sequences of 512..8192 tokens
    (H=32, d=128), token-major [total, H, d].  FLOPs: 4*H*d*len^2/2 per
    sequence forward (the causal convention of the main metric), 2.5x that
    backward."""
    import numpy as np
    c = VARLEN
    lens = varlen_lengths(inputs.SEED + 100 * rank + 11)
    total = sum(lens)
    g = torch.Generator().manual_seed(inputs.SEED + 100 * rank + 12)
    q, k, v, do = (torch.randn(total, h, c["d"], generator=g).to(torch.bfloat16).cuda()
                   for h in (c["Hq"], c["Hkv"], c["Hkv"], c["Hq"]))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(c["Hq"], total, device="cuda")
    ws = torch.empty(api.varlen_bwd_workspace_bytes(len(lens), total, c["Hq"]), device="cuda", dtype=torch.uint8)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

    def run():
        api.attn_varlen_fwd(q, k, v, cu, max(lens), causal=True, out=o, lse=lse)
        api.attn_varlen_bwd(q, k, v, o, lse, do, cu, max(lens), causal=True, workspace=ws, dq=grads[0],
                            dk=grads[1], dv=grads[2])

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    api.trace_enable(8 * reps)
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    api.trace_disable()
    recs, _ = api.trace_read(8 * reps)
    fwd_ms = sum(t for n, t in recs if n == "varlen_fwd") / reps
    bwd_ms = sum(t for n, t in recs if n.startswith("bwd_")) / reps
    flops = sum(4.0 * c["Hq"] * c["d"] * n * n * 0.5 for n in lens)
    return dict(workload=f"{c['B']} sequences, {c['min_len']}..{c['max_len']} tokens (total {total}), "
                         f"Hq={c['Hq']} Hkv={c['Hkv']} d={c['d']} causal, packed [total, H, d]",
                fwd_ms=fwd_ms, fwd_tflops=flops / (fwd_ms * 1e-3) / 1e12,
                bwd_ms=bwd_ms, bwd_tflops=2.5 * flops / (bwd_ms * 1e-3) / 1e12,
                fwd_frac_of_burst_peak=flops / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"])



def fp8_leg(api, inputs, torch, peaks, rank, reps=10):
    """Causal forward on E4M3 Q, K, V (per-tensor scales) at the GPT shape:
    B=2, H=32, N=8192, d=128.  Both products run on the fp8 tensor core; its
    peak is taken as twice the measured bf16 burst peak (the nominal fp8:bf16
    ratio).  The V transpose the kernel needs is timed separately."""
    c = FP8
    B, Hq, Hkv, N, d = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"]
    q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(B, Hq, Hkv, N, d, seed=inputs.SEED + 100 * rank + 7)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    ws = torch.empty(api.fwd_fp8_workspace_bytes(B, Hkv, N, d), device="cuda", dtype=torch.uint8)
    o = torch.empty((B, Hq, N, d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((B, Hq, N), device="cuda", dtype=torch.float32)

    def run():
        api.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=True, out=o, lse=lse, workspace=ws)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    api.trace_enable(4 * reps)
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    api.trace_disable()
    recs, _ = api.trace_read(4 * reps)
    fwd_ms = sum(ms for n, ms in recs if n == "fwd_fp8") / reps
    tr_ms = sum(ms for n, ms in recs if n == "fp8_transpose_v") / reps
    flops = fwd_flops(B, Hq, N, d, True)
    peak8 = 2.0 * peaks["bf16_tflops"]
    tr_bytes = 2.0 * B * Hkv * N * d
    ach = flops / (fwd_ms * 1e-3) / 1e12
    roof = dict(bound="tensor", achieved=ach, peak=peak8, unit="TFLOP/s", frac=ach / peak8,
                traffic=profile_traffic("fwd_fp8", c["name"]), kernel="fwd_fp8",
                peak_source="2 x measured bf16_tflops (burst; kernel timed alone), the nominal fp8:bf16 ratio")
    return dict(workload=f"B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} causal, e4m3 Q/K/V", roofline=roof,
                fwd_ms=fwd_ms, transpose_v_ms=tr_ms, fwd_tflops=flops / (fwd_ms * 1e-3) / 1e12,
                with_transpose_tflops=flops / ((fwd_ms + tr_ms) * 1e-3) / 1e12,
                fp8_peak_tflops=peak8, fwd_frac_of_fp8_peak=flops / (fwd_ms * 1e-3) / 1e12 / peak8,
                transpose_v_gbs=tr_bytes / (tr_ms * 1e-3) / 1e9)

if __name__ == "__main__":
    sys.exit(main())

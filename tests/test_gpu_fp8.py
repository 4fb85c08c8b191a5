"""GPU parity for the E4M3 (fp8) forward: attn_fwd_fp8 through the C ABI
against the fp64 oracle on the dequantised codes.

The kernel feeds the softmax weights to the second product as E4M3, so O is
compared element by element against the oracle's rigorous rounding bound
(``oracle.fp8_error_model``) plus the bf16 rounding of O, and its RMS error
against twice the model's expected rounding error (``_fp8_check.check``; a
CPU test shows that check failing on a wrong V tile, a dropped key tile and
reversed V rows); the LSE, which comes from fp32 sums of unrounded weights,
is held to 1e-3.  Cases cover ragged tails, causal, sliding-window and
block-sparse masks, GQA, peaked rows (the reference max moves), a single row,
and sampled rows of the full-size causal workload."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _fp8_check import check
from _gpu_helpers import mask_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def _np(t):
    return t.numpy() if t.device.type == "cpu" else t.cpu().numpy()


def run_case(B, Hq, Hkv, N, mask="none", window=0, density=0.25, kd_mul=1.0, seed=inputs.SEED):
    q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(B, Hq, Hkv, N, 128, seed)
    kd *= kd_mul
    scale = 1.0 / math.sqrt(128)
    bm = None
    kw = {}
    if mask == "causal":
        kw["causal"] = True
    elif mask == "sliding_window":
        kw["window"] = window
    elif mask == "block_sparse":
        nb = -(-N // 128)
        bm = inputs.block_sparse_mask(nb, nb, density, seed)
        kw["block_mask"] = torch.from_numpy(bm).cuda()
    o, lse = api.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, **kw)
    torch.cuda.synchronize()
    spec = mask_spec(mask, bm, False, window)
    args = (_np(q8), _np(k8), _np(v8), qd, kd, vd, scale, spec)
    o_ref, l_ref = oracle.fp8_forward(*args)
    bound, msq = oracle.fp8_error_model(*args)
    return o, lse, o_ref, l_ref, bound, msq


CASES = [
    (1, 2, 2, 128, "none", 0), (1, 2, 2, 300, "none", 0), (1, 2, 2, 300, "causal", 0),
    (2, 4, 2, 520, "causal", 0), (1, 3, 1, 777, "none", 0), (1, 2, 2, 1000, "sliding_window", 200),
    (1, 2, 2, 1000, "sliding_window", 129), (1, 2, 2, 1100, "block_sparse", 0), (1, 1, 1, 1, "none", 0),
    (1, 1, 1, 129, "causal", 0), (1, 2, 2, 2048, "causal", 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_N{}_{}{}".format(*c))
def test_fp8_fwd(case):
    B, Hq, Hkv, N, mask, w = case
    o, lse, o_ref, l_ref, bound, msq = run_case(B, Hq, Hkv, N, mask, w)
    check(o, lse, o_ref, l_ref, bound, msq, f"{mask} B{B} H{Hq}/{Hkv} N{N}")


@pytest.mark.parametrize("kd_mul", [4.0, 30.0])
def test_fp8_fwd_peaked_rows(kd_mul):
    """Larger K factors sharpen the rows: the reference max moves inside a row
    and most weights fall deep below the row max."""
    o, lse, o_ref, l_ref, bound, msq = run_case(1, 2, 2, 1500, "causal", kd_mul=kd_mul)
    check(o, lse, o_ref, l_ref, bound, msq, f"peaked x{kd_mul}")


def test_fp8_fwd_accepts_float8_tensors_and_matches_codes():
    q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(1, 2, 2, 256, 128)
    a = api.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, causal=True)
    b = api.attn_fwd_fp8(*(t.cuda().view(torch.float8_e4m3fn) for t in (q8, k8, v8)), qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_fwd_rejects_d64():
    q8 = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception):
        api.attn_fwd_fp8(q8, q8, q8)


def test_fp8_fwd_full_size_sampled_rows():
    """The benchmark's workload (B=2, H=32, N=8192, d=128, causal), sampled
    heads and rows against the oracle."""
    w = inputs.WORKLOADS["gpt_causal_fp8"]
    q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(w.B, w.Hq, w.Hkv, w.N, w.d)
    o, lse = api.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 4095, 4096, w.N - 129, w.N - 1],
                                     rng.integers(0, w.N, 40)]))
    spec = mask_spec("causal")
    for b, h in [(0, 0), (1, 31), (0, 17)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        args = (_np(q8[sl]), _np(k8[sl]), _np(v8[sl]), qd, kd, vd, w.scale, spec)
        o_ref, l_ref = oracle.fp8_forward(*args, heads=[(0, 0)], rows=rows)
        bound, msq = oracle.fp8_error_model(*args, heads=[(0, 0)], rows=rows)
        check(o[b, h][rows][None], lse[b, h][rows][None], o_ref, l_ref, bound, msq, f"full size b{b} h{h}")

"""The E4M3 forward's parity check can fail: on the GPU test's own causal
N=2048 case, the oracle's exact result with the E4M3 rounding of the weights
simulated (what a correct kernel computes) passes, and the same result with
a slip a kernel could make (key tile 3 multiplied with tile 2's V, key tile
0's P.V dropped, V rows reversed inside a tile, an all-zero O) fails."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import inputs
from _fp8_check import check

N, H = 2048, 2


@pytest.fixture(scope="module")
def case():
    q8, k8, v8, (qd, kd, vd) = inputs.make_qkv_e4m3(1, H, H, N, 128, inputs.SEED)
    q8, k8, v8 = q8.numpy(), k8.numpy(), v8.numpy()
    scale = 1.0 / math.sqrt(128)
    spec = oracle.MaskSpec("causal")
    args = (q8, k8, v8, qd, kd, vd, scale, spec)
    o_ref, l_ref = oracle.fp8_forward(*args)
    bound, msq = oracle.fp8_error_model(*args)
    q = qd * oracle.e4m3_decode(q8)
    k = kd * oracle.e4m3_decode(k8)
    v = vd * oracle.e4m3_decode(v8)
    s = np.where(np.tril(np.ones((N, N), bool)), scale * np.einsum("bhid,bhjd->bhij", q, k), -np.inf)
    w = np.exp(s - s.max(-1, keepdims=True))
    return dict(args=args, o_ref=o_ref, l_ref=l_ref, bound=bound, msq=msq, w=w, v=v)


def bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


def run_check(c, o):
    check(o, c["l_ref"], c["o_ref"], c["l_ref"], c["bound"], c["msq"], "planted")


@pytest.mark.parametrize("t", [7.0, 7.5, 8.0])
def test_simulated_correct_kernel_passes(case, t):
    w, v = case["w"], case["v"]
    p = torch.from_numpy(w * 2.0 ** t).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    o = np.einsum("bhij,bhjd->bhid", p, v) / (w * 2.0 ** t).sum(-1, keepdims=True)
    run_check(case, bf16(o))


def _fwd_with_v(case, v8_new):
    q8, k8, _, qd, kd, vd, scale, spec = case["args"]
    return oracle.fp8_forward(q8, k8, v8_new, qd, kd, vd, scale, spec)[0]


def test_wrong_v_tile_fails(case):
    v8 = case["args"][2].copy()
    v8[:, :, 384:512] = v8[:, :, 256:384]         # key tile 3 with tile 2's values
    with pytest.raises(AssertionError):
        run_check(case, bf16(_fwd_with_v(case, v8)))


def test_reversed_v_rows_fail(case):
    v8 = case["args"][2].copy()
    v8[:, :, 128:256] = v8[:, :, 128:256][:, :, ::-1]
    with pytest.raises(AssertionError):
        run_check(case, bf16(_fwd_with_v(case, v8)))


def test_dropped_key_tile_fails(case):
    w, v = case["w"], case["v"]
    part = np.einsum("bhij,bhjd->bhid", w[..., :128], v[:, :, :128]) / w.sum(-1, keepdims=True)
    with pytest.raises(AssertionError):
        run_check(case, bf16(case["o_ref"] - part))


def test_zero_output_fails(case):
    with pytest.raises(AssertionError):
        run_check(case, np.zeros_like(case["o_ref"]))

"""GPU parity for the sliding-window (local causal) mask: attn_fwd, attn_bwd,
attn_partial_fwd and the chunked merge through the C ABI against the fp64
oracle on the same seeded bf16 inputs.  Windows straddle tile edges (1, 100,
128, 129, ...), cover ragged sequence tails, GQA, both head sizes, peaked rows
and windows wider than the sequence (which must equal causal attention)."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_grad, assert_o_lse, f64, make, mask_spec, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def fwd_bwd(B, Hq, Hkv, N, d, w, k_mul=1.0):
    q, k, v, do = make(B, Hq, Hkv, N, d, k_mul=k_mul)
    o, lse = api.attn_fwd(q, k, v, window=w)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, window=w)
    torch.cuda.synchronize()
    return (q, k, v, do), (o, lse), (dq, dk, dv)


FWD_CASES = [
    (1, 2, 2, 1000, 128, 1), (1, 2, 2, 1000, 128, 100), (1, 2, 2, 1000, 128, 128), (1, 2, 2, 1000, 128, 129),
    (1, 2, 2, 1000, 64, 300), (2, 4, 2, 520, 64, 200), (1, 3, 1, 777, 128, 256), (1, 2, 2, 1000, 128, 999),
    (1, 2, 2, 300, 128, 5000), (1, 1, 1, 1, 64, 1),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "B{}_H{}-{}_N{}_d{}_w{}".format(*c))
def test_window_fwd(case):
    B, Hq, Hkv, N, d, w = case
    q, k, v, _ = make(B, Hq, Hkv, N, d)
    o, lse = api.attn_fwd(q, k, v, window=w)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), mask_spec("sliding_window",
                                                                                                  window=w))
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"window {w} B{B} H{Hq}/{Hkv} N{N} d{d}")


BWD_CASES = [
    (1, 2, 2, 1000, 128, 1), (1, 2, 2, 1000, 128, 100), (1, 2, 2, 1000, 128, 129), (1, 2, 2, 700, 64, 300),
    (2, 4, 2, 520, 64, 200), (1, 4, 2, 777, 128, 256), (1, 2, 2, 300, 128, 5000),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "B{}_H{}-{}_N{}_d{}_w{}".format(*c))
def test_window_bwd(case):
    B, Hq, Hkv, N, d, w = case
    (q, k, v, do), _, (dq, dk, dv) = fwd_bwd(B, Hq, Hkv, N, d, w)
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), 1 / math.sqrt(d),
                                           mask_spec("sliding_window", window=w))
    tag = f"window {w} B{B} H{Hq}/{Hkv} N{N} d{d}"
    assert_grad(f64(dq), gq, "dQ " + tag)
    assert_grad(f64(dk), gk, "dK " + tag)
    assert_grad(f64(dv), gv, "dV " + tag)


def test_window_peaked_rows():
    """K scaled by 4: peaked rows move the running max inside the window."""
    B, Hq, Hkv, N, d, w = 1, 2, 2, 1024, 128, 333
    (q, k, v, do), (o, lse), (dq, dk, dv) = fwd_bwd(B, Hq, Hkv, N, d, w, k_mul=4.0)
    mask = mask_spec("sliding_window", window=w)
    o_ref, l_ref = oracle.attention_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), mask)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, "peaked window")
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), 1 / math.sqrt(d), mask)
    assert_grad(f64(dq), gq, "dQ peaked window")
    assert_grad(f64(dk), gk, "dK peaked window")
    assert_grad(f64(dv), gv, "dV peaked window")


def test_wide_window_equals_causal():
    B, Hq, Hkv, N, d = 1, 2, 2, 640, 128
    q, k, v, do = make(B, Hq, Hkv, N, d)
    o_w, l_w = api.attn_fwd(q, k, v, window=N)
    o_c, l_c = api.attn_fwd(q, k, v, causal=True)
    g_w = api.attn_bwd(q, k, v, o_w, l_w, do, window=N + 7)
    g_c = api.attn_bwd(q, k, v, o_c, l_c, do, causal=True)
    torch.cuda.synchronize()
    assert max_err(f64(o_w), f64(o_c)) == 0.0 and max_err(f64(l_w), f64(l_c)) == 0.0
    for a, b in zip(g_w, g_c):
        assert max_err(f64(a), f64(b)) == 0.0


@pytest.mark.parametrize("d", [64, 128])
def test_window_partial_offsets_and_merge(d):
    """Chunk pairs with global offsets under the window, merged per query chunk,
    against the oracle and against the monolithic windowed forward."""
    B, Hq, Hkv, N, w = 1, 4, 2, 1024, 300
    n_chunks = 4
    c = N // n_chunks
    q, k, v, _ = make(B, Hq, Hkv, N, d)
    o_full, l_full = api.attn_fwd(q, k, v, window=w)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq, N), device="cuda", dtype=torch.float32)
    mask = mask_spec("sliding_window", window=w)
    for qc in range(n_chunks):
        parts = []
        for kc in range(qc + 1):
            qs, ks, vs = q[:, :, qc * c:(qc + 1) * c], k[:, :, kc * c:(kc + 1) * c], v[:, :, kc * c:(kc + 1) * c]
            op, lp = api.attn_partial_fwd(qs, ks, vs, qc * c, kc * c, window=w)
            torch.cuda.synchronize()
            ro, rl = oracle.attention_forward(f64(qs), f64(ks), f64(vs), 1 / math.sqrt(d), mask, qc * c, kc * c)
            assert_o_lse(f64(op), f64(lp), ro, rl, f"partial q{qc} k{kc}")
            parts.append((op, lp))
        api.attn_merge_lse([p[0] for p in parts], [p[1] for p in parts], out=o[:, :, qc * c:(qc + 1) * c],
                           lse_out=l[:, :, qc * c:(qc + 1) * c])
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), mask)
    assert_o_lse(f64(o), f64(l), o_ref, l_ref, "chunked window vs oracle")
    assert max_err(f64(o), f64(o_full)) <= 1e-2
    assert max_err(f64(l), f64(l_full)) <= 2e-3


def test_window_bad_width_is_rejected():
    q, k, v, _ = make(1, 1, 1, 128, 64)
    with pytest.raises(ValueError):
        api.attn_fwd(q, k, v, window=0)

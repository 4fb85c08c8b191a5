"""GPU parity for ragged batches (attn_varlen_fwd through the C ABI, packed
token-major tensors) against the fp64 oracle on the same seeded bf16 inputs:
lengths at and around tile edges (1, 127..129, 255..257), an empty sequence,
causal, non-causal and sliding-window masks, GQA and both head sizes; plus
agreement with the padded batched forward when all lengths are equal."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_o_lse, f64, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def packed(lens, Hq, Hkv, d, seed=inputs.SEED):
    total = int(sum(lens))
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(total, Hq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(total, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(total, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
    return q, k, v, cu


CASES = [
    # lens, Hq, Hkv, d, mask
    ([300, 1, 128, 129, 1000], 4, 2, 128, "causal"),
    ([300, 1, 128, 129, 1000], 4, 2, 64, "none"),
    ([255, 256, 257, 0, 127], 2, 2, 128, "causal"),
    ([700, 33, 512], 8, 2, 64, "causal"),
    ([1000, 400, 1], 4, 4, 128, ("window", 200)),
    ([2048], 2, 1, 128, "causal"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "lens{}_H{}-{}_d{}_{}".format(len(c[0]), c[1], c[2], c[3],
                                                                                        c[4] if isinstance(c[4], str)
                                                                                        else "window"))
def test_varlen_matches_oracle(case):
    lens, Hq, Hkv, d, mk = case
    q, k, v, cu = packed(lens, Hq, Hkv, d)
    window = mk[1] if isinstance(mk, tuple) else None
    causal = mk == "causal"
    o, lse = api.attn_varlen_fwd(q, k, v, cu, causal=causal, window=window)
    torch.cuda.synchronize()
    mask = (oracle.MaskSpec("sliding_window", window=window) if window else oracle.MaskSpec(mk))
    o_ref, l_ref = oracle.varlen_forward(f64(q), f64(k), f64(v), cu.cpu().numpy(), 1 / math.sqrt(d), mask)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"varlen {lens} {mk}")


def test_varlen_equal_lengths_match_batched_forward():
    B, Hq, Hkv, n, d = 3, 4, 2, 640, 128
    q, k, v, cu = packed([n] * B, Hq, Hkv, d)
    o, lse = api.attn_varlen_fwd(q, k, v, cu, causal=True)
    unpack = lambda x: x.view(B, n, x.shape[1], d).transpose(1, 2).contiguous()
    ob, lb = api.attn_fwd(unpack(q), unpack(k), unpack(v), causal=True)
    torch.cuda.synchronize()
    assert max_err(f64(o), f64(ob.transpose(1, 2).reshape(B * n, Hq, d))) == 0.0
    assert max_err(f64(lse), f64(lb.transpose(0, 1).reshape(Hq, B * n))) == 0.0


BWD_CASES = [
    # lens, Hq, Hkv, d, mask
    ([300, 1, 128, 129, 1000], 4, 2, 128, "causal"),
    ([255, 256, 257, 0, 127], 2, 2, 64, "causal"),
    ([700, 33, 512], 4, 4, 128, "none"),
    ([1000, 400, 1], 4, 2, 128, ("window", 200)),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "lens{}_H{}-{}_d{}_{}".format(len(c[0]), c[1], c[2], c[3],
                                                                                            c[4] if isinstance(c[4], str)
                                                                                            else "window"))
def test_varlen_backward_matches_oracle(case):
    from _gpu_helpers import assert_grad
    lens, Hq, Hkv, d, mk = case
    q, k, v, cu = packed(lens, Hq, Hkv, d)
    g = torch.Generator().manual_seed(inputs.SEED + 3)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16).cuda()
    window = mk[1] if isinstance(mk, tuple) else None
    causal = mk == "causal"
    o, lse = api.attn_varlen_fwd(q, k, v, cu, causal=causal, window=window)
    dq, dk, dv = api.attn_varlen_bwd(q, k, v, o, lse, do, cu, causal=causal, window=window)
    torch.cuda.synchronize()
    mask = (oracle.MaskSpec("sliding_window", window=window) if window else oracle.MaskSpec(mk))
    gq, gk, gv = oracle.varlen_backward(f64(q), f64(k), f64(v), f64(do), cu.cpu().numpy(), 1 / math.sqrt(d), mask)
    tag = f"varlen {lens} {mk}"
    assert_grad(f64(dq), gq, "dQ " + tag)
    assert_grad(f64(dk), gk, "dK " + tag)
    assert_grad(f64(dv), gv, "dV " + tag)


def test_varlen_backward_equal_lengths_match_batched_backward():
    B, Hq, Hkv, n, d = 2, 4, 2, 640, 128
    q, k, v, cu = packed([n] * B, Hq, Hkv, d)
    g = torch.Generator().manual_seed(inputs.SEED + 4)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16).cuda()
    o, lse = api.attn_varlen_fwd(q, k, v, cu, causal=True)
    grads = api.attn_varlen_bwd(q, k, v, o, lse, do, cu, causal=True)
    unpack = lambda x: x.view(B, n, x.shape[1], d).transpose(1, 2).contiguous()
    ob, lb = api.attn_fwd(unpack(q), unpack(k), unpack(v), causal=True)
    gb = api.attn_bwd(unpack(q), unpack(k), unpack(v), ob, lb, unpack(do), causal=True)
    torch.cuda.synchronize()
    for a, b in zip(grads, gb):
        assert max_err(f64(a), f64(b.transpose(1, 2).reshape(B * n, b.shape[1], d))) == 0.0

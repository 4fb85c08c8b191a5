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


def test_malformed_cu_seqlens_are_skipped_and_reported():
    """Device-side bounds check: a sequence whose cu_seqlens range runs past
    the packed tensors (or holds more than max_len tokens) is skipped by every
    kernel and reported by attn_get_status as ATTN_ERR_DEVICE_BOUNDS; the
    well-formed sequences of the same call are still exact."""
    from io_aware_exact_attn_gb300 import _ffi
    Hq, Hkv, d = 4, 2, 128
    total = 700
    q, k, v, _ = packed([total], Hq, Hkv, d)
    do = torch.randn(total, Hq, d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    cu = torch.tensor([0, 300, 600, 900], dtype=torch.int32).cuda()   # sequence 2 ends past total
    sentinel = 5.0
    o = torch.full_like(q, sentinel)
    lse = torch.full((Hq, total), sentinel, device="cuda")
    api.attn_varlen_fwd(q, k, v, cu, max_len=300, causal=True, out=o, lse=lse)
    dq = torch.full_like(q, sentinel)
    dk = torch.full_like(k, sentinel)
    dv = torch.full_like(v, sentinel)
    api.attn_varlen_bwd(q, k, v, o, lse, do, cu, max_len=300, causal=True, dq=dq, dk=dk, dv=dv)
    assert api.get_status() == -8 and _ffi.STATUS[-8] == "ATTN_ERR_DEVICE_BOUNDS"
    assert api.get_status() == 0              # read and cleared
    # the skipped sequence's rows are untouched, the others are exact
    assert bool((o[600:] == sentinel).all()) and bool((dq[600:] == sentinel).all())
    good = cu[:3].cpu().numpy()
    qf, kf, vf, dof = (f64(t[:600]) for t in (q, k, v, do))
    mask = oracle.MaskSpec("causal")
    o_ref, l_ref = oracle.varlen_forward(qf, kf, vf, good, 1 / math.sqrt(d), mask)
    assert_o_lse(f64(o[:600]), f64(lse[:, :600]), o_ref, l_ref, "well-formed sequences")
    gq, gk, gv = oracle.varlen_backward(qf, kf, vf, dof, good, 1 / math.sqrt(d), mask)
    for name, got, want in (("dQ", dq[:600], gq), ("dK", dk[:600], gk), ("dV", dv[:600], gv)):
        e = max_err(f64(got), want) / np.abs(want).max()
        assert e <= 3e-2, f"{name} of well-formed sequences: {e:.3e}"
    # a sequence longer than the max_len the caller promised is skipped too,
    # and so is one whose end precedes its start
    for bad in ([0, 300, 600], [0, 300, 200, 700]):
        api.attn_varlen_fwd(q[:bad[-1]], k[:bad[-1]], v[:bad[-1]], torch.tensor(bad, dtype=torch.int32).cuda(),
                            max_len=256 if len(bad) == 3 else 500, causal=True)
        assert api.get_status() == -8

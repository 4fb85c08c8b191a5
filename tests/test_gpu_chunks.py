"""GPU: the host-buffer step cut into (batch, head-block) chunks on three
streams (copies in, kernels, copies out) gives bit-identical results to the
same step run whole on one stream.  Each (batch, head) problem is independent,
so the chunks run the same per-head arithmetic; the test checks the slicing of
the contiguous [B, H, N, d] tensors into head blocks, the GQA head grouping and
the stream/event ordering between chunks, and pins the chunked result to the
fp64 oracle on one head."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_grad, assert_o_lse, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def chunked_step(host_in, outs, B, Hq, Hkv, causal, kv_per_chunk, steps=2):
    """The pipelined step: per chunk, copies in on one stream, forward and
    backward on a second, copies out on a third; device buffers are reused
    across steps and chunks wait for the previous step's use of their slice."""
    g = Hq // Hkv
    dev_in = [torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in host_in]
    dev_out = [torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in outs]
    pieces = [(b, h0) for b in range(B) for h0 in range(0, Hkv, kv_per_chunk)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in pieces]
    ev_done = [torch.cuda.Event() for _ in pieces]
    ev_out = [torch.cuda.Event() for _ in pieces]

    def sl(b, h0, per):
        return (slice(b, b + 1), slice(h0 * per, (h0 + kv_per_chunk) * per))

    for step in range(steps):
        for c, (b, h0) in enumerate(pieces):
            with torch.cuda.stream(s_in):
                if step:
                    s_in.wait_event(ev_done[c])
                for i, (dst, src) in enumerate(zip(dev_in, host_in)):
                    idx = sl(b, h0, g if i in (0, 3) else 1)
                    dst[idx].copy_(src[idx], non_blocking=True)
                ev_in[c].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[c])
                if step:
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
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,kvc", [
    (2, 8, 8, 384, 128, True, 4),     # MHA, two head blocks per batch
    (2, 8, 2, 300, 64, False, 1),     # GQA groups of 4 query heads, ragged N
])
def test_chunked_step_equals_whole_step(B, Hq, Hkv, N, d, causal, kvc):
    host_in = [t.pin_memory() for t in inputs.make_qkvdo(B, Hq, Hkv, N, N, d)]
    outs = [torch.empty(B, Hq, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hq, N, dtype=torch.float32).pin_memory(),
            torch.empty(B, Hq, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16).pin_memory()]
    chunked_step(host_in, outs, B, Hq, Hkv, causal, kvc)

    q, k, v, do = (t.cuda() for t in host_in)
    o, lse = api.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    for name, got, want in zip(("O", "LSE", "dQ", "dK", "dV"), outs, (o, lse, dq, dk, dv)):
        assert torch.equal(got, want.cpu()), f"{name} differs between the chunked and the whole step"

    # and one (batch, kv head) of the chunked result against the oracle
    b, hk = B - 1, Hkv - 1
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d)
    spec = oracle.MaskSpec("causal" if causal else "none")
    hq_ = slice(hk * g, (hk + 1) * g)
    o_ref, l_ref = oracle.attention_forward(f64(host_in[0][b:b + 1, hq_]), f64(host_in[1][b:b + 1, hk:hk + 1]),
                                            f64(host_in[2][b:b + 1, hk:hk + 1]), scale, spec)
    assert_o_lse(f64(outs[0][b:b + 1, hq_]), f64(outs[1][b:b + 1, hq_]), o_ref, l_ref, "chunked")
    dq_ref, dk_ref, dv_ref = oracle.attention_backward(
        f64(host_in[0][b:b + 1, hq_]), f64(host_in[1][b:b + 1, hk:hk + 1]), f64(host_in[2][b:b + 1, hk:hk + 1]),
        f64(host_in[3][b:b + 1, hq_]), scale, spec)
    assert_grad(f64(outs[2][b:b + 1, hq_]), dq_ref, "chunked dQ")
    assert_grad(f64(outs[3][b:b + 1, hk:hk + 1]), dk_ref, "chunked dK")
    assert_grad(f64(outs[4][b:b + 1, hk:hk + 1]), dv_ref, "chunked dV")

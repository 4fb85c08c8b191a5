"""Full-size parity on the benchmark workloads, in the launch configuration
bench.py times.  The fp64 oracle checks seeded samples it can compute in
seconds: O and LSE on sampled (head, row) pairs, dQ on sampled rows (each dQ
row depends only on its own row), and dK/dV of whole sampled heads.  Where the
oracle cannot afford a full head (the 32768-long chunked workload), properties
that hold at any size are checked GPU-against-GPU: chunked partial+merge equals
monolithic attention, and GQA gradients equal repeated-KV MHA gradients summed
over each group."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_grad, assert_o_lse, f64, mask_spec, max_err

pytestmark = pytest.mark.gpu

SAMPLE_SEED = 99


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    torch.cuda.empty_cache()
    assert api.get_status() == 0


def sample_heads_rows(B, H, N, n_heads=4, n_rows=256, seed=SAMPLE_SEED):
    rng = np.random.default_rng(seed)
    heads = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, B, n_heads * 3), rng.integers(0, H, n_heads * 3))})
    heads = heads[:n_heads]
    rows = np.unique(np.concatenate([rng.choice(N, n_rows - 3, replace=False), [0, N - 1, min(N - 1, 128)]]))
    return heads, rows


def gpu_fwd_bwd(w, bm=None):
    q, k, v, do = (t.cuda() for t in w.tensors())
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    causal = w.mask == "causal"
    win = w.window if w.mask == "sliding_window" else None
    o, lse = api.attn_fwd(q, k, v, causal=causal, block_mask=bmt, window=win)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=causal, block_mask=bmt, window=win)
    torch.cuda.synchronize()
    return (q, k, v, do), (o, lse), (dq, dk, dv)


def check_sampled(w, bm=None, n_kv_heads_full=1):
    (q, k, v, do), (o, lse), (dq, dk, dv) = gpu_fwd_bwd(w, bm)
    scale = 1.0 / math.sqrt(w.d)
    mask = mask_spec(w.mask, bm, window=w.window)
    heads, rows = sample_heads_rows(w.B, w.Hq, w.N)
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    o_ref, l_ref = oracle.attention_forward(qf, kf, vf, scale, mask, heads=heads, rows=rows)
    o_gpu = np.stack([f64(o[b, h, rows]) for b, h in heads])
    l_gpu = np.stack([f64(lse[b, h, rows]) for b, h in heads])
    assert_o_lse(o_gpu, l_gpu, o_ref, l_ref, w.name)
    for b, h in heads[:2]:
        ref = oracle.attention_backward_dq_rows(qf, kf, vf, dof, scale, b, h, rows, mask)
        assert_grad(f64(dq[b, h, rows]), ref, f"dQ rows {w.name} ({b},{h})")
    g = w.Hq // w.Hkv
    for b, h in heads[:n_kv_heads_full]:
        hk = h // g
        _, dk_ref, dv_ref = oracle.attention_backward(qf, kf, vf, dof, scale, mask, kv_heads=[(b, hk)])
        assert_grad(f64(dk[b, hk]), dk_ref[0], f"dK head {w.name} ({b},{hk})")
        assert_grad(f64(dv[b, hk]), dv_ref[0], f"dV head {w.name} ({b},{hk})")


def test_gpt_causal_full_size():
    check_sampled(inputs.WORKLOADS["gpt_causal"])


def test_gpt_causal_peaked_full_size():
    check_sampled(inputs.WORKLOADS["gpt_causal_peaked"])


def test_gpt_noncausal_full_size():
    check_sampled(inputs.WORKLOADS["gpt_noncausal"], n_kv_heads_full=1)


def test_gpt_sliding_window_full_size():
    check_sampled(inputs.WORKLOADS["gpt_sliding_window"])


def test_block_sparse_full_size():
    w = inputs.WORKLOADS["block_sparse"]
    bm = w.block_mask()
    assert int(bm.sum()) == 2160
    check_sampled(w, bm)


def test_chunked_gqa_full_size():
    """N=32768, Hq=32, Hkv=8, 8 chunks: 36 partial forwards in the load-balanced
    order, one merge per query chunk; equal to monolithic causal attn_fwd, and
    to the oracle on a sampled GQA group."""
    w = inputs.WORKLOADS["chunked_gqa"]
    q, k, v, do = (t.cuda() for t in w.tensors())
    L = w.N // w.chunks
    sched = api.build_chunk_schedule(w.chunks)
    assert sorted(sched) == sorted((a, b) for a in range(w.chunks) for b in range(a + 1))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.N, device="cuda", dtype=torch.float32)
    parts = {}
    for qc, kc in sched:
        parts[(qc, kc)] = api.attn_partial_fwd(q[:, :, qc * L:(qc + 1) * L], k[:, :, kc * L:(kc + 1) * L],
                                               v[:, :, kc * L:(kc + 1) * L], qc * L, kc * L, causal=True)
    for qc in range(w.chunks):
        api.attn_merge_lse([parts[(qc, kc)][0] for kc in range(qc + 1)],
                           [parts[(qc, kc)][1] for kc in range(qc + 1)],
                           out=o[:, :, qc * L:(qc + 1) * L], lse_out=lse[:, :, qc * L:(qc + 1) * L])
    del parts
    o_m, l_m = api.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert float((o.float() - o_m.float()).abs().max()) <= 1e-2
    assert float((lse - l_m).abs().max()) <= 2e-3
    scale = 1.0 / math.sqrt(w.d)
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    rng = np.random.default_rng(SAMPLE_SEED)
    rows = np.unique(np.concatenate([rng.choice(w.N, 125, replace=False), [0, L - 1, L, w.N - 1]]))
    hk = int(rng.integers(0, w.Hkv))
    heads = [(0, hk * 4 + j) for j in range(4)]            # one whole GQA group
    o_ref, l_ref = oracle.attention_forward(qf, kf, vf, scale, oracle.MaskSpec("causal"), heads=heads, rows=rows)
    o_gpu = np.stack([f64(o[b, h, rows]) for b, h in heads])
    l_gpu = np.stack([f64(lse[b, h, rows]) for b, h in heads])
    assert_o_lse(o_gpu, l_gpu, o_ref, l_ref, "chunked")
    # chunked backward on the merged result: one preprocess per query chunk,
    # the 36 pairs in the load-balanced order on two streams, into float32
    dq, dk, dv = api.chunked_bwd(q, k, v, o, lse, do, w.chunks, n_streams=2)
    dq_m, dk_m, dv_m = api.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    for name, got, want in (("dQ", dq, dq_m), ("dK", dk, dk_m), ("dV", dv, dv_m)):
        err = float((got - want.float()).abs().max() / want.float().abs().max())
        assert err <= 3e-2, f"chunked {name} vs monolithic: {err:.3e}"
    del dq_m, dk_m, dv_m
    # dQ rows against the oracle
    for b, h in heads[:2]:
        ref = oracle.attention_backward_dq_rows(qf, kf, vf, dof, scale, b, h, rows[:64], oracle.MaskSpec("causal"))
        assert_grad(f64(dq[b, h, rows[:64]]), ref, f"chunked dQ rows ({b},{h})")
    # dK / dV of the last two key tiles of one kv head: under the causal mask
    # only the last 256 query rows see them, and those rows' merged LSE and
    # D come from the oracle's own forward of those rows over all keys
    g = w.Hq // w.Hkv
    last = np.arange(w.N - 256, w.N)
    grp = [(0, hk * g + j) for j in range(g)]
    o_r, l_r = oracle.attention_forward(qf, kf, vf, scale, oracle.MaskSpec("causal"), heads=grp, rows=last)
    hq = [h for _, h in grp]
    dsum = (dof[0][hq][:, last] * o_r).sum(-1)
    _, dk_ref, dv_ref = oracle.partial_backward(qf[:, hq][:, :, last], kf[:, hk:hk + 1, last], vf[:, hk:hk + 1, last],
                                                dof[:, hq][:, :, last], l_r[None], dsum[None], scale,
                                                oracle.MaskSpec("causal"), w.N - 256, w.N - 256)
    assert_grad(f64(dk[0, hk, last]), dk_ref[0, 0], f"chunked dK last key tiles (kv head {hk})")
    assert_grad(f64(dv[0, hk, last]), dv_ref[0, 0], f"chunked dV last key tiles (kv head {hk})")
    del dq, dk, dv
    # GQA property at full size: dK/dV equal repeated-KV MHA gradients summed per group
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=True)
    kr, vr = k.repeat_interleave(g, dim=1).contiguous(), v.repeat_interleave(g, dim=1).contiguous()
    o_r, l_r = api.attn_fwd(q, kr, vr, causal=True)
    dq_r, dk_r, dv_r = api.attn_bwd(q, kr, vr, o_r, l_r, do, causal=True)
    torch.cuda.synchronize()
    dk_sum = dk_r.float().view(w.B, w.Hkv, g, w.N, w.d).sum(2)
    dv_sum = dv_r.float().view(w.B, w.Hkv, g, w.N, w.d).sum(2)
    for got, want, name in ((dk, dk_sum, "dK"), (dv, dv_sum, "dV")):
        err = float((got.float() - want).abs().max() / want.abs().max())
        assert err <= 3e-2, f"GQA {name} vs summed MHA: {err:.3e}"
    assert max_err(f64(dq_r), f64(dq)) / float(dq.float().abs().max()) <= 3e-2

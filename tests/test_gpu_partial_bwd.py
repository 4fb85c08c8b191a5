"""Chunked backward pass on the GPU: attn_bwd_preprocess once per query chunk
with the merged O and LSE, then attn_partial_bwd for every (query chunk, key
chunk) pair adding into float32 dQ, dK, dV.  Checked against the fp64 oracle
(its whole-sequence gradient, and its per-pair terms), with chunk sizes that
are not multiples of the 128-row tile so that the position offset between a
pair's queries and keys cuts through tiles, for causal, sliding-window,
non-causal and block-sparse masks and GQA."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api
from _gpu_helpers import assert_grad, f64, make, mask_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def run_pairs(q, k, v, o, lse, do, bounds, pairs, causal=False, window=None, bm=None, streams=1):
    """Chunk edges `bounds` (row starts, then N); every pair in `pairs` adds
    into zeroed float32 gradients."""
    dq = torch.zeros(q.shape, device="cuda", dtype=torch.float32)
    dk = torch.zeros(k.shape, device="cuda", dtype=torch.float32)
    dv = torch.zeros(v.shape, device="cuda", dtype=torch.float32)
    sl = [slice(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    ws = {c: api.attn_bwd_preprocess(o[:, :, sl[c]], lse[:, :, sl[c]], do[:, :, sl[c]]) for c in range(len(sl))}
    side = [torch.cuda.Stream() for _ in range(streams)] if streams > 1 else None
    if side:
        ev = torch.cuda.Event()
        ev.record()
        for s in side:
            s.wait_event(ev)
    for i, (qc, kc) in enumerate(pairs):
        pbm = None
        if bm is not None:   # the pair's own tiles of the block mask
            pbm = bm[bounds[qc] // 128:(bounds[qc + 1] + 127) // 128, bounds[kc] // 128:(bounds[kc + 1] + 127) // 128]
            pbm = torch.as_tensor(np.ascontiguousarray(pbm), dtype=torch.uint8).cuda()
        ctx = torch.cuda.stream(side[i % streams]) if side else torch.cuda.stream(torch.cuda.current_stream())
        with ctx:
            api.attn_partial_bwd(q[:, :, sl[qc]], k[:, :, sl[kc]], v[:, :, sl[kc]], do[:, :, sl[qc]], ws[qc],
                                 dq[:, :, sl[qc]], dk[:, :, sl[kc]], dv[:, :, sl[kc]], bounds[qc], bounds[kc],
                                 causal=causal, window=window, block_mask=pbm)
    if side:
        for s in side:
            torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return dq, dk, dv


CASES = [
    # B, Hq, Hkv, N, d, mask, chunk edges
    (1, 4, 2, 700, 128, "causal", [0, 256, 556, 700]),
    (2, 2, 2, 600, 64, "causal", [0, 200, 450, 600]),
    (1, 2, 1, 520, 128, "none", [0, 300, 520]),
    (1, 4, 4, 640, 64, "sliding_window", [0, 130, 390, 640]),
    (1, 2, 2, 512, 128, "block_sparse", [0, 256, 512]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[5]}-d{c[4]}-N{c[3]}" for c in CASES])
def test_chunked_backward_matches_oracle(case):
    B, Hq, Hkv, N, d, kind, bounds = case
    q, k, v, do = make(B, Hq, Hkv, N, d)
    scale = 1.0 / math.sqrt(d)
    window = 150 if kind == "sliding_window" else None
    bm = None
    if kind == "block_sparse":
        rng = np.random.default_rng(5)
        bm = rng.random((4, 4)) < 0.5
        bm[np.arange(4), np.arange(4)] = True
    causal = kind == "causal"
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    o, lse = api.attn_fwd(q, k, v, causal=causal, window=window, block_mask=bmt)
    n = len(bounds) - 1
    local = kind in ("causal", "sliding_window")
    pairs = [(a, b) for a in range(n) for b in range(n) if not local or b <= a]
    dq, dk, dv = run_pairs(q, k, v, o, lse, do, bounds, pairs, causal, window, bm)
    mask = mask_spec(kind, bm, window=window or 0)
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), scale, mask)
    for name, got, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        assert_grad(f64(got), want, f"chunked {name} {kind}")
    # the monolithic backward gives the same gradients
    ref = api.attn_bwd(q, k, v, o, lse, do, causal=causal, window=window, block_mask=bmt)
    torch.cuda.synchronize()
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(got), f64(want), f"chunked vs monolithic {name} {kind}")


def test_partial_backward_single_pair_against_oracle_terms():
    """One off-diagonal pair with offsets that cut tiles (query chunk at 300,
    key chunk at 90), its terms stored (accumulate off), against the oracle's
    per-pair terms computed with the oracle's own merged LSE and D."""
    B, Hq, Hkv, N, d = 1, 2, 1, 560, 128
    q, k, v, do = make(B, Hq, Hkv, N, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = api.attn_fwd(q, k, v, causal=True)
    qs, ks = slice(300, 560), slice(90, 410)
    ws = api.attn_bwd_preprocess(o[:, :, qs], lse[:, :, qs], do[:, :, qs])
    dq = torch.full((B, Hq, 260, d), 7.0, device="cuda")       # stored over: no stale values survive
    dk = torch.full((B, Hkv, 320, d), 7.0, device="cuda")
    dv = torch.full((B, Hkv, 320, d), 7.0, device="cuda")
    api.attn_partial_bwd(q[:, :, qs].contiguous(), k[:, :, ks].contiguous(), v[:, :, ks].contiguous(),
                         do[:, :, qs].contiguous(), ws, dq, dk, dv, 300, 90, causal=True, accumulate=False)
    torch.cuda.synchronize()
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    o_ref, l_ref = oracle.attention_forward(qf, kf, vf, scale, oracle.MaskSpec("causal"))
    dsum = (dof * o_ref).sum(-1)
    gq, gk, gv = oracle.partial_backward(qf[:, :, qs], kf[:, :, ks], vf[:, :, ks], dof[:, :, qs],
                                         l_ref[:, :, qs], dsum[:, :, qs], scale, oracle.MaskSpec("causal"), 300, 90)
    for name, got, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        assert_grad(f64(got), want, f"pair term {name}")


def test_pair_that_sees_nothing_adds_nothing_and_stores_zeros():
    B, Hq, Hkv, N, d = 1, 2, 2, 256, 64
    q, k, v, do = make(B, Hq, Hkv, N, d)
    o, lse = api.attn_fwd(q, k, v, causal=True)
    ws = api.attn_bwd_preprocess(o[:, :, :128], lse[:, :, :128], do[:, :, :128])
    # queries 0..127 against keys 128..255: all in the future
    dq = torch.full((B, Hq, 128, d), 3.0, device="cuda")
    dk = torch.full((B, Hkv, 128, d), 3.0, device="cuda")
    dv = torch.full((B, Hkv, 128, d), 3.0, device="cuda")
    qc, kc, vc, dc = (t.contiguous() for t in (q[:, :, :128], k[:, :, 128:], v[:, :, 128:], do[:, :, :128]))
    args = (qc, kc, vc, dc, ws, dq, dk, dv, 0, 128)
    api.attn_partial_bwd(*args, causal=True, accumulate=True)
    torch.cuda.synchronize()
    assert bool((dq == 3.0).all()) and bool((dk == 3.0).all()) and bool((dv == 3.0).all())
    api.attn_partial_bwd(*args, causal=True, accumulate=False)
    torch.cuda.synchronize()
    assert bool((dq == 0).all()) and bool((dk == 0).all()) and bool((dv == 0).all())


def test_chunked_backward_on_several_streams_matches_one_stream():
    """Pairs dealt to three streams at once (their float32 reductions overlap
    on shared outputs) give the one-stream gradients up to summation order."""
    B, Hq, Hkv, N, d = 1, 8, 2, 1024, 128
    q, k, v, do = make(B, Hq, Hkv, N, d)
    o, lse = api.chunked_fwd(q, k, v, 4)
    one = api.chunked_bwd(q, k, v, o, lse, do, 4)
    three = api.chunked_bwd(q, k, v, o, lse, do, 4, n_streams=3)
    torch.cuda.synchronize()
    for a, b in zip(one, three):
        assert float((a - b).abs().max()) <= 1e-5 * float(a.abs().max()) + 1e-6


def test_chunked_forward_backward_helpers_match_monolithic():
    B, Hq, Hkv, N, d = 1, 4, 1, 1024, 64
    q, k, v, do = make(B, Hq, Hkv, N, d)
    o, lse = api.chunked_fwd(q, k, v, 4)
    o_m, l_m = api.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = api.chunked_bwd(q, k, v, o, lse, do, 4, n_streams=2)
    ref = api.attn_bwd(q, k, v, o_m, l_m, do, causal=True)
    torch.cuda.synchronize()
    assert float((o.float() - o_m.float()).abs().max()) <= 1e-2
    assert float((lse - l_m).abs().max()) <= 2e-3
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(got), f64(want), f"helpers {name}")


def test_preprocess_writes_the_statistics_operand():
    """The workspace of attn_bwd_preprocess: D (rowsum(dO * O), checked against
    the oracle's forward output) and LSE * log2 e as float32, then per padded
    row 16 bf16 values [l l l, l l l, l l l, e e e, 0 0 0 0] (l = -LSE log2 e,
    e = -D, each a three-term split) in 128-row blocks of two 16-byte planes;
    the three terms sum to the float32 value to 2^-20 relative and padding rows
    hold -2^100 and 0."""
    B, Hq, Nq, d = 1, 2, 200, 64
    q, k, v, do = make(B, Hq, Hq, Nq, d)
    o, lse = api.attn_fwd(q, k, v, causal=True)
    ws = api.attn_bwd_preprocess(o, lse, do)
    torch.cuda.synchronize()
    Np = 256
    rows = B * Hq * Np
    arr = (rows * 4 + 255) // 256 * 256
    raw = ws.cpu()
    dsum = raw[:rows * 4].view(torch.float32).double().numpy()
    lse2 = raw[arr:arr + rows * 4].view(torch.float32).double().numpy()
    qx = raw[2 * arr:2 * arr + rows * 32].view(torch.bfloat16).double().numpy().reshape(rows // 128, 2, 128, 8)
    qx = np.concatenate([qx[:, 0], qx[:, 1]], axis=-1).reshape(rows, 16)   # row-major [row][16]
    valid = np.zeros(rows, bool)
    for h in range(B * Hq):
        valid[h * Np:h * Np + Nq] = True
    # D against the oracle's O and the same dO
    of, _ = oracle.attention_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), mask_spec("causal"))
    d_ref = (of * f64(do)).sum(-1).reshape(-1)
    np.testing.assert_allclose(dsum[valid], d_ref, rtol=2e-2, atol=2e-2)
    np.testing.assert_allclose(lse2[valid], lse.cpu().double().numpy().reshape(-1) * math.log2(math.e), rtol=1e-6)
    assert np.all(dsum[~valid] == 0) and np.all(np.isposinf(lse2[~valid]))
    l3 = qx[:, 0:3].sum(1)
    for rep in (3, 6):   # the lse2 triple three times
        assert np.array_equal(qx[:, rep:rep + 3], qx[:, 0:3])
    e3 = qx[:, 9:12].sum(1)
    assert np.all(qx[:, 12:] == 0)
    np.testing.assert_allclose(l3[valid], -lse2[valid], rtol=2 ** -20, atol=0)
    np.testing.assert_allclose(e3[valid], -dsum[valid], rtol=2 ** -20, atol=1e-30)
    assert np.all(l3[~valid] == -2.0 ** 100) and np.all(e3[~valid] == 0)

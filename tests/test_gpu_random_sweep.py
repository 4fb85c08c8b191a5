"""Seeded random sweep of GPU parity: configurations drawn from a fixed seed
(batch, query and key/value heads, sequence lengths around tile edges, head
size, mask kind, window, block mask density, chunk offsets) so that
combinations the hand-written cases miss are exercised, each checked against
the fp64 oracle at the problem statement's tolerances.  Sizes stay small
enough for the oracle to run every case in well under a second."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_grad, assert_o_lse, f64, make, mask_spec

pytestmark = pytest.mark.gpu

SWEEP_SEED = 20261202


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def draw(i):
    rng = np.random.default_rng(SWEEP_SEED + i)
    hkv = int(rng.choice([1, 2, 3]))
    g = int(rng.choice([1, 2, 4]))
    n = int(rng.choice([1, 7, 127, 128, 129, 255, 256, 300, 383, 511, 640]))
    return dict(B=int(rng.choice([1, 2])), Hkv=hkv, Hq=hkv * g, N=n, d=int(rng.choice([64, 128])),
                kind=str(rng.choice(["none", "causal", "sliding_window", "block_sparse"])),
                window=int(rng.choice([1, 50, 128, 200, 1000])), density=float(rng.choice([0.2, 0.5, 1.0])),
                cib=bool(rng.integers(0, 2)), seed=int(rng.integers(0, 1 << 30)))


def block_mask(c, nb):
    rng = np.random.default_rng(c["seed"])
    bm = rng.random((nb, nb)) < c["density"]
    bm[np.arange(nb), np.arange(nb)] = True
    return bm


@pytest.mark.parametrize("i", range(24))
def test_forward_backward_random(i):
    c = draw(i)
    B, Hq, Hkv, N, d = c["B"], c["Hq"], c["Hkv"], c["N"], c["d"]
    q, k, v, do = make(B, Hq, Hkv, N, d, seed=c["seed"])
    scale = 1.0 / math.sqrt(d)
    bm = block_mask(c, -(-N // 128)) if c["kind"] == "block_sparse" else None
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    window = c["window"] if c["kind"] == "sliding_window" else None
    cib = c["cib"] and bm is not None
    o, lse = api.attn_fwd(q, k, v, causal=c["kind"] == "causal", block_mask=bmt, causal_in_blocks=cib,
                          window=window)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=c["kind"] == "causal", block_mask=bmt,
                              causal_in_blocks=cib, window=window)
    torch.cuda.synchronize()
    mask = mask_spec(c["kind"], bm, cib, window or 0)
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    o_ref, l_ref = oracle.attention_forward(qf, kf, vf, scale, mask)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"case {i} {c}")
    gq, gk, gv = oracle.attention_backward(qf, kf, vf, dof, scale, mask)
    for name, got, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        assert_grad(f64(got), want, f"{name} case {i} {c}")


@pytest.mark.parametrize("i", range(12))
def test_chunk_pair_random(i):
    """One (query chunk, key chunk) pair at random global offsets: the partial
    forward against the oracle at those offsets, and the pair's backward
    terms (merged LSE and D from the oracle's own forward over the whole
    sequence) against the oracle's pair terms."""
    c = draw(100 + i)
    rng = np.random.default_rng(SWEEP_SEED + 1000 + i)
    B, Hq, Hkv, d = c["B"], c["Hq"], c["Hkv"], c["d"]
    N = max(c["N"], 260)
    q0 = int(rng.integers(0, N - 1))
    nq = int(rng.integers(1, N - q0 + 1))
    k0 = int(rng.integers(0, N - 1))
    nk = int(rng.integers(1, N - k0 + 1))
    q, k, v, do = make(B, Hq, Hkv, N, d, seed=c["seed"])
    scale = 1.0 / math.sqrt(d)
    kind = "sliding_window" if c["kind"] == "sliding_window" else ("none" if c["kind"] == "none" else "causal")
    window = c["window"] if kind == "sliding_window" else None
    mask = mask_spec(kind, window=window or 0)
    qs, ks = slice(q0, q0 + nq), slice(k0, k0 + nk)
    qc, kc, vc, doc = (t.contiguous() for t in (q[:, :, qs], k[:, :, ks], v[:, :, ks], do[:, :, qs]))
    o_c, l_c = api.attn_partial_fwd(qc, kc, vc, q0, k0, causal=kind == "causal", window=window)
    torch.cuda.synchronize()
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    o_ref, l_ref = oracle.attention_forward(qf[:, :, qs], kf[:, :, ks], vf[:, :, ks], scale, mask, q0, k0)
    assert_o_lse(f64(o_c), f64(l_c), o_ref, l_ref, f"partial fwd case {i} q0={q0} nq={nq} k0={k0} nk={nk}")
    # the pair's backward terms: the merged statistics over the whole sequence
    o_full, l_full = api.attn_fwd(q, k, v, causal=kind == "causal", window=window)
    ws = api.attn_bwd_preprocess(o_full[:, :, qs], l_full[:, :, qs], do[:, :, qs])
    dq = torch.zeros(qc.shape, device="cuda")
    dk = torch.zeros(kc.shape, device="cuda")
    dv = torch.zeros(vc.shape, device="cuda")
    api.attn_partial_bwd(qc, kc, vc, doc, ws, dq, dk, dv, q0, k0, causal=kind == "causal", window=window)
    torch.cuda.synchronize()
    of, lf = oracle.attention_forward(qf, kf, vf, scale, mask)
    dsum = (dof * of).sum(-1)
    gq, gk, gv = oracle.partial_backward(qf[:, :, qs], kf[:, :, ks], vf[:, :, ks], dof[:, :, qs], lf[:, :, qs],
                                         dsum[:, :, qs], scale, mask, q0, k0)
    for name, got, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        assert_grad(f64(got), want, f"pair {name} case {i} q0={q0} nq={nq} k0={k0} nk={nk}")


@pytest.mark.parametrize("i", range(8))
def test_ragged_batch_random(i):
    rng = np.random.default_rng(SWEEP_SEED + 2000 + i)
    nseq = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.choice([0, 1, 17, 128, 129, 200, 300, 513], nseq)]
    if sum(lens) == 0:
        lens[0] = 5
    hkv = int(rng.choice([1, 2]))
    Hq, d = hkv * int(rng.choice([1, 2])), int(rng.choice([64, 128]))
    kind = str(rng.choice(["none", "causal", "sliding_window"]))
    window = int(rng.choice([1, 60, 300])) if kind == "sliding_window" else None
    total = sum(lens)
    g = torch.Generator().manual_seed(int(rng.integers(0, 1 << 30)))
    q, k, v, do = (torch.randn(total, h, d, generator=g).to(torch.bfloat16).cuda() for h in (Hq, hkv, hkv, Hq))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
    causal = kind == "causal"
    o, lse = api.attn_varlen_fwd(q, k, v, cu, max(max(lens), 1), causal=causal, window=window)
    dq, dk, dv = api.attn_varlen_bwd(q, k, v, o, lse, do, cu, max(max(lens), 1), causal=causal, window=window)
    torch.cuda.synchronize()
    mask = mask_spec(kind, window=window or 0)
    cu_h = cu.cpu().numpy()
    o_ref, l_ref = oracle.varlen_forward(f64(q), f64(k), f64(v), cu_h, 1 / math.sqrt(d), mask)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"ragged {lens} {kind} {window}")
    gq, gk, gv = oracle.varlen_backward(f64(q), f64(k), f64(v), f64(do), cu_h, 1 / math.sqrt(d), mask)
    for name, got, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        assert_grad(f64(got), want, f"ragged {name} {lens} {kind} {window}")


@pytest.mark.parametrize("i", range(6))
def test_decode_random(i):
    rng = np.random.default_rng(SWEEP_SEED + 3000 + i)
    B, hkv = int(rng.integers(1, 4)), int(rng.choice([1, 2]))
    g = int(rng.choice([1, 4, 8]))
    nq = int(rng.choice([1, 2, 3]))
    nk = int(rng.choice([nq, 129, 700, 1500]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    q, k, v, _ = make(B, hkv * g, hkv, nq, d, seed=int(rng.integers(0, 1 << 30)), Nk=nk)
    lens = torch.tensor(rng.integers(nq, nk + 1, B), dtype=torch.int32)
    o, lse = api.attn_decode(q, k, v, lens.cuda(), causal=causal, n_splits=int(rng.choice([0, 1, 3])))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), lens.numpy(), causal)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"decode case {i}")

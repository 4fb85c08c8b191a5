"""Pins for the fp64 oracle: each check ties it to something other than itself.

Closed forms (Q = 0, constant V, one dominant logit, a single key), hand-worked
golden fixtures, central finite differences, a library softmax and PyTorch's
float64 scaled-dot-product attention with autograd, and invariants (chunked
merge == monolithic, GQA == repeated MHA, all-ones block mask == dense,
block-triangular + causal == causal, a window wider than the sequence ==
causal, a window of one == identity).  ``test_planted_mistakes`` shows that a
plausible slip in the oracle (a dropped term, a sign, an off-by-one, a
transposed operand, a missing merge weight, a wrong E4M3 exponent bias, a lost
scale factor) fails at least one pin.
"""
import glob
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import MaskSpec
from oracle import attention as oa

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(7)


def rnd(*shape, rng=None):
    return (rng or RNG).standard_normal(shape)


def masks_for(n, block=4, rng=None):
    rng = rng or np.random.default_rng(3)
    nb = -(-n // block)
    bm = rng.random((nb, nb)) < 0.5
    bm[np.arange(nb), np.arange(nb)] = True
    return [MaskSpec("none"), MaskSpec("causal"),
            MaskSpec("block_sparse", bm, block),
            MaskSpec("block_sparse", bm, block, causal_in_blocks=True)]


# ---------------------------------------------------------------- closed forms

def check_q_zero(fwd):
    for nq, nk, qo, ko in [(7, 7, 0, 0), (5, 9, 4, 0), (6, 6, 0, 2), (9, 5, 3, 3)]:
        for mask in masks_for(max(nq, nk)):
            if mask.kind == "block_sparse" and (qo or ko):
                continue
            q = np.zeros((1, 1, nq, 3))
            k = rnd(1, 1, nk, 3)
            v = rnd(1, 1, nk, 3)
            o, lse = fwd(q, k, v, 0.37, mask, qo, ko)
            for i in range(nq):
                vis = []
                for j in range(nk):
                    ok = True
                    if mask.kind == "causal" or mask.causal_in_blocks:
                        ok = ok and ko + j <= qo + i
                    if mask.kind == "block_sparse":
                        ok = ok and bool(mask.block_mask[i // mask.block, j // mask.block])
                    if ok:
                        vis.append(j)
                if not vis:
                    assert np.all(o[0, 0, i] == 0) and lse[0, 0, i] == -np.inf
                else:
                    np.testing.assert_allclose(o[0, 0, i], v[0, 0, vis].mean(axis=0), rtol=0, atol=1e-13)
                    assert abs(lse[0, 0, i] - np.log(len(vis))) < 1e-13


def test_q_zero_gives_mean_of_visible_rows():
    check_q_zero(oracle.attention_forward)


def test_constant_v_rows():
    q, k = rnd(1, 2, 9, 4), rnd(1, 1, 9, 4)
    vrow = rnd(4)
    v = np.broadcast_to(vrow, (1, 1, 9, 4)).copy()
    do = rnd(1, 2, 9, 4)
    for mask in masks_for(9):
        o, _ = oracle.attention_forward(q, k, v, 0.5, mask)
        np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), atol=1e-13)
        dq, dk, _ = oracle.attention_backward(q, k, v, do, 0.5, mask)
        assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_dominant_logit():
    n, d, i, js = 16, 8, 5, 11
    q, k, v = rnd(1, 1, n, d), rnd(1, 1, n, d), rnd(1, 1, n, d)
    scale = 0.35
    others = scale * (q[0, 0, i] @ np.delete(k[0, 0], js, axis=0).T)
    qq = q[0, 0, i] @ q[0, 0, i]
    alpha = (others.max() + 40.0) / (scale * qq)
    k[0, 0, js] = alpha * q[0, 0, i]
    o, lse = oracle.attention_forward(q, k, v, scale)
    assert np.abs(o[0, 0, i] - v[0, 0, js]).max() < 1e-15 * 1e2 + n * np.exp(-40.0) * np.abs(v).max()
    assert abs(lse[0, 0, i] - scale * alpha * qq) < 1e-12


def test_single_key():
    q, k, v = rnd(2, 3, 1, 8), rnd(2, 3, 1, 8), rnd(2, 3, 1, 8)
    o, lse = oracle.attention_forward(q, k, v, 0.125)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.125 * (q * k).sum(-1), atol=1e-14)


def test_lse_bounds_and_rows_sum_to_one():
    q, k, v = rnd(1, 2, 33, 8), rnd(1, 2, 33, 8), rnd(1, 2, 33, 8)
    for mask in masks_for(33):
        o, lse = oracle.attention_forward(q, k, v, 0.4, mask)
        # P rows sum to one: attention of a constant-one value column is one
        ones = np.ones((1, 2, 33, 1))
        o1, _ = oracle.attention_forward(q, k, ones, 0.4, mask)
        for h in range(2):
            vis = oracle.visible(np.arange(33), 33, mask)
            s = np.where(vis, 0.4 * q[0, h] @ k[0, h].T, -np.inf)
            smax = s.max(1)
            cnt = vis.sum(1)
            ok = cnt > 0
            assert np.all(lse[0, h, ok] >= smax[ok] - 1e-12)
            assert np.all(lse[0, h, ok] <= smax[ok] + np.log(cnt[ok]) + 1e-12)
            np.testing.assert_allclose(o1[0, h, ok, 0], 1.0, atol=1e-14)


# ---------------------------------------------------------------- golden files

def _mask_from(g, n):
    if g.get("mask", "none") == "block_sparse":
        return MaskSpec("block_sparse", np.array(g["block_mask"], bool), g["block"])
    return MaskSpec(g.get("mask", "none"))


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(HERE, "golden", "*.json"))),
                         ids=os.path.basename)
def test_golden(path):
    g = json.load(open(path))
    assert g["source"]
    if g.get("kind") == "chunk_schedule":
        for c in g["cases"]:
            got = oracle.chunk_pair_schedule(c["n_chunks"], c["n_lanes"])
            assert got == [tuple(p) for p in c["order"]], c
            loads = [sum(1 if q == k else 2 for q, k in lane)
                     for lane in oracle.chunk_pair_lanes(c["n_chunks"], c["n_lanes"])]
            assert loads == c["lane_loads"], c
        return
    if g.get("kind") == "fwd_units":
        for c in g["cases"]:
            got = oracle.fwd_work_units(c["mask"], c["B"], c["Hq"], c["N"], c["N"], Hkv=c["Hkv"], d=c["d"])
            assert got == [tuple(u) for u in c["units"]], c
        return
    if "o_parts" in g:
        o, lse = oracle.merge_partials([np.array(x) for x in g["o_parts"]],
                                       [np.array(x) for x in g["lse_parts"]])
        np.testing.assert_allclose(o, g["o"], atol=1e-12)
        np.testing.assert_allclose(lse, g["lse"], atol=1e-12)
        return
    q = np.array(g["q"])[None, None]
    k = np.array(g["k"])[None, None]
    v = np.array(g["v"])[None, None]
    mask = _mask_from(g, q.shape[2])
    o, lse = oracle.attention_forward(q, k, v, g["scale"], mask)
    np.testing.assert_allclose(o[0, 0], g["o"], atol=1e-12)
    if "lse" in g:
        np.testing.assert_allclose(lse[0, 0], g["lse"], atol=1e-12)
    if "dq" in g:
        do = np.array(g["do"])[None, None]
        dq, dk, dv = oracle.attention_backward(q, k, v, do, g["scale"], mask)
        np.testing.assert_allclose(dq[0, 0], g["dq"], atol=1e-12)
        np.testing.assert_allclose(dk[0, 0], g["dk"], atol=1e-12)
        np.testing.assert_allclose(dv[0, 0], g["dv"], atol=1e-12)


# ---------------------------------------------------------------- finite differences

def fd_check(fwd, bwd, mask, qo=0, ko=0, nq=6, nk=6, hq=2, hkv=1, d=3, seed=11):
    rng = np.random.default_rng(seed)
    q, k, v = rnd(1, hq, nq, d, rng=rng), rnd(1, hkv, nk, d, rng=rng), rnd(1, hkv, nk, d, rng=rng)
    do = rnd(1, hq, nq, d, rng=rng)
    scale = 0.6

    def loss(q_, k_, v_):
        o, _ = fwd(q_, k_, v_, scale, mask, qo, ko)
        return float((o * do).sum())

    dq, dk, dv = bwd(q, k, v, do, scale, mask, qo, ko)
    h = 1e-6
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = loss(q, k, v)
            x[idx] = old - h
            fm = loss(q, k, v)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        scale_ref = max(1.0, np.abs(num).max())
        err = np.abs(num - gx).max() / scale_ref
        assert err < 1e-7, (mask.kind, err)


@pytest.mark.parametrize("mi", range(4))
def test_finite_difference_gradients(mi):
    mask = masks_for(8, block=3)[mi]
    fd_check(oracle.attention_forward, oracle.attention_backward, mask, nq=8, nk=8)


def test_finite_difference_gradients_offsets():
    fd_check(oracle.attention_forward, oracle.attention_backward, MaskSpec("causal"),
             qo=5, ko=2, nq=5, nk=7)


# ---------------------------------------------------------------- library routines

def test_library_softmax_scipy():
    q, k, v = rnd(1, 2, 40, 8), rnd(1, 2, 40, 8), rnd(1, 2, 40, 8)
    for mask in masks_for(40, block=8):
        o, lse = oracle.attention_forward(q, k, v, 0.3, mask)
        for h in range(2):
            vis = np.zeros((40, 40), bool)
            for i in range(40):
                for j in range(40):
                    ok = True
                    if mask.kind == "causal" or mask.causal_in_blocks:
                        ok &= j <= i
                    if mask.kind == "block_sparse":
                        ok &= bool(mask.block_mask[i // 8, j // 8])
                    vis[i, j] = ok
            s = np.where(vis, 0.3 * np.einsum("id,jd->ij", q[0, h], k[0, h]), -np.inf)
            p = scipy.special.softmax(s, axis=1)
            np.testing.assert_allclose(o[0, h], p @ v[0, h], atol=1e-12)
            np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(s, axis=1), atol=1e-12)


def test_library_torch_sdpa_fwd_bwd():
    """PyTorch's float64 CPU scaled_dot_product_attention and its autograd agree."""
    F = torch.nn.functional
    for causal, hq, hkv in [(False, 4, 4), (True, 4, 4), (True, 4, 2), (False, 6, 2)]:
        q, k, v, do = rnd(2, hq, 24, 16), rnd(2, hkv, 24, 16), rnd(2, hkv, 24, 16), rnd(2, hq, 24, 16)
        mask = MaskSpec("causal" if causal else "none")
        o, _ = oracle.attention_forward(q, k, v, 0.25, mask)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.25, mask)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        g = hq // hkv
        to = F.scaled_dot_product_attention(tq, tk.repeat_interleave(g, 1), tv.repeat_interleave(g, 1),
                                            is_causal=causal, scale=0.25)
        to.backward(torch.tensor(do))
        np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


# ---------------------------------------------------------------- invariants

def test_chunked_merge_equals_monolithic():
    n, d = 48, 8
    q, k, v = rnd(1, 2, n, d), rnd(1, 1, n, d), rnd(1, 1, n, d)
    full_o, full_l = oracle.attention_forward(q, k, v, 0.3, MaskSpec("causal"))
    for nc in (1, 2, 3, 4, 6, 8, 12, 16, 24, 48):
        c = n // nc
        for qc in range(nc):
            qs = slice(qc * c, (qc + 1) * c)
            parts = []
            for kc in range(qc + 1):
                ks = slice(kc * c, (kc + 1) * c)
                parts.append(oracle.attention_forward(q[:, :, qs], k[:, :, ks], v[:, :, ks], 0.3,
                                                      MaskSpec("causal"), qc * c, kc * c))
            o, l = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
            np.testing.assert_allclose(o, full_o[:, :, qs], atol=1e-12)
            np.testing.assert_allclose(l, full_l[:, :, qs], atol=1e-12)


def test_merge_with_empty_parts():
    o1, l1 = rnd(3, 4), rnd(3)
    o, l = oracle.merge_partials([o1, rnd(3, 4)], [l1, np.full(3, -np.inf)])
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, l1, atol=1e-15)
    o, l = oracle.merge_partials([o1, o1], [np.full(3, -np.inf)] * 2)
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_gqa_equals_repeated_mha():
    q, k, v, do = rnd(2, 6, 10, 4), rnd(2, 2, 10, 4), rnd(2, 2, 10, 4), rnd(2, 6, 10, 4)
    for mask in masks_for(10):
        o, l = oracle.attention_forward(q, k, v, 0.5, mask)
        kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
        o2, l2 = oracle.attention_forward(q, kr, vr, 0.5, mask)
        np.testing.assert_allclose(o, o2, atol=1e-14)
        np.testing.assert_allclose(l, l2, atol=1e-14)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, mask)
        dq2, dk2, dv2 = oracle.attention_backward(q, kr, vr, do, 0.5, mask)
        np.testing.assert_allclose(dq, dq2, atol=1e-13)
        np.testing.assert_allclose(dk, dk2.reshape(2, 2, 3, 10, 4).sum(2), atol=1e-13)
        np.testing.assert_allclose(dv, dv2.reshape(2, 2, 3, 10, 4).sum(2), atol=1e-13)


def test_block_mask_special_cases():
    q, k, v, do = rnd(1, 2, 20, 4), rnd(1, 2, 20, 4), rnd(1, 2, 20, 4), rnd(1, 2, 20, 4)
    ones = MaskSpec("block_sparse", np.ones((5, 5), bool), 4)
    tri = MaskSpec("block_sparse", np.tril(np.ones((5, 5), bool)), 4, causal_in_blocks=True)
    for sparse, dense in ((ones, MaskSpec("none")), (tri, MaskSpec("causal"))):
        a = oracle.attention_forward(q, k, v, 0.5, sparse)
        b = oracle.attention_forward(q, k, v, 0.5, dense)
        np.testing.assert_allclose(a[0], b[0], atol=1e-14)
        np.testing.assert_allclose(a[1], b[1], atol=1e-14)
        ga = oracle.attention_backward(q, k, v, do, 0.5, sparse)
        gb = oracle.attention_backward(q, k, v, do, 0.5, dense)
        for x, y in zip(ga, gb):
            np.testing.assert_allclose(x, y, atol=1e-13)


def test_backward_identities():
    """rowsum(dO*O) equals rowsum(P*dP), and sum_j dS_ij = 0 (so dQ is unchanged
    when one vector is added to every key)."""
    q, k, v, do = rnd(1, 1, 12, 5), rnd(1, 1, 12, 5), rnd(1, 1, 12, 5), rnd(1, 1, 12, 5)
    for mask in masks_for(12):
        o, _ = oracle.attention_forward(q, k, v, 0.7, mask)
        vis = oracle.visible(np.arange(12), 12, mask)
        s = np.where(vis, 0.7 * q[0, 0] @ k[0, 0].T, -np.inf)
        p = scipy.special.softmax(s, axis=1)
        dp = do[0, 0] @ v[0, 0].T
        np.testing.assert_allclose((do * o).sum(-1)[0, 0], (p * dp).sum(1), atol=1e-13)
        dq, _, _ = oracle.attention_backward(q, k, v, do, 0.7, mask)
        dq2, _, _ = oracle.attention_backward(q, k + rnd(5), v, do, 0.7, mask)
        np.testing.assert_allclose(dq, dq2, atol=1e-12)


def test_sampled_rows_match_full():
    q, k, v, do = rnd(2, 4, 30, 8), rnd(2, 2, 30, 8), rnd(2, 2, 30, 8), rnd(2, 4, 30, 8)
    mask = MaskSpec("causal")
    o, l = oracle.attention_forward(q, k, v, 0.3, mask)
    rows = np.array([0, 7, 29])
    os_, ls_ = oracle.attention_forward(q, k, v, 0.3, mask, heads=[(1, 3), (0, 0)], rows=rows)
    np.testing.assert_allclose(os_[0], o[1, 3, rows], atol=0)
    np.testing.assert_allclose(ls_[1], l[0, 0, rows], atol=0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.3, mask)
    dqs = oracle.attention_backward_dq_rows(q, k, v, do, 0.3, 1, 3, rows, mask)
    np.testing.assert_allclose(dqs, dq[1, 3, rows], atol=1e-14)
    dqg, dks, dvs = oracle.attention_backward(q, k, v, do, 0.3, mask, kv_heads=[(1, 1)])
    np.testing.assert_allclose(dks[0], dk[1, 1], atol=1e-14)
    np.testing.assert_allclose(dvs[0], dv[1, 1], atol=1e-14)
    np.testing.assert_allclose(dqg[0], dq[1, 2:4], atol=1e-14)


# ---------------------------------------------------------------- sliding window

def _window_visible_loops(nq, nk, w, qo=0, ko=0):
    """Visibility written out element by element: key j lies 0..w-1 positions
    behind query i (global positions)."""
    vis = np.zeros((nq, nk), bool)
    for i in range(nq):
        for j in range(nk):
            back = (qo + i) - (ko + j)
            vis[i, j] = 0 <= back < w
    return vis


def test_sliding_window_q_zero_gives_mean_of_window():
    for nq, nk, qo, ko, w in [(9, 9, 0, 0, 1), (9, 9, 0, 0, 3), (7, 11, 4, 0, 5), (8, 6, 0, 3, 2), (6, 9, 9, 1, 4)]:
        q = np.zeros((1, 1, nq, 3))
        k, v = rnd(1, 1, nk, 3), rnd(1, 1, nk, 3)
        o, lse = oracle.attention_forward(q, k, v, 0.4, MaskSpec("sliding_window", window=w), qo, ko)
        vis = _window_visible_loops(nq, nk, w, qo, ko)
        for i in range(nq):
            js = np.flatnonzero(vis[i])
            if js.size == 0:
                assert np.all(o[0, 0, i] == 0) and lse[0, 0, i] == -np.inf
            else:
                np.testing.assert_allclose(o[0, 0, i], v[0, 0, js].mean(axis=0), rtol=0, atol=1e-13)
                assert abs(lse[0, 0, i] - np.log(js.size)) < 1e-13


def test_sliding_window_of_one_is_identity():
    q, k, v = rnd(2, 3, 10, 8), rnd(2, 3, 10, 8), rnd(2, 3, 10, 8)
    o, lse = oracle.attention_forward(q, k, v, 0.3, MaskSpec("sliding_window", window=1))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * (q * k).sum(-1), atol=1e-14)


def test_wide_sliding_window_equals_causal():
    q, k, v, do = rnd(1, 4, 13, 5), rnd(1, 2, 13, 5), rnd(1, 2, 13, 5), rnd(1, 4, 13, 5)
    for w in (13, 14, 100):
        a = oracle.attention_forward(q, k, v, 0.5, MaskSpec("sliding_window", window=w))
        b = oracle.attention_forward(q, k, v, 0.5, MaskSpec("causal"))
        np.testing.assert_allclose(a[0], b[0], atol=1e-15)
        np.testing.assert_allclose(a[1], b[1], atol=1e-15)
        for x, y in zip(oracle.attention_backward(q, k, v, do, 0.5, MaskSpec("sliding_window", window=w)),
                        oracle.attention_backward(q, k, v, do, 0.5, MaskSpec("causal"))):
            np.testing.assert_allclose(x, y, atol=1e-14)


def test_sliding_window_torch_sdpa_with_explicit_mask():
    """PyTorch's float64 attention with the boolean mask written out by loops."""
    F = torch.nn.functional
    for nq, w, hq, hkv in [(20, 1, 2, 2), (20, 5, 4, 2), (24, 7, 2, 1), (17, 30, 2, 2)]:
        q, k, v, do = rnd(1, hq, nq, 8), rnd(1, hkv, nq, 8), rnd(1, hkv, nq, 8), rnd(1, hq, nq, 8)
        mask = MaskSpec("sliding_window", window=w)
        o, _ = oracle.attention_forward(q, k, v, 0.35, mask)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.35, mask)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        g = hq // hkv
        am = torch.tensor(_window_visible_loops(nq, nq, w))
        to = F.scaled_dot_product_attention(tq, tk.repeat_interleave(g, 1), tv.repeat_interleave(g, 1),
                                            attn_mask=am, scale=0.35)
        to.backward(torch.tensor(do))
        np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("w,qo,ko", [(1, 0, 0), (3, 0, 0), (4, 5, 2), (9, 0, 0)])
def test_finite_difference_gradients_sliding_window(w, qo, ko):
    fd_check(oracle.attention_forward, oracle.attention_backward, MaskSpec("sliding_window", window=w),
             qo=qo, ko=ko, nq=7, nk=8)


def test_sliding_window_chunked_merge_equals_monolithic():
    n, d, w = 48, 8, 11
    mask = MaskSpec("sliding_window", window=w)
    q, k, v = rnd(1, 2, n, d), rnd(1, 1, n, d), rnd(1, 1, n, d)
    full_o, full_l = oracle.attention_forward(q, k, v, 0.3, mask)
    for nc in (2, 3, 4, 6, 8, 16):
        c = n // nc
        for qc in range(nc):
            qs = slice(qc * c, (qc + 1) * c)
            parts = [oracle.attention_forward(q[:, :, qs], k[:, :, kc * c:(kc + 1) * c], v[:, :, kc * c:(kc + 1) * c],
                                              0.3, mask, qc * c, kc * c) for kc in range(qc + 1)]
            o, l = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
            np.testing.assert_allclose(o, full_o[:, :, qs], atol=1e-12)
            np.testing.assert_allclose(l, full_l[:, :, qs], atol=1e-12)


# ---------------------------------------------------------------- chunked backward

def chunked_backward(q, k, v, do, scale, mask, nc, bm=None, block=4):
    """Gradient of the whole sequence assembled from oracle.partial_backward
    over every (query chunk, key chunk) pair, with the merged LSE and
    D = rowsum(dO * O) of the whole forward pass."""
    n = q.shape[2]
    c = n // nc
    o, lse = oracle.attention_forward(q, k, v, scale, mask)
    dsum = (do * o).sum(-1)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for qc in range(nc):
        qs = slice(qc * c, (qc + 1) * c)
        for kc in range(nc):
            ks = slice(kc * c, (kc + 1) * c)
            m = mask
            if mask.kind == "block_sparse":   # the pair's own tiles of the block mask
                m = MaskSpec("block_sparse", bm[qc * c // block:(qc + 1) * c // block,
                                                kc * c // block:(kc + 1) * c // block], block,
                             mask.causal_in_blocks)
            a, bk, bv = oracle.partial_backward(q[:, :, qs], k[:, :, ks], v[:, :, ks], do[:, :, qs],
                                                lse[:, :, qs], dsum[:, :, qs], scale, m, qc * c, kc * c)
            dq[:, :, qs] += a
            dk[:, :, ks] += bk
            dv[:, :, ks] += bv
    return dq, dk, dv


def test_chunked_backward_equals_monolithic():
    """Summed over every chunk pair, the chunk terms give the gradient of the
    whole sequence (itself pinned by finite differences and torch autograd),
    for every mask kind, GQA, and chunk counts down to one row per chunk."""
    n, d = 24, 4
    rng = np.random.default_rng(11)
    q, k, v, do = rnd(2, 4, n, d, rng=rng), rnd(2, 2, n, d, rng=rng), rnd(2, 2, n, d, rng=rng), \
        rnd(2, 4, n, d, rng=rng)
    bm = rng.random((6, 6)) < 0.5
    bm[np.arange(6), np.arange(6)] = True
    masks = [MaskSpec("none"), MaskSpec("causal"), MaskSpec("sliding_window", window=5),
             MaskSpec("block_sparse", bm, 4), MaskSpec("block_sparse", bm, 4, causal_in_blocks=True)]
    for mask in masks:
        want = oracle.attention_backward(q, k, v, do, 0.45, mask)
        for nc in (1, 2, 3, 6) if mask.kind == "block_sparse" else (1, 2, 3, 4, 6, 8, 24):
            got = chunked_backward(q, k, v, do, 0.45, mask, nc, bm)
            for x, y in zip(got, want):
                np.testing.assert_allclose(x, y, atol=1e-12, err_msg=f"{mask.kind} nc={nc}")


def test_partial_backward_of_an_invisible_chunk_is_zero():
    """A key chunk entirely after the query chunk (causal) contributes nothing,
    and a row with LSE = -inf (it sees no key anywhere) has zero terms."""
    q, k, v, do = rnd(1, 2, 6, 3), rnd(1, 1, 6, 3), rnd(1, 1, 6, 3), rnd(1, 2, 6, 3)
    lse, dsum = rnd(1, 2, 6), rnd(1, 2, 6)
    for x in oracle.partial_backward(q, k, v, do, lse, dsum, 0.5, MaskSpec("causal"), 0, 6):
        assert np.all(x == 0)
    lse[0, 1] = -np.inf
    dq, dk, dv = oracle.partial_backward(q, k, v, do, lse, dsum, 0.5, MaskSpec("none"))
    assert np.all(dq[0, 1] == 0)
    dq0, dk0, dv0 = oracle.partial_backward(q[:, :1], k, v, do[:, :1], lse[:, :1], dsum[:, :1], 0.5,
                                            MaskSpec("none"))
    np.testing.assert_allclose(dk, dk0, atol=1e-14)
    np.testing.assert_allclose(dv, dv0, atol=1e-14)


# ---------------------------------------------------------------- decoding against a KV cache

def test_decode_equals_last_rows_of_causal_attention():
    """The newest Nq positions attending to the cache give the last Nq rows of
    causal attention over the whole sequence (the pinned forward)."""
    B, Hq, Hkv, N, d = 3, 4, 2, 20, 6
    lens = [20, 13, 5]
    for nq in (1, 3):
        q_all, k, v = rnd(B, Hq, N, d), rnd(B, Hkv, N, d), rnd(B, Hkv, N, d)
        q = np.stack([q_all[b, :, lens[b] - nq:lens[b]] for b in range(B)])
        o, lse = oracle.decode_forward(q, k, v, 0.4, lens, causal=True)
        for b in range(B):
            n = lens[b]
            of, lf = oracle.attention_forward(q_all[b:b + 1, :, :n], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.4,
                                              MaskSpec("causal"))
            np.testing.assert_allclose(o[b], of[0, :, n - nq:], atol=1e-14)
            np.testing.assert_allclose(lse[b], lf[0, :, n - nq:], atol=1e-14)


def test_decode_q_zero_gives_mean_of_cached_values():
    B, Hq, Hkv, Nk, d, nq = 2, 4, 1, 9, 3, 2
    lens = [9, 4]
    k, v = rnd(B, Hkv, Nk, d), rnd(B, Hkv, Nk, d)
    q = np.zeros((B, Hq, nq, d))
    for causal in (False, True):
        o, lse = oracle.decode_forward(q, k, v, 0.5, lens, causal)
        for b in range(B):
            for i in range(nq):
                top = lens[b] - nq + i + 1 if causal else lens[b]     # keys 0..top-1 are visible
                for h in range(Hq):
                    np.testing.assert_allclose(o[b, h, i], v[b, 0, :top].mean(axis=0), atol=1e-14)
                    assert abs(lse[b, h, i] - np.log(top)) < 1e-13


def test_decode_empty_sequence():
    q, k, v = rnd(2, 2, 1, 4), rnd(2, 2, 5, 4), rnd(2, 2, 5, 4)
    o, lse = oracle.decode_forward(q, k, v, 0.5, [0, 5])
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(lse[1]))


# ---------------------------------------------------------------- ragged (packed) batches

def test_varlen_equal_lengths_equal_batched_forward():
    B, Hq, Hkv, n, d = 3, 4, 2, 11, 5
    q, k, v = rnd(B, Hq, n, d), rnd(B, Hkv, n, d), rnd(B, Hkv, n, d)
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * n, x.shape[1], d)
    cu = [0, n, 2 * n, 3 * n]
    for mask in (MaskSpec("none"), MaskSpec("causal"), MaskSpec("sliding_window", window=4)):
        o, lse = oracle.varlen_forward(pack(q), pack(k), pack(v), cu, 0.45, mask)
        ob, lb = oracle.attention_forward(q, k, v, 0.45, mask)
        np.testing.assert_allclose(o, pack(ob), atol=1e-15)
        np.testing.assert_allclose(lse, lb.transpose(1, 0, 2).reshape(Hq, B * n), atol=1e-15)


def test_varlen_q_zero_sees_only_its_own_sequence():
    lens = [5, 1, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    k, v = rnd(total, 2, 3), rnd(total, 2, 3)
    q = np.zeros((total, 4, 3))
    for causal in (False, True):
        o, lse = oracle.varlen_forward(q, k, v, cu, 0.7, MaskSpec("causal" if causal else "none"))
        for b, n in enumerate(lens):
            for i in range(n):
                t = cu[b] + i
                top = i + 1 if causal else n                 # keys cu[b] .. cu[b] + top - 1 are visible
                for h in range(4):
                    np.testing.assert_allclose(o[t, h], v[cu[b]:cu[b] + top, h // 2].mean(axis=0), atol=1e-14)
                    assert abs(lse[h, t] - np.log(top)) < 1e-13


def test_varlen_backward_equal_lengths_and_finite_differences():
    B, Hq, Hkv, n, d = 2, 4, 2, 7, 3
    q, k, v, do = rnd(B, Hq, n, d), rnd(B, Hkv, n, d), rnd(B, Hkv, n, d), rnd(B, Hq, n, d)
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * n, x.shape[1], d)
    cu = [0, n, 2 * n]
    for mask in (MaskSpec("causal"), MaskSpec("sliding_window", window=3)):
        got = oracle.varlen_backward(pack(q), pack(k), pack(v), pack(do), cu, 0.5, mask)
        want = oracle.attention_backward(q, k, v, do, 0.5, mask)
        for a, b in zip(got, want):
            np.testing.assert_allclose(a, pack(b), atol=1e-14)
    # ragged: central differences of <O, dO> through varlen_forward
    lens = [3, 1, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    rng = np.random.default_rng(5)
    qq, kk, vv, dd = (rng.standard_normal((8, h, 3)) for h in (2, 1, 1, 2))
    mask = MaskSpec("causal")
    gq, gk, gv = oracle.varlen_backward(qq, kk, vv, dd, cu, 0.6, mask)
    h = 1e-6
    for x, gx in ((qq, gq), (kk, gk), (vv, gv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = float((oracle.varlen_forward(qq, kk, vv, cu, 0.6, mask)[0] * dd).sum())
            x[idx] = old - h
            fm = float((oracle.varlen_forward(qq, kk, vv, cu, 0.6, mask)[0] * dd).sum())
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.abs(num - gx).max() / max(1.0, np.abs(num).max()) < 1e-7


# ---------------------------------------------------------------- e4m3 operands

def test_e4m3_decode_matches_torch_float8():
    """All 256 codes against torch's own float8_e4m3fn -> float64 conversion."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_closed_forms():
    d = oracle.e4m3_decode
    assert d(0x38) == 1.0 and d(0xB8) == -1.0 and d(0x40) == 2.0 and d(0x3C) == 1.5
    assert d(0x7E) == 448.0 == oracle.E4M3_MAX
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9 and d(0x08) == 2.0 ** -6
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert np.nanmax(d(np.arange(256, dtype=np.uint8))) == 448.0


def _codes(*shape, rng, lo=-60.0, hi=60.0):
    x = torch.from_numpy(rng.uniform(lo, hi, shape).astype(np.float32))
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_forward_descale_invariances():
    """Only the product of the Q and K factors matters; O is linear in the V
    factor and the LSE does not see it."""
    rng = np.random.default_rng(11)
    q8, k8, v8 = _codes(1, 2, 9, 4, rng=rng), _codes(1, 1, 9, 4, rng=rng), _codes(1, 1, 9, 4, rng=rng)
    for mask in (MaskSpec("none"), MaskSpec("causal"), MaskSpec("sliding_window", window=3)):
        o1, l1 = oracle.fp8_forward(q8, k8, v8, 0.02, 0.015, 0.1, 0.5, mask)
        o2, l2 = oracle.fp8_forward(q8, k8, v8, 0.04, 0.0075, 0.1, 0.5, mask)
        o3, l3 = oracle.fp8_forward(q8, k8, v8, 0.02, 0.015, 0.3, 0.5, mask)
        np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o3, 3.0 * o1, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l3, l1, rtol=1e-12, atol=1e-14)


def test_fp8_forward_q_zero_gives_mean_of_visible_values():
    rng = np.random.default_rng(12)
    q8 = np.zeros((1, 1, 6, 4), np.uint8)
    k8, v8 = _codes(1, 1, 6, 4, rng=rng), _codes(1, 1, 6, 4, rng=rng)
    vv = 0.25 * oracle.e4m3_decode(v8)[0, 0]
    o, lse = oracle.fp8_forward(q8, k8, v8, 1.0, 1.0, 0.25, 0.7, MaskSpec("causal"))
    for i in range(6):
        np.testing.assert_allclose(o[0, 0, i], vv[:i + 1].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - np.log(i + 1)) < 1e-13


def _simulated_rounding_error(q8, k8, v8, qd, kd, vd, scale, t):
    """O_sim - O_exact per element ([rows, d]) for one head: O_sim from the
    weights w * 2^t rounded to E4M3 by torch (round to nearest), normalised by
    the exact sum of the unrounded weights."""
    q = qd * oracle.e4m3_decode(q8)[0, 0]
    k = kd * oracle.e4m3_decode(k8)[0, 0]
    v = vd * oracle.e4m3_decode(v8)[0, 0]
    s = scale * q @ k.T
    w = np.exp(s - s.max(axis=1, keepdims=True))
    p = torch.from_numpy(w * 2.0 ** t).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    o_sim = (p @ v) / (w * 2.0 ** t).sum(axis=1, keepdims=True)
    o_ex = (w @ v) / w.sum(axis=1, keepdims=True)
    return o_sim - o_ex


def test_fp8_error_bound_holds_for_simulated_rounding():
    rng = np.random.default_rng(13)
    for n, krange in ((40, 60.0), (300, 200.0)):
        q8, k8, v8 = _codes(1, 1, n, 8, rng=rng), _codes(1, 1, n, 8, rng=rng, lo=-krange, hi=krange), \
            _codes(1, 1, n, 8, rng=rng)
        bound, _ = oracle.fp8_error_model(q8, k8, v8, 0.01, 0.01, 0.02, 0.3)
        for t in (7.0, 7.25, 7.5, 7.75, 8.0):
            err = np.abs(_simulated_rounding_error(q8, k8, v8, 0.01, 0.01, 0.02, 0.3, t))
            assert np.all(err <= bound[0, 0]), (n, t)


def test_fp8_error_bound_is_nearly_reached():
    """Two keys: one at the row max with v = 0, one whose weight 2^7 w lands
    just above the midpoint 1 + 2^-4 of two E4M3 neighbours, so it rounds down
    by almost 2^-4 of itself (1 - 2^-8 from 17 - 2^-8 to 16): the error is
    16 (1 - 2^-8) / (17 - 2^-8) = 0.938 of the bound."""
    q8 = np.full((1, 1, 1, 1), 0x38, np.uint8)              # q = 1
    k8 = np.array([0x00, 0xB8], np.uint8).reshape(1, 1, 2, 1)   # scores 0 and -scale
    v8 = np.array([0x00, 0x38], np.uint8).reshape(1, 1, 2, 1)   # v = 0 and 1
    w2 = (1.0 + 2.0 ** -4 - 2.0 ** -12) * 2.0 ** -3          # P = 2^7 w2 = 16 (1 + 2^-4 - 2^-12)
    scale = -np.log(w2)
    err = abs(_simulated_rounding_error(q8, k8, v8, 1.0, 1.0, 1.0, scale, 7.0)[0, 0])
    bound, _ = oracle.fp8_error_model(q8, k8, v8, 1.0, 1.0, 1.0, scale)
    assert err <= bound[0, 0, 0, 0] and err >= 0.93 * bound[0, 0, 0, 0], (err, bound[0, 0, 0, 0])


def test_fp8_expected_squared_error_brackets_simulated_rounding():
    """Over many elements the mean squared rounding error lies between a
    quarter of the model's upper estimate (grid steps half as large) and the
    estimate itself, for every offset t in [7, 8]."""
    rng = np.random.default_rng(17)
    n = 400
    q8, k8, v8 = _codes(1, 1, n, 16, rng=rng), _codes(1, 1, n, 16, rng=rng, lo=-100.0, hi=100.0), \
        _codes(1, 1, n, 16, rng=rng)
    for mask in (MaskSpec("none"), MaskSpec("causal")):
        _, msq = oracle.fp8_error_model(q8, k8, v8, 0.01, 0.01, 0.02, 0.3, mask)
        for t in (7.0, 7.5, 8.0):
            if mask.kind == "causal":
                q = 0.01 * oracle.e4m3_decode(q8)[0, 0]
                k = 0.01 * oracle.e4m3_decode(k8)[0, 0]
                v = 0.02 * oracle.e4m3_decode(v8)[0, 0]
                s = np.where(np.tril(np.ones((n, n), bool)), 0.3 * q @ k.T, -np.inf)
                w = np.exp(s - s.max(axis=1, keepdims=True))
                p = torch.from_numpy(w * 2.0 ** t).to(torch.float8_e4m3fn).to(torch.float64).numpy()
                err = (p @ v) / (w * 2.0 ** t).sum(1, keepdims=True) - (w @ v) / w.sum(1, keepdims=True)
            else:
                err = _simulated_rounding_error(q8, k8, v8, 0.01, 0.01, 0.02, 0.3, t)
            m_sim, m_mod = float((err ** 2).mean()), float(msq.mean())
            assert m_mod / 8 <= m_sim <= 1.25 * m_mod, (mask.kind, t, m_sim, m_mod)


def test_fp8_error_bound_subnormal_term():
    """One key at the row max and 16384 keys whose weights (2.45 * 2^-16 of it)
    land on the subnormal grid at t = 7, all rounded the same way: the error
    exceeds the 2^-4 relative term (0 here: the only normal weight meets
    v = 0) and the bound still covers it."""
    n = 16384
    q8 = np.full((1, 1, 1, 1), 0x38, np.uint8)               # q = 1
    k8 = np.full((1, 1, n + 1, 1), 0xB8, np.uint8)           # k = -1 ...
    k8[0, 0, 0, 0] = 0x00                                    # ... but key 0 at score 0
    v8 = np.full((1, 1, n + 1, 1), 0x38, np.uint8)           # v = 1 ...
    v8[0, 0, 0, 0] = 0x00                                    # ... but 0 for the max key
    scale = -np.log(2.45 * 2.0 ** -16)
    err = abs(_simulated_rounding_error(q8, k8, v8, 1.0, 1.0, 1.0, scale, 7.0)[0, 0])
    bound, _ = oracle.fp8_error_model(q8, k8, v8, 1.0, 1.0, 1.0, scale)
    assert err > 2.0 ** -4
    assert err <= bound[0, 0, 0, 0]


# ---------------------------------------------------------------- planted mistakes

def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_mistakes(monkeypatch):
    """Each plausible slip in the oracle fails at least one of the pins above."""
    good_bwd = oa.head_backward
    good_vis = oa.visible
    good_fwd = oa.head_forward

    def bwd_no_rowsum(q, k, v, do, scale, vis):          # dropped term in dS
        p = oa._probs(q, k, scale, vis)
        dp = do @ v.T
        ds = p * dp
        return scale * (ds @ k), scale * (ds.T @ q), p.T @ do

    def bwd_sign(q, k, v, do, scale, vis):               # wrong sign in dS
        dq, dk, dv = good_bwd(q, k, v, do, scale, vis)
        return -dq, dk, dv

    def bwd_transposed(q, k, v, do, scale, vis):         # dV from P instead of P^T
        dq, dk, dv = good_bwd(q, k, v, do, scale, vis)
        p = oa._probs(q, k, scale, vis)
        return dq, dk, (p @ do) if p.shape[0] == p.shape[1] else dv * 1.5

    def vis_off_by_one(rows, nk, mask, q_offset=0, kv_offset=0):   # strict causal
        m = good_vis(rows, nk, mask, q_offset, kv_offset)
        if mask.kind == "causal":
            rows = np.asarray(rows)
            m &= (kv_offset + np.arange(nk))[None, :] < (q_offset + rows)[:, None]
        return m

    def fwd_no_scale_in_lse(q, k, v, scale, vis):        # LSE of unscaled logits
        o, lse = good_fwd(q, k, v, scale, vis)
        o2, lse2 = good_fwd(q, k, v, 1.0, vis)
        return o, lse2

    def merge_no_weights(o_parts, lse_parts):            # plain average of parts
        return (np.mean(np.stack(o_parts), 0),
                np.logaddexp.reduce(np.stack(lse_parts), axis=0))

    checks_bwd = [lambda: fd_check(oracle.attention_forward, oracle.attention_backward, MaskSpec("none")),
                  lambda: fd_check(oracle.attention_forward, oracle.attention_backward, MaskSpec("causal"))]
    for bad in (bwd_no_rowsum, bwd_sign, bwd_transposed):
        monkeypatch.setattr(oa, "head_backward", bad)
        assert any(_fails(c) for c in checks_bwd + [test_library_torch_sdpa_fwd_bwd]), bad.__name__
        monkeypatch.setattr(oa, "head_backward", good_bwd)

    monkeypatch.setattr(oa, "visible", vis_off_by_one)
    assert _fails(test_q_zero_gives_mean_of_visible_rows)
    monkeypatch.setattr(oa, "visible", good_vis)

    def vis_window_one_too_wide(rows, nk, mask, q_offset=0, kv_offset=0):   # back <= w
        if mask.kind != "sliding_window":
            return good_vis(rows, nk, mask, q_offset, kv_offset)
        return good_vis(rows, nk, MaskSpec("sliding_window", window=mask.window + 1), q_offset, kv_offset)

    monkeypatch.setattr(oa, "visible", vis_window_one_too_wide)
    assert _fails(test_sliding_window_q_zero_gives_mean_of_window)
    assert _fails(test_sliding_window_of_one_is_identity)
    monkeypatch.setattr(oa, "visible", good_vis)

    monkeypatch.setattr(oa, "head_forward", fwd_no_scale_in_lse)
    assert _fails(test_library_softmax_scipy)
    monkeypatch.setattr(oa, "head_forward", good_fwd)

    from oracle import fp8 as of
    good_dec = of.e4m3_decode

    def dec_bias_8(codes):                               # exponent bias off by one
        return 0.5 * good_dec(codes)

    def dec_no_subnormals(codes):                        # exponent field 0 read as normal
        c = np.asarray(codes, np.uint8)
        x = good_dec(codes)
        sub = ((c >> 3) & 0xF) == 0
        return np.where(sub & ((c & 7) != 0), np.sign(x) * (1 + (c & 7) / 8.0) * 2.0 ** -7, x)

    for bad in (dec_bias_8, dec_no_subnormals):
        monkeypatch.setattr(of, "e4m3_decode", bad)
        monkeypatch.setattr(oracle, "e4m3_decode", bad)
        assert _fails(test_e4m3_decode_matches_torch_float8) and _fails(test_e4m3_decode_closed_forms), bad.__name__
        monkeypatch.setattr(of, "e4m3_decode", good_dec)
        monkeypatch.setattr(oracle, "e4m3_decode", good_dec)

    good_fp8 = of.fp8_forward

    def fwd_k_descale_dropped(q8, k8, v8, qd, kd, vd, scale, mask=MaskSpec(), heads=None, rows=None):
        return good_fp8(q8, k8, v8, qd, 1.0, vd, scale, mask, heads=heads, rows=rows)

    monkeypatch.setattr(oracle, "fp8_forward", fwd_k_descale_dropped)
    assert _fails(test_fp8_forward_descale_invariances)
    monkeypatch.setattr(oracle, "fp8_forward", good_fp8)

    good_model = of.fp8_error_model

    def model_normal_only(*a, **kw):                     # subnormal term dropped
        q8, k8, v8, qd, kd, vd, scale = a[:7]
        mask = a[7] if len(a) > 7 else kw.get("mask", MaskSpec())
        q = qd * of.e4m3_decode(q8)[0, 0]
        k = kd * of.e4m3_decode(k8)[0, 0]
        v = vd * of.e4m3_decode(v8)[0, 0]
        vis = oracle.visible(np.arange(q.shape[0]), k.shape[0], mask)
        s = np.where(vis, scale * q @ k.T, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        b = (2.0 ** -4 * w) @ np.abs(v) / w.sum(1, keepdims=True)
        return b[None, None], good_model(*a, **kw)[1]

    def model_half_relative(*a, **kw):                   # 2^-5 instead of 2^-4
        b, m = good_model(*a, **kw)
        return 0.5 * b, m

    def model_step_too_small(*a, **kw):                  # expected error from half the grid step
        b, m = good_model(*a, **kw)
        return b, m / 4

    monkeypatch.setattr(oracle, "fp8_error_model", model_normal_only)
    assert _fails(test_fp8_error_bound_subnormal_term)
    monkeypatch.setattr(oracle, "fp8_error_model", model_half_relative)
    assert _fails(test_fp8_error_bound_is_nearly_reached)
    monkeypatch.setattr(oracle, "fp8_error_model", model_step_too_small)
    assert _fails(test_fp8_expected_squared_error_brackets_simulated_rounding)
    monkeypatch.setattr(oracle, "fp8_error_model", good_model)

    monkeypatch.setattr(oa, "merge_partials", merge_no_weights)
    monkeypatch.setattr(oracle, "merge_partials", merge_no_weights)
    assert _fails(test_chunked_merge_equals_monolithic)

    from oracle import schedule as osch
    good_lanes = osch.chunk_pair_lanes
    sched_golden = os.path.join(HERE, "golden", "chunk_schedule_hand_worked.json")
    units_golden = os.path.join(HERE, "golden", "fwd_units_hand_worked.json")

    def lanes_ties_to_highest(n_chunks, n_lanes=0):        # ties broken toward the highest lane
        lanes = n_lanes if n_lanes > 0 else n_chunks
        pairs = sorted(((q, k) for q in range(n_chunks) for k in range(q + 1)),
                       key=lambda p: (-osch.pair_cost(p), -p[0], p[1]))
        load, per = [0] * lanes, [[] for _ in range(lanes)]
        for p in pairs:
            best = min(range(lanes), key=lambda l: (load[l], -l))
            load[best] += osch.pair_cost(p)
            per[best].append(p)
        return per

    def lanes_qc_ascending(n_chunks, n_lanes=0):           # lighter query chunks first
        lanes = n_lanes if n_lanes > 0 else n_chunks
        pairs = sorted(((q, k) for q in range(n_chunks) for k in range(q + 1)),
                       key=lambda p: (-osch.pair_cost(p), p[0], p[1]))
        load, per = [0] * lanes, [[] for _ in range(lanes)]
        for p in pairs:
            best = min(range(lanes), key=lambda l: (load[l], l))
            load[best] += osch.pair_cost(p)
            per[best].append(p)
        return per

    for bad in (lanes_ties_to_highest, lanes_qc_ascending):
        monkeypatch.setattr(osch, "chunk_pair_lanes", bad)
        assert _fails(lambda: test_golden(sched_golden)), bad.__name__
        monkeypatch.setattr(osch, "chunk_pair_lanes", good_lanes)

    good_units = osch.fwd_work_units

    def units_chunks_ascending(kind, B, Hq, nq, nk, *a, **kw):   # light chunks first
        u = good_units(kind, B, Hq, nq, nk, *a, **kw)
        return sorted(u, key=lambda x: (x[1], x[0]))

    def units_heads_outer(kind, B, Hq, nq, nk, *a, **kw):        # head-major, not chunk-major in a group
        u = good_units(kind, B, Hq, nq, nk, *a, **kw)
        return sorted(u, key=lambda x: (x[0], -x[1]))

    for bad in (units_chunks_ascending, units_heads_outer):
        monkeypatch.setattr(oracle, "fwd_work_units", bad)
        assert _fails(lambda: test_golden(units_golden)), bad.__name__
        monkeypatch.setattr(oracle, "fwd_work_units", good_units)

    good_pb = oa.partial_backward

    def pb_local_normaliser(q, k, v, do, lse, dsum, scale, mask=MaskSpec(), q_offset=0, kv_offset=0):
        # each chunk normalised over its own keys instead of the merged LSE
        _, lse_c = oracle.attention_forward(q, k, v, scale, mask, q_offset, kv_offset)
        return good_pb(q, k, v, do, lse_c, dsum, scale, mask, q_offset, kv_offset)

    def pb_no_dsum(q, k, v, do, lse, dsum, scale, mask=MaskSpec(), q_offset=0, kv_offset=0):
        return good_pb(q, k, v, do, lse, np.zeros_like(dsum), scale, mask, q_offset, kv_offset)

    def pb_dk_unscaled(q, k, v, do, lse, dsum, scale, mask=MaskSpec(), q_offset=0, kv_offset=0):
        dq, dk, dv = good_pb(q, k, v, do, lse, dsum, scale, mask, q_offset, kv_offset)
        return dq, dk / scale, dv

    def pb_offsets_swapped(q, k, v, do, lse, dsum, scale, mask=MaskSpec(), q_offset=0, kv_offset=0):
        return good_pb(q, k, v, do, lse, dsum, scale, mask, kv_offset, q_offset)

    for bad in (pb_local_normaliser, pb_no_dsum, pb_dk_unscaled, pb_offsets_swapped):
        monkeypatch.setattr(oracle, "partial_backward", bad)
        assert _fails(test_chunked_backward_equals_monolithic), bad.__name__
        monkeypatch.setattr(oracle, "partial_backward", good_pb)

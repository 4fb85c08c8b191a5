"""GPU: every CTA's own record of the work it did (attn_debug_set_tile_counts)
against a brute-force count from the mask definition.  For each work unit the
expected number of key tiles a query tile visits (or query tiles a key tile
visits, in the dK/dV kernel) is the number of 128 x 128 tile pairs holding at
least one visible (query, key) pair, found by evaluating the oracle's
element-wise visibility rule over the whole tile pair; the kernels instead
skip tiles by ranges and block-mask rows ("FlashAttention-2" reviews, fourth
review: fully masked blocks are skipped; causal masking makes later chunks
heavier, "DISTFLASHATTN" reviews, first review point 1).  The records also
pin each CTA's unit identity (every unit exactly once) and, for the forward,
the heaviest-first launch order of the oracle's schedule restatement."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import schedule as osched
from io_aware_exact_attn_gb300 import _ffi, api, inputs
from _gpu_helpers import make, mask_spec

pytestmark = pytest.mark.gpu

T = 128
F = 8   # int32 fields per CTA record


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    api.debug_set_tile_counts(None)
    assert api.get_status() == 0


def cdiv(a, b):
    return -(-a // b)


def tiles_seen(rows, nk, spec, q_off=0, kv_off=0, kt_range=None):
    """Key tiles holding at least one key visible to one of ``rows``."""
    if len(rows) == 0 or nk == 0:
        return set()
    vis = oracle.visible(np.asarray(rows), nk, spec, q_off, kv_off)
    any_col = vis.any(axis=0)
    kts = range(cdiv(nk, T)) if kt_range is None else kt_range
    return {kt for kt in kts if any_col[kt * T:(kt + 1) * T].any()}


class Recorder:
    """A device record array larger than the launches need, filled with -1,
    so untouched records and writes past the last CTA both show."""

    def __init__(self, ctas):
        self.ctas = ctas
        self.buf = torch.full(((ctas + 16) * F,), -1, dtype=torch.int32, device="cuda")
        api.debug_set_tile_counts(self.buf)

    def records(self, first=0, n=None):
        torch.cuda.synchronize()
        a = self.buf.view(-1, F).cpu().numpy()
        n = self.ctas - first if n is None else n
        tail = a[first + n:] if first + n >= self.ctas else a[self.ctas:]
        assert (tail == -1).all(), "a record was written past the launch's CTAs"
        return a[first:first + n]


def check_records(recs, expected, allow_empty=0):
    """``expected``: {identity (4 ints): counts (4 ints)}; every unit exactly once."""
    got = {}
    empty = 0
    for r in recs:
        if (r == -1).all():
            empty += 1
            continue
        key = tuple(int(x) for x in r[:4])
        assert key not in got, f"unit {key} ran twice"
        got[key] = tuple(int(x) for x in r[4:])
    assert empty == allow_empty, f"{empty} CTAs left no record, expected {allow_empty}"
    assert got.keys() == expected.keys()
    bad = {k: (got[k], expected[k]) for k in expected if got[k] != expected[k]}
    assert not bad, f"{len(bad)} units differ, e.g. {list(bad.items())[:3]}"


def ragged_grid(B, heads, total, max_len, rows):
    """CTAs a ragged launch has: one unit per head and tile of every sequence,
    bounded by heads * (ceil(total / rows) + B) (the unit order is sequence
    by sequence, so the CTAs past the last unit do nothing)."""
    return heads * min(B * cdiv(max_len, rows), cdiv(total, rows) + B)


def fwd_expected(B, Hq, Nq, Nk, spec, q_off=0, kv_off=0):
    exp = {}
    for qc in range(cdiv(Nq, 256)):
        per_t = []
        for t in range(2):
            r0 = qc * 256 + t * T
            per_t.append(tiles_seen(range(r0, min(Nq, r0 + T)), Nk, spec, q_off, kv_off))
        counts = (len(per_t[0] | per_t[1]), 0, len(per_t[0]), len(per_t[1]))
        for bh in range(B * Hq):
            exp[(bh, qc * 256, 0, 0)] = counts
    return exp


FWD_CASES = [
    # B, Hq, Hkv, N, d, kind, extra
    (1, 4, 2, 1000, 128, "causal", {}),
    (2, 2, 2, 700, 64, "none", {}),
    (1, 3, 1, 1500, 128, "sliding_window", {"window": 300}),
    (1, 2, 2, 1024, 64, "block_sparse", {"cib": False}),
    (1, 2, 2, 1024, 128, "block_sparse", {"cib": True}),
]


def block_mask_with_gaps(nb):
    bm = inputs.block_sparse_mask(nb, nb, 0.35, seed=21)
    bm[2, :] = False   # a query block row with nothing to see
    bm[:, 5] = False   # a key block column nobody sees
    return bm


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: f"{c[5]}-N{c[3]}-d{c[4]}")
def test_forward_records_match_the_mask(case):
    B, Hq, Hkv, N, d, kind, extra = case
    q, k, v, _ = make(B, Hq, Hkv, N, d)
    bm = block_mask_with_gaps(cdiv(N, T)) if kind == "block_sparse" else None
    cib = extra.get("cib", False)
    window = extra.get("window")
    spec = mask_spec(kind, bm, cib, window or 0)
    ctas = B * Hq * cdiv(N, 256)
    rec = Recorder(ctas)
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    api.attn_fwd(q, k, v, causal=kind == "causal", block_mask=bmt, causal_in_blocks=cib, window=window)
    recs = rec.records()
    check_records(recs, fwd_expected(B, Hq, N, N, spec))
    # launch order and per-unit key-tile counts of the schedule restatement
    sched = osched.fwd_work_units(kind, B, Hq, N, N, block_mask=bm, causal_in_blocks=cib, Hkv=Hkv, d=d,
                                  window=window or 0)
    assert [(int(r[0]), int(r[1]) // 256, int(r[4])) for r in recs] == [tuple(u) for u in sched]


def test_partial_forward_records_with_offsets():
    """A (query chunk, key chunk) pair at global offsets: tiles are skipped by
    global positions."""
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 512, 384, 128
    q_off, kv_off = 640, 256
    q, k, v, _ = make(B, Hq, Hkv, Nq, d, Nk=Nk)
    rec = Recorder(B * Hq * cdiv(Nq, 256))
    api.attn_partial_fwd(q, k, v, q_offset=q_off, kv_offset=kv_off, causal=True)
    check_records(rec.records(), fwd_expected(B, Hq, Nq, Nk, oracle.MaskSpec("causal"), q_off, kv_off))
    # the diagonal: the query chunk's first rows sit before part of the key chunk
    rec = Recorder(B * Hq * cdiv(Nq, 256))
    api.attn_partial_fwd(q, k, v, q_offset=300, kv_offset=400, causal=True)
    check_records(rec.records(), fwd_expected(B, Hq, Nq, Nk, oracle.MaskSpec("causal"), 300, 400))


def test_varlen_forward_records():
    lens = [300, 800, 30, 1100]
    Hq, Hkv, d = 4, 2, 64
    total = sum(lens)
    q = inputs.randn_bf16((total, Hq, d), seed=31).cuda()
    k = inputs.randn_bf16((total, Hkv, d), seed=32).cuda()
    v = inputs.randn_bf16((total, Hkv, d), seed=33).cuda()
    cu_h = np.concatenate([[0], np.cumsum(lens)])
    cu = torch.tensor(cu_h, dtype=torch.int32).cuda()
    B = len(lens)
    grid = ragged_grid(B, Hq, total, max(lens), 256)
    rec = Recorder(grid)
    api.attn_varlen_fwd(q, k, v, cu, causal=True)
    exp = {}
    spec = oracle.MaskSpec("causal")
    for b, n in enumerate(lens):
        for qc in range(cdiv(n, 256)):
            per_t = [tiles_seen(range(qc * 256 + t * T, min(n, qc * 256 + t * T + T)), n, spec) for t in range(2)]
            for h in range(Hq):
                exp[(h, qc * 256, 0, int(cu_h[b]))] = (len(per_t[0] | per_t[1]), 0, len(per_t[0]), len(per_t[1]))
    check_records(rec.records(), exp, allow_empty=grid - len(exp))


def test_decode_records():
    """Split-KV decoding: each split visits its share of the sequence's key
    tiles; splits past a short sequence's end visit none."""
    B, Hq, Hkv, Nq, Nk, d, ns = 2, 8, 2, 1, 5000, 128, 3
    q = inputs.randn_bf16((B, Hq, Nq, d), seed=41).cuda()
    kc = inputs.randn_bf16((B, Hkv, Nk, d), seed=42).cuda()
    vc = inputs.randn_bf16((B, Hkv, Nk, d), seed=43).cuda()
    lens = [5000, 200]
    sl = torch.tensor(lens, dtype=torch.int32).cuda()
    rec = Recorder(B * Hkv * ns)
    api.attn_decode(q, kc, vc, seq_lens=sl, n_splits=ns)
    st = cdiv(cdiv(Nk, T), ns)   # key tiles per split
    g = Hq // Hkv
    rows = g * Nq
    # the g * Nq rows fit one tile: both query tiles take them, tile t the
    # split's key tiles kt with kt % 2 == t
    assert rows <= T and 2 * ns <= 64
    exp = {}
    for b in range(B):
        n = lens[b]
        nkt = cdiv(n, T)
        for hk in range(Hkv):
            for s in range(ns):
                kr = range(min(s * st, nkt), min((s + 1) * st, nkt))
                seen = tiles_seen(np.arange(rows) % Nq, n, oracle.MaskSpec("causal"), q_off=n - Nq, kt_range=kr)
                per_t = [{kt for kt in seen if kt % 2 == t} for t in range(2)]
                exp[(b * Hkv + hk, 0, s, 0)] = (len(per_t[0] | per_t[1]), 0, len(per_t[0]), len(per_t[1]))
    check_records(rec.records(), exp)


def bwd_expected(B, Hq, Hkv, N, spec, tok0=0):
    """dK/dV: per (b*Hkv + kv head, key tile) the (query head, query tile)
    pairs with a visible pair; dQ: per (b*Hq + h, query tile) the key tiles."""
    nt = cdiv(N, T)
    g = Hq // Hkv
    seen = [tiles_seen(range(qt * T, min(N, qt * T + T)), N, spec) for qt in range(nt)]
    dkdv, dq = {}, {}
    for kt in range(nt):
        c = g * sum(kt in seen[qt] for qt in range(nt))
        for bkv in range(B * Hkv):
            dkdv[(bkv, kt, 0, tok0)] = (c, c, c, c)
    for qt in range(nt):
        c = len(seen[qt])
        for bh in range(B * Hq):
            dq[(bh, qt, 0, tok0)] = (c, c, c, c)
    return dkdv, dq


BWD_CASES = [
    (1, 4, 2, 1000, 128, "causal", {}),
    (1, 2, 2, 1500, 64, "sliding_window", {"window": 300}),
    (2, 2, 1, 1024, 64, "block_sparse", {"cib": False}),
    (1, 2, 2, 1024, 128, "block_sparse", {"cib": True}),
    (1, 2, 2, 640, 128, "none", {}),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"{c[5]}-N{c[3]}-d{c[4]}")
@pytest.mark.parametrize("entry", ["attn_bwd", "static_scratch"])
def test_backward_records_match_the_mask(case, entry):
    B, Hq, Hkv, N, d, kind, extra = case
    q, k, v, do = make(B, Hq, Hkv, N, d)
    bm = block_mask_with_gaps(cdiv(N, T)) if kind == "block_sparse" else None
    cib = extra.get("cib", False)
    window = extra.get("window")
    spec = mask_spec(kind, bm, cib, window or 0)
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    kw = dict(causal=kind == "causal", block_mask=bmt, causal_in_blocks=cib, window=window)
    o, lse = api.attn_fwd(q, k, v, **kw)
    n_dkdv, n_dq = B * Hkv * cdiv(N, T), B * Hq * cdiv(N, T)
    rec = Recorder(n_dkdv + n_dq)
    if entry == "attn_bwd":
        api.attn_bwd(q, k, v, o, lse, do, **kw)
    else:
        if kind in ("block_sparse", "sliding_window"):
            pytest.skip("the static-scratch entry point is exercised with the plain masks")
        grads = [torch.empty_like(t) for t in (q, k, v)]
        m, _ = api.mask_desc(causal=kind == "causal")
        rc = _ffi.lib().attn_bwd_static_scratch(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            *[g.data_ptr() for g in grads], B, Hq, Hkv, N, d, 1.0 / math.sqrt(d),
            ctypes.byref(m) if m is not None else None, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, _ffi.lib().attn_last_error_message()
    exp_dkdv, exp_dq = bwd_expected(B, Hq, Hkv, N, spec)
    check_records(rec.records(0, n_dkdv), exp_dkdv)
    check_records(rec.records(n_dkdv, n_dq), exp_dq)


def test_varlen_backward_records():
    lens = [300, 800, 30]
    Hq, Hkv, d = 2, 1, 128
    total = sum(lens)
    q = inputs.randn_bf16((total, Hq, d), seed=51).cuda()
    k = inputs.randn_bf16((total, Hkv, d), seed=52).cuda()
    v = inputs.randn_bf16((total, Hkv, d), seed=53).cuda()
    do = inputs.randn_bf16((total, Hq, d), seed=54).cuda()
    cu_h = np.concatenate([[0], np.cumsum(lens)])
    cu = torch.tensor(cu_h, dtype=torch.int32).cuda()
    o, lse = api.attn_varlen_fwd(q, k, v, cu, causal=True)
    B = len(lens)
    n_dkdv, n_dq = ragged_grid(B, Hkv, total, max(lens), T), ragged_grid(B, Hq, total, max(lens), T)
    rec = Recorder(n_dkdv + n_dq)
    api.attn_varlen_bwd(q, k, v, o, lse, do, cu, causal=True)
    exp_dkdv, exp_dq = {}, {}
    spec = oracle.MaskSpec("causal")
    for b, n in enumerate(lens):
        e_kv, e_q = bwd_expected(1, Hq, Hkv, n, spec, tok0=int(cu_h[b]))
        for (bkv, kt, z, t0), c in e_kv.items():
            exp_dkdv[(b * Hkv + bkv, kt, z, t0)] = c
        for (bh, qt, z, t0), c in e_q.items():
            exp_dq[(b * Hq + bh, qt, z, t0)] = c
    check_records(rec.records(0, n_dkdv), exp_dkdv, allow_empty=n_dkdv - len(exp_dkdv))
    check_records(rec.records(n_dkdv, n_dq), exp_dq, allow_empty=n_dq - len(exp_dq))


def test_record_array_too_small_is_refused():
    q, k, v, _ = make(1, 2, 2, 512, 64)
    small = torch.full((8 * 3,), -1, dtype=torch.int32, device="cuda")   # 3 records; the launch has 4 CTAs
    api.debug_set_tile_counts(small)
    with pytest.raises(_ffi.AttnError, match="debug record"):
        api.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert (small.cpu() == -1).all(), "a refused launch wrote records"
    api.debug_set_tile_counts(None)
    api.attn_fwd(q, k, v, causal=True)   # recording off: runs as usual

"""Exact attention, its gradient and the log-sum-exp merge, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain definitions,
full score rows, no online softmax.  Query rows are independent of one another
by definition (each row has its own softmax), so long sequences are processed
in blocks of whole query rows purely to bound memory; within a block every
row sees all of its keys at once.

Notation: ``S = scale * Q K^T``, ``P = softmax_rows(S)`` over the visible keys,
``O = P V``, ``LSE_i = log sum_j exp(S_ij)`` (natural log).  Backward for the
loss ``<O, dO>``: ``dV = P^T dO``, ``dP = dO V^T``,
``dS = P * (dP - rowsum(P * dP))`` (the softmax Jacobian applied row by row),
``dQ = scale * dS K``, ``dK = scale * dS^T Q``.

Readings where the pages are silent:
* scale is an explicit argument (the DISTFLASHATTN review writes
  ``softmax(QK^T)V`` with no scale);
* causal visibility uses global positions: key ``j`` is visible to query ``i``
  iff ``kv_offset + j <= q_offset + i``;
* a query row with no visible key has ``O = 0``, ``LSE = -inf`` and zero
  gradients;
* grouped-query attention maps query head ``h`` to key/value head
  ``h // (Hq // Hkv)``, and dK/dV sum over the query heads of a group;
* block-sparse: a kept ``block x block`` block is dense, a dropped one is
  masked out entirely (FlashAttention abstract; BurstAttention author
  responses: sparse attention only changes the mask matrix);
* sliding window of width ``w`` (the local attention the FlashAttention-2
  reviews mention for Mistral): key ``j`` is visible to query ``i`` iff
  ``0 <= (q_offset + i) - (kv_offset + j) < w``, i.e. the causal rule plus
  the ``w`` most recent positions, the query's own included.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

ROW_BLOCK = 1024  # query rows per block when a head is processed in pieces


@dataclass(frozen=True)
class MaskSpec:
    """Which keys a query may see.

    kind: ``"none"``, ``"causal"``, ``"block_sparse"`` or ``"sliding_window"``.
    block_mask: for ``block_sparse``, a boolean ``[ceil(Nq/block), ceil(Nk/block)]``
        array shared by every batch and head; ``True`` keeps the block.
    causal_in_blocks: for ``block_sparse``, additionally apply the element
        causal rule inside kept blocks.
    window: for ``sliding_window``, how many positions a query looks back,
        its own included (``>= 1``).
    """

    kind: str = "none"
    block_mask: Optional[np.ndarray] = None
    block: int = 128
    causal_in_blocks: bool = False
    window: int = 0

    def __post_init__(self):
        if self.kind not in ("none", "causal", "block_sparse", "sliding_window"):
            raise ValueError(f"unknown mask kind {self.kind!r}")
        if self.kind == "block_sparse" and self.block_mask is None:
            raise ValueError("block_sparse needs a block_mask")
        if self.kind == "sliding_window" and self.window < 1:
            raise ValueError("sliding_window needs window >= 1")


def visible(rows: np.ndarray, nk: int, mask: MaskSpec,
            q_offset: int = 0, kv_offset: int = 0) -> np.ndarray:
    """Boolean ``[len(rows), nk]``: True where key ``j`` is visible to query ``rows[i]``.

    ``rows`` are local query indices of this call; positions used by the
    causal rule are ``q_offset + row`` and ``kv_offset + j``.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(nk, dtype=np.int64)
    vis = np.ones((rows.size, nk), dtype=bool)
    causal = mask.kind in ("causal", "sliding_window") or (mask.kind == "block_sparse" and mask.causal_in_blocks)
    back = (q_offset + rows)[:, None] - (kv_offset + cols)[None, :]   # how far key j lies behind query i
    if causal:
        vis &= back >= 0
    if mask.kind == "sliding_window":
        vis &= back < mask.window
    if mask.kind == "block_sparse":
        bm = np.asarray(mask.block_mask, dtype=bool)
        vis &= bm[(rows // mask.block)[:, None], (cols // mask.block)[None, :]]
    return vis


def head_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                 vis: np.ndarray):
    """One head, a set of query rows: returns ``(O [r, d], LSE [r])``.

    ``q`` is ``[r, d]`` (the query rows), ``k``/``v`` are ``[nk, d]``, ``vis``
    is the boolean ``[r, nk]`` visibility of each key.
    """
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has = np.isfinite(m)
    m0 = np.where(has, m, 0.0)
    e = np.exp(s - m0[:, None])            # exp(-inf) = 0 for hidden keys
    l = e.sum(axis=1)
    p = e / np.where(has, l, 1.0)[:, None]
    o = p @ v
    lse = np.where(has, m0 + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def _probs(q, k, scale, vis):
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has = np.isfinite(m)
    e = np.exp(s - np.where(has, m, 0.0)[:, None])
    l = e.sum(axis=1)
    return e / np.where(has, l, 1.0)[:, None]


def head_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                  scale: float, vis: np.ndarray):
    """One head, a set of query rows: returns ``(dQ [r,d], dK [nk,d], dV [nk,d])``.

    dK and dV are the contributions of these rows only (sum them over row sets
    and over the query heads of a group).
    """
    p = _probs(q, k, scale, vis)
    dv = p.T @ do
    dp = do @ v.T
    # softmax Jacobian-vector product, row by row: dS = P * (dP - <P, dP>)
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def _group(hq: int, hkv: int) -> int:
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // hkv


def attention_forward(q, k, v, scale: float, mask: MaskSpec = MaskSpec(),
                      q_offset: int = 0, kv_offset: int = 0,
                      heads: Optional[Sequence] = None,
                      rows: Optional[np.ndarray] = None):
    """Exact attention forward in float64.

    ``q`` is ``[B, Hq, Nq, d]``, ``k``/``v`` are ``[B, Hkv, Nk, d]``.
    Without ``heads``/``rows`` returns full ``O [B,Hq,Nq,d]`` and
    ``LSE [B,Hq,Nq]``.  With ``heads`` (a list of ``(b, h)``) and ``rows``
    (local query indices) returns ``O [len(heads), len(rows), d]`` and
    ``LSE [len(heads), len(rows)]`` for that sample only.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = _group(Hq, Hkv)
    sample = heads is not None
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    rows = np.arange(Nq) if rows is None else np.asarray(rows, np.int64)
    o_out = np.zeros((len(heads), rows.size, d))
    l_out = np.zeros((len(heads), rows.size))
    for n, (b, h) in enumerate(heads):
        kk, vv = k[b, h // g], v[b, h // g]
        for s0 in range(0, rows.size, ROW_BLOCK):
            r = rows[s0:s0 + ROW_BLOCK]
            vis = visible(r, Nk, mask, q_offset, kv_offset)
            o, l = head_forward(q[b, h, r], kk, vv, scale, vis)
            o_out[n, s0:s0 + r.size] = o
            l_out[n, s0:s0 + r.size] = l
    if sample:
        return o_out, l_out
    return o_out.reshape(B, Hq, rows.size, d), l_out.reshape(B, Hq, rows.size)


def attention_backward(q, k, v, do, scale: float, mask: MaskSpec = MaskSpec(),
                       q_offset: int = 0, kv_offset: int = 0,
                       kv_heads: Optional[Sequence] = None):
    """Exact gradient of ``<O, dO>`` with respect to Q, K, V, in float64.

    Without ``kv_heads`` returns full ``dQ [B,Hq,Nq,d]``, ``dK``/``dV``
    ``[B,Hkv,Nk,d]``.  With ``kv_heads`` (a list of ``(b, hkv)``) computes only
    those key/value heads and the query heads of their groups, returning
    ``dQ [len, g, Nq, d]``, ``dK [len, Nk, d]``, ``dV [len, Nk, d]``.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); do = np.asarray(do, np.float64)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = _group(Hq, Hkv)
    sample = kv_heads is not None
    if kv_heads is None:
        kv_heads = [(b, hk) for b in range(B) for hk in range(Hkv)]
    dq = np.zeros((len(kv_heads), g, Nq, d))
    dk = np.zeros((len(kv_heads), Nk, d))
    dv = np.zeros((len(kv_heads), Nk, d))
    for n, (b, hk) in enumerate(kv_heads):
        for j in range(g):
            h = hk * g + j
            for s0 in range(0, Nq, ROW_BLOCK):
                r = np.arange(s0, min(Nq, s0 + ROW_BLOCK))
                vis = visible(r, Nk, mask, q_offset, kv_offset)
                a, bk, bv = head_backward(q[b, h, r], k[b, hk], v[b, hk], do[b, h, r], scale, vis)
                dq[n, j, r] = a
                dk[n] += bk
                dv[n] += bv
    if sample:
        return dq, dk, dv
    return dq.reshape(B, Hq, Nq, d), dk.reshape(B, Hkv, Nk, d), dv.reshape(B, Hkv, Nk, d)


def attention_backward_dq_rows(q, k, v, do, scale: float, b: int, h: int, rows,
                               mask: MaskSpec = MaskSpec(), q_offset: int = 0,
                               kv_offset: int = 0):
    """dQ for selected query rows of one head (each dQ row depends on its own row only)."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); do = np.asarray(do, np.float64)
    g = _group(q.shape[1], k.shape[1])
    rows = np.asarray(rows, np.int64)
    vis = visible(rows, k.shape[2], mask, q_offset, kv_offset)
    dq, _, _ = head_backward(q[b, h, rows], k[b, h // g], v[b, h // g], do[b, h, rows], scale, vis)
    return dq


def partial_backward(q, k, v, do, lse, dsum, scale: float, mask: MaskSpec = MaskSpec(),
                     q_offset: int = 0, kv_offset: int = 0):
    """One (query chunk, key/value chunk) term of the gradient of ``<O, dO>``.

    Attention over a sequence cut into chunks is a sum over key chunks, so its
    gradient is too, once every row's softmax normaliser is the one over ALL
    of the row's keys (DISTFLASHATTN reviews, first review summary: forward and
    backward computed chunk by chunk over workers; BurstAttention author
    responses: local results tied together by the online-softmax statistics).
    Given the merged ``lse [B, Hq, Nq]`` (natural log, over every key of the
    row) and ``dsum = rowsum(dO * O) [B, Hq, Nq]`` of the merged output ``O``,
    the chunk's probabilities are ``P_ij = exp(S_ij - lse_i)`` on its visible
    keys (0 elsewhere and on rows with ``lse = -inf``), and its terms are
    ``dV = P^T dO``, ``dP = dO V^T``, ``dS = P * (dP - dsum)``,
    ``dQ = scale dS K``, ``dK = scale dS^T Q``; dK and dV sum over the query
    heads of a GQA group.  Summed over the key chunks (dQ) and the query chunks
    (dK, dV) these terms give ``attention_backward`` of the whole sequence.

    ``q``, ``do`` ``[B, Hq, Nq, d]``; ``k``, ``v`` ``[B, Hkv, Nk, d]``; positions
    ``q_offset + i`` and ``kv_offset + j`` as in ``visible``.  Returns
    ``dQ [B,Hq,Nq,d]``, ``dK``, ``dV [B,Hkv,Nk,d]``.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); do = np.asarray(do, np.float64)
    lse = np.asarray(lse, np.float64); dsum = np.asarray(dsum, np.float64)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = _group(Hq, Hkv)
    dq = np.zeros((B, Hq, Nq, d))
    dk = np.zeros((B, Hkv, Nk, d))
    dv = np.zeros((B, Hkv, Nk, d))
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            for s0 in range(0, Nq, ROW_BLOCK):
                r = np.arange(s0, min(Nq, s0 + ROW_BLOCK))
                vis = visible(r, Nk, mask, q_offset, kv_offset)
                s = scale * (q[b, h, r] @ k[b, hk].T)
                l = lse[b, h, r]
                fin = np.isfinite(l)
                with np.errstate(invalid="ignore", over="ignore"):
                    p = np.where(vis & fin[:, None], np.exp(s - np.where(fin, l, 0.0)[:, None]), 0.0)
                dp = do[b, h, r] @ v[b, hk].T
                ds = p * (dp - dsum[b, h, r][:, None])
                dq[b, h, r] = scale * (ds @ k[b, hk])
                dk[b, hk] += scale * (ds.T @ q[b, h, r])
                dv[b, hk] += p.T @ do[b, h, r]
    return dq, dk, dv


def varlen_forward(q, k, v, cu_seqlens, scale: float, mask: MaskSpec = MaskSpec()):
    """Exact attention over sequences packed back to back, in float64.

    ``q`` is ``[total, Hq, d]`` and ``k``/``v`` ``[total, Hkv, d]`` (token-major);
    sequence ``b`` is tokens ``cu_seqlens[b]:cu_seqlens[b+1]``.  Each sequence
    is attended on its own with local positions (no key of one sequence is
    visible to another's queries).  Returns ``O [total, Hq, d]`` and
    ``LSE [Hq, total]``.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    total, Hq, d = q.shape
    o = np.zeros((total, Hq, d))
    lse = np.full((Hq, total), -np.inf)
    cu = [int(x) for x in cu_seqlens]
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        if s1 <= s0:
            continue
        ob, lb = attention_forward(q[s0:s1].transpose(1, 0, 2)[None], k[s0:s1].transpose(1, 0, 2)[None],
                                   v[s0:s1].transpose(1, 0, 2)[None], scale, mask)
        o[s0:s1] = ob[0].transpose(1, 0, 2)
        lse[:, s0:s1] = lb[0]
    return o, lse


def varlen_backward(q, k, v, do, cu_seqlens, scale: float, mask: MaskSpec = MaskSpec()):
    """Exact gradient of ``<O, dO>`` for sequences packed back to back (the
    layouts of ``varlen_forward``): each sequence on its own.  Returns
    ``dQ [total, Hq, d]``, ``dK``/``dV`` ``[total, Hkv, d]``."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); do = np.asarray(do, np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    cu = [int(x) for x in cu_seqlens]
    t = lambda x: x.transpose(1, 0, 2)[None]
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        if s1 <= s0:
            continue
        a, bk, bv = attention_backward(t(q[s0:s1]), t(k[s0:s1]), t(v[s0:s1]), t(do[s0:s1]), scale, mask)
        dq[s0:s1], dk[s0:s1], dv[s0:s1] = (x[0].transpose(1, 0, 2) for x in (a, bk, bv))
    return dq, dk, dv


def decode_forward(q, k_cache, v_cache, scale: float, seq_lens=None, causal: bool = True):
    """Attention of the newest ``Nq`` positions of each sequence against its
    key/value cache, in float64 (the decoding step of a KV-cache model;
    FlashAttention-2 reviews: splitting the KV cache among thread blocks).

    ``q`` is ``[B, Hq, Nq, d]``; ``k_cache``/``v_cache`` are ``[B, Hkv, Nk, d]``
    of which sequence ``b`` uses the first ``seq_lens[b]`` positions (all
    ``Nk`` when ``seq_lens`` is None).  Query ``i`` of sequence ``b`` sits at
    position ``seq_lens[b] - Nq + i``; with ``causal`` it sees the cached keys
    at positions up to its own, otherwise every cached key of its sequence.
    Returns ``O [B, Hq, Nq, d]`` and ``LSE [B, Hq, Nq]``.
    """
    q = np.asarray(q, np.float64)
    B, Hq, Nq, d = q.shape
    Nk = np.asarray(k_cache).shape[2]
    lens = [Nk] * B if seq_lens is None else [int(x) for x in seq_lens]
    o = np.zeros((B, Hq, Nq, d))
    lse = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        n = lens[b]
        if n <= 0:
            continue
        ob, lb = attention_forward(q[b:b + 1], np.asarray(k_cache)[b:b + 1, :, :n], np.asarray(v_cache)[b:b + 1, :, :n],
                                   scale, MaskSpec("causal" if causal else "none"), q_offset=n - Nq, kv_offset=0)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine partial attention results over disjoint key sets.

    Each part ``c`` holds ``O_c`` (normalised over its own keys) and
    ``LSE_c``.  The result over the union of keys is
    ``LSE = log sum_c exp(LSE_c)`` and ``O = sum_c exp(LSE_c - LSE) O_c``;
    a part with ``LSE_c = -inf`` weighs zero, and a row where every part is
    ``-inf`` gives ``O = 0``, ``LSE = -inf``.
    (BurstAttention author responses: online-softmax combination of local
    attention results across devices.)
    """
    lse = np.stack([np.asarray(x, np.float64) for x in lse_parts])
    o = np.stack([np.asarray(x, np.float64) for x in o_parts])
    total = np.logaddexp.reduce(lse, axis=0)
    fin = np.isfinite(total)
    with np.errstate(invalid="ignore"):
        w = np.where(fin[None], np.exp(lse - np.where(fin, total, 0.0)[None]), 0.0)
    out = (w[..., None] * o).sum(axis=0)
    return out, total

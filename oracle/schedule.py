"""Integer work schedules, restated in plain Python.

TEST INFRASTRUCTURE ONLY (see the package docstring).  These are the
bookkeeping rules the CUDA library follows; tests compare the library's
exported builders with these element by element.

Readings (the pages describe load balancing only in words: DISTFLASHATTN
reviews, first review points 1-2 and third review summary; FlashAttention-2
reviews, fourth review on causal block skipping; none prints the schedule):

* Forward work unit = one CTA = 256 query rows (two 128-row tiles) of one
  (batch, query head).  Heads are taken in groups of
  ``G = clamp((Hq/Hkv) * floor(64 MiB / (4*Nk*d)), 1, B*Hq)`` consecutive heads
  (the last group may be smaller), so that a group's K and V fit in L2.  Inside
  a group units go heaviest first: the latest query chunk of each head of the
  group (heads in order), then the next latest, and so on.  Under a causal
  mask later query chunks see more key tiles, so this is a
  longest-processing-time-first order that the hardware block scheduler then
  assigns greedily to free SMs.
* A unit's key tiles are the union of the key tiles its two query tiles see.
* Chunk pairs for chunked causal attention: every ``(qc, kc)`` with
  ``kc <= qc``; an off-diagonal pair costs 2, a diagonal pair (half masked)
  costs 1.  Pairs are sorted by (cost desc, qc desc, kc asc) and each is given
  to the least-loaded of ``n_lanes`` virtual lanes (lowest lane on ties);
  the output interleaves the lanes round-robin by position.
"""
from __future__ import annotations

import numpy as np

TILE = 128          # rows of a query tile / key tile
UNIT_ROWS = 256     # query rows of one forward work unit


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def kv_tile_range_causal(r_first: int, r_last: int, nk: int,
                         q_offset: int, kv_offset: int) -> int:
    """Number of leading key tiles with any key visible to query rows
    ``r_first..r_last`` (local, inclusive) under the causal rule."""
    nkt = _cdiv(nk, TILE)
    if r_last < r_first:
        return 0
    last_pos = q_offset + r_last
    if last_pos < kv_offset:
        return 0
    return min(nkt, (last_pos - kv_offset) // TILE + 1)


def _tile_kv_set(t_row: int, nq: int, nk: int, kind: str, q_offset: int,
                 kv_offset: int, block_mask, causal_in_blocks: bool, window: int = 0):
    """Set of key tiles visible to query tile ``t_row`` (row-block index)."""
    nkt = _cdiv(nk, TILE)
    r0 = t_row * TILE
    if r0 >= nq:
        return set()
    r1 = min(nq, r0 + TILE) - 1
    if kind == "none":
        return set(range(nkt))
    if kind == "sliding_window":
        # brute force over the tile's rows and every key: a key tile counts
        # when any of its keys lies 0..window-1 positions behind any row
        back = (q_offset + np.arange(r0, r1 + 1))[:, None] - (kv_offset + np.arange(nk))[None, :]
        seen = ((back >= 0) & (back < window)).any(axis=0)
        return {kt for kt in range(nkt) if seen[kt * TILE:(kt + 1) * TILE].any()}
    lim = kv_tile_range_causal(r0, r1, nk, q_offset, kv_offset)
    if kind == "causal":
        return set(range(lim))
    bm = np.asarray(block_mask, dtype=bool)
    keep = {kt for kt in range(nkt) if bm[t_row, kt]}
    if causal_in_blocks:
        keep = {kt for kt in keep if kt < lim}
    return keep


L2_GROUP_BYTES = 64 * 2 ** 20


def head_group(B: int, Hq: int, Hkv: int, nk: int, d: int) -> int:
    """Heads per group: as many query heads as share <= 64 MiB of K and V."""
    g = (Hq // Hkv) * (L2_GROUP_BYTES // (4 * nk * d))
    return max(1, min(B * Hq, g))


def fwd_work_units(kind: str, B: int, Hq: int, nq: int, nk: int,
                   q_offset: int = 0, kv_offset: int = 0, block_mask=None,
                   causal_in_blocks: bool = False, Hkv: int = None, d: int = 128,
                   window: int = 0):
    """Forward work units in launch order: list of ``(bh, qchunk, n_kv_tiles)``."""
    Hkv = Hq if Hkv is None else Hkv
    bh_n = B * Hq
    nqc = _cdiv(nq, UNIT_ROWS)
    G = head_group(B, Hq, Hkv, nk, d)
    order = []
    for first in range(0, bh_n, G):
        heads = list(range(first, min(bh_n, first + G)))
        for pos in range(nqc):
            for bh in heads:
                order.append((bh, nqc - 1 - pos))
    out = []
    for bh, qc in order:
        kv = set()
        for t in range(2):
            kv |= _tile_kv_set(2 * qc + t, nq, nk, kind, q_offset, kv_offset,
                               block_mask, causal_in_blocks, window)
        out.append((bh, qc, len(kv)))
    return out


def pair_cost(p) -> int:
    """Half-tile-squares of work of a causal chunk pair: 2 off the diagonal, 1 on it."""
    return 1 if p[0] == p[1] else 2


def chunk_pair_lanes(n_chunks: int, n_lanes: int = 0):
    """The causal (q-chunk, kv-chunk) pairs dealt to ``n_lanes`` virtual lanes
    (``n_chunks`` when ``n_lanes <= 0``): pairs sorted by (cost desc, q-chunk
    desc, kv-chunk asc), each to the least-loaded lane, lowest lane on ties.
    Returns one list of pairs per lane, in the order each lane received them."""
    if n_chunks <= 0:
        return []
    lanes = n_lanes if n_lanes > 0 else n_chunks
    pairs = [(qc, kc) for qc in range(n_chunks) for kc in range(qc + 1)]
    pairs.sort(key=lambda p: (-pair_cost(p), -p[0], p[1]))
    load = [0] * lanes
    per_lane = [[] for _ in range(lanes)]
    for p in pairs:
        best = min(range(lanes), key=lambda l: (load[l], l))
        load[best] += pair_cost(p)
        per_lane[best].append(p)
    return per_lane


def chunk_pair_schedule(n_chunks: int, n_lanes: int = 0):
    """Load-balanced order of the causal (q-chunk, kv-chunk) pairs: the lanes
    of ``chunk_pair_lanes`` emitted round-robin by position."""
    per_lane = chunk_pair_lanes(n_chunks, n_lanes)
    if not per_lane:
        return []
    lanes = len(per_lane)
    out = []
    depth = max(len(x) for x in per_lane)
    for pos in range(depth):
        for l in range(lanes):
            if pos < len(per_lane[l]):
                out.append(per_lane[l][pos])
    return out

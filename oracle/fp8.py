"""Exact attention on 8-bit floating-point (e4m3) inputs, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "FlashAttention: Fast and Memory-Efficient Exact Attention with
IO-Awareness", related papers, the FlashAttention-3 entry: attention with FP8
operands on H100.  The page gives no format or scaling, so the plain reading
is used:

* the operands are stored as E4M3 codes (the 8-bit format with 1 sign bit,
  4 exponent bits of bias 7 and 3 mantissa bits; exponent field 0 holds the
  subnormals ``m/8 * 2^-6``; exponent field 15 with mantissa 7 is NaN; no
  infinities, largest finite value 448);
* each tensor carries one per-tensor dequantisation factor: the value of a
  code ``c`` of Q is ``q_descale * e4m3(c)`` (likewise K, V);
* the attention itself is the exact one of ``attention.py`` on those values.

``fp8_row_error_bound`` states how far a kernel that feeds the softmax
weights to the second product as e4m3 (round to nearest) may fall from that
exact result, per query row; it is what the GPU tests compare against.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .attention import MaskSpec, attention_forward, visible, _group

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Float64 values of E4M3 codes (uint8 array); NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def fp8_forward(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                scale: float, mask: MaskSpec = MaskSpec(),
                heads: Optional[Sequence] = None, rows: Optional[np.ndarray] = None):
    """Exact attention of the dequantised operands: returns ``(O, LSE)`` as
    ``attention_forward`` does (same shapes, same ``heads``/``rows`` sampling).

    ``q8`` ``[B,Hq,N,d]`` and ``k8``/``v8`` ``[B,Hkv,N,d]`` are uint8 E4M3 codes.
    """
    q = q_descale * e4m3_decode(q8)
    k = k_descale * e4m3_decode(k8)
    v = v_descale * e4m3_decode(v8)
    return attention_forward(q, k, v, scale, mask, heads=heads, rows=rows)


def fp8_row_error_bound(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                        scale: float, mask: MaskSpec = MaskSpec(),
                        heads: Optional[Sequence] = None, rows: Optional[np.ndarray] = None):
    """Per query row, the largest ``max_d |O - O_exact|`` that rounding the
    softmax weights to E4M3 can cause, returned as ``[len(heads), len(rows)]``
    (``[B, Hq, N]`` without sampling).

    Let ``w_j = exp(S_ij - max_j S_ij)`` over the visible keys (so the largest
    is 1) and ``Vmax`` the largest ``|v_jd|`` over the visible keys.  The
    kernel holds each weight as ``P_j = w_j * 2^t`` with ``t >= 7`` (the
    weights are taken against a reference at or below the row max, offset by
    7 in log2 units).  Round-to-nearest E4M3 changes a normal ``P_j``
    (``>= 2^-6``, i.e. whenever ``w_j >= 2^-13``) by at most ``2^-4 P_j`` and a
    subnormal one by at most half the subnormal step, ``2^-10``, which is at
    most ``2^-17`` in units of ``w``.  Dividing by the exact row sum gives::

        |O_i - O_exact_i| <= Vmax * (2^-4 + 2^-17 * n_small / sum_j w_j)

    with ``n_small`` the number of visible keys with ``w_j < 2^-13``.  Rows
    with no visible key get 0.
    """
    q = q_descale * e4m3_decode(q8)
    k = k_descale * e4m3_decode(k8)
    v = v_descale * e4m3_decode(v8)
    B, Hq, N, _ = q.shape
    g = _group(Hq, k.shape[1])
    sample = heads is not None
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    rows = np.arange(N) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(heads), rows.size))
    for n, (b, h) in enumerate(heads):
        kk, vv = k[b, h // g], v[b, h // g]
        vis = visible(rows, kk.shape[0], mask)
        s = np.where(vis, scale * (q[b, h, rows] @ kk.T), -np.inf)
        m = s.max(axis=1)
        has = np.isfinite(m)
        w = np.exp(s - np.where(has, m, 0.0)[:, None])
        small = (vis & (w < 2.0 ** -13)).sum(axis=1)
        vabs = np.abs(vv).max(axis=1)
        vmax = np.where(vis, vabs[None, :], 0.0).max(axis=1)
        bound = vmax * (2.0 ** -4 + 2.0 ** -17 * small / np.where(has, w.sum(axis=1), 1.0))
        out[n] = np.where(has, bound, 0.0)
    if sample:
        return out
    return out.reshape(B, Hq, rows.size)

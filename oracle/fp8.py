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

``fp8_error_model`` states how far a kernel that feeds the softmax weights
to the second product as e4m3 (round to nearest) may fall from that exact
result, per output element, and how far it is expected to fall on average;
the GPU tests compare against both.
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


def fp8_error_model(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                    scale: float, mask: MaskSpec = MaskSpec(),
                    heads: Optional[Sequence] = None, rows: Optional[np.ndarray] = None):
    """Error that rounding the softmax weights to E4M3 adds to each output
    element, against the exact attention of the dequantised operands.

    Returns ``(bound, msq)``, each ``[len(heads), len(rows), d]``
    (``[B, Hq, N, d]`` without sampling): ``bound`` is the largest
    ``|O_id - O_exact_id|`` the rounding can cause, ``msq`` the expected
    squared error when the rounding errors behave as independent uniform
    variables (the usual model of round to nearest).

    The model.  Let ``w_j = exp(S_ij - max_j S_ij)`` over the visible keys (the
    largest is 1).  The weights enter the second product as
    ``P_j = w_j * 2^t`` rounded to E4M3, with ``t`` in ``[7, 8]`` (the
    reference is the running max offset by 7 in log2 units, moved once the row
    max passes it by more than 1), and the sum that normalises ``O`` is the
    exact one.  So ``O_id - O_exact_id = sum_j delta_j v_jd / sum_j w_j`` with
    ``delta_j`` the rounding error of ``P_j`` in units of ``w``:

    * a normal ``P_j`` (``>= 2^-6``, certain once ``w_j >= 2^-13``) has 3
      mantissa bits, so ``|delta_j| <= 2^-4 w_j`` and its grid step is at most
      ``2^-3 w_j``;
    * otherwise ``P_j`` falls on the subnormal grid (step ``2^-9``), so
      ``|delta_j| <= 2^-10 / 2^t <= 2^-17`` with step ``<= 2^-16``.

    Hence ``bound_id = sum_j e_j |v_jd| / sum_j w_j`` with ``e_j = 2^-4 w_j``
    (``w_j >= 2^-13``) or ``2^-17`` (below), and, with a uniform error of
    variance ``step^2 / 12``, ``msq_id = sum_j (step_j^2 / 12) v_jd^2 /
    (sum_j w_j)^2`` using the largest step of each case (so ``msq`` is an upper
    estimate, at most 4 times the mean for steps half as large).  Rows with no
    visible key get 0.
    """
    q = q_descale * e4m3_decode(q8)
    k = k_descale * e4m3_decode(k8)
    v = v_descale * e4m3_decode(v8)
    B, Hq, N, d = q.shape
    g = _group(Hq, k.shape[1])
    sample = heads is not None
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    rows = np.arange(N) if rows is None else np.asarray(rows, np.int64)
    bound = np.zeros((len(heads), rows.size, d))
    msq = np.zeros((len(heads), rows.size, d))
    for n, (b, h) in enumerate(heads):
        kk, vv = k[b, h // g], v[b, h // g]
        vis = visible(rows, kk.shape[0], mask)
        s = np.where(vis, scale * (q[b, h, rows] @ kk.T), -np.inf)
        m = s.max(axis=1)
        has = np.isfinite(m)
        w = np.exp(s - np.where(has, m, 0.0)[:, None])      # 0 on hidden keys
        normal = w >= 2.0 ** -13
        e = np.where(vis, np.where(normal, 2.0 ** -4 * w, 2.0 ** -17), 0.0)
        var = np.where(vis, np.where(normal, (2.0 ** -3 * w) ** 2, (2.0 ** -16) ** 2) / 12.0, 0.0)
        tot = np.where(has, w.sum(axis=1), 1.0)[:, None]
        bound[n] = np.where(has[:, None], (e @ np.abs(vv)) / tot, 0.0)
        msq[n] = np.where(has[:, None], (var @ (vv * vv)) / (tot * tot), 0.0)
    if sample:
        return bound, msq
    return bound.reshape(B, Hq, rows.size, d), msq.reshape(B, Hq, rows.size, d)

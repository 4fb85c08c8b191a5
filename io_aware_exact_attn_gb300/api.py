"""PyTorch-facing wrappers over the C ABI (argument marshalling only).

Every function checks shapes, dtypes and layouts, allocates outputs with
torch (device memory is torch's), and calls one entry point of ``libattn.so``
on the current CUDA stream.  All arithmetic happens in the library's kernels.
"""
from __future__ import annotations

import ctypes as C
import math
from typing import Optional, Sequence

import numpy as np
import torch

from . import _ffi
from ._ffi import attn_mask_t, check

__all__ = ["attn_fwd", "attn_fwd_fp8", "fwd_fp8_workspace_bytes", "attn_partial_fwd", "attn_merge_lse", "attn_bwd",
           "bwd_workspace_bytes", "attn_bwd_preprocess", "attn_partial_bwd", "chunked_fwd", "chunked_bwd",
           "build_schedule", "build_chunk_schedule", "get_status", "set_wait_limit_ns",
           "selftest_wait_timeout", "mask_desc", "trace_enable", "trace_disable", "trace_read"]


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _rows_view(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    """Check a [B, H, N, d] tensor whose rows are contiguous; return its head stride in rows."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, N, d]")
    B, H, N, d = t.shape
    if t.stride(3) != 1 or (N > 1 and t.stride(2) != d):
        raise ValueError(f"{name}: rows must be contiguous with stride d")
    if B * H == 1:
        return N          # one head: no stride between heads to honour
    if t.stride(1) % d or t.stride(1) // d < N or (B > 1 and t.stride(0) != H * t.stride(1)):
        raise ValueError(f"{name}: heads must be evenly strided")
    return t.stride(1) // d


def _contig(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def mask_desc(causal: bool = False, block_mask: Optional[torch.Tensor] = None,
              causal_in_blocks: bool = False, window: Optional[int] = None):
    """Build the C mask descriptor; returns (descriptor or None, tensor to keep alive).

    ``window`` selects the sliding-window mask: a query sees itself and the
    ``window - 1`` positions before it (causal implied).
    """
    if window is not None:
        if block_mask is not None:
            raise ValueError("a sliding window and a block mask do not combine")
        if int(window) < 1:
            raise ValueError("window must be >= 1")
        return attn_mask_t(_ffi.MASK_SLIDING_WINDOW, 0, None, int(window)), None
    if block_mask is not None:
        bm = block_mask
        if bm.dtype != torch.uint8:
            bm = bm.to(torch.uint8)
        bm = bm.contiguous()
        if not bm.is_cuda:
            raise ValueError("block_mask must be on the GPU")
        m = attn_mask_t(_ffi.MASK_BLOCK_SPARSE, 1 if causal_in_blocks else 0, bm.data_ptr(), 0)
        return m, bm
    if causal:
        return attn_mask_t(_ffi.MASK_CAUSAL, 0, None, 0), None
    return None, None


def _mp(m):
    return C.byref(m) if m is not None else None


def attn_fwd(q, k, v, scale: Optional[float] = None, causal: bool = False,
             block_mask: Optional[torch.Tensor] = None, causal_in_blocks: bool = False,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             window: Optional[int] = None):
    """Exact attention forward: returns ``(O [B,Hq,N,d] bf16, LSE [B,Hq,N] f32)``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _contig(t, n)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    o = torch.empty_like(q) if out is None else out
    _contig(o, "out")
    l = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32) if lse is None else lse
    _contig(l, "lse", torch.float32)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, block_mask, causal_in_blocks, window)
    check(_ffi.lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                              B, Hq, Hkv, N, d, sc, _mp(m), _stream(q)), "attn_fwd")
    del keep
    return o, l


def fwd_fp8_workspace_bytes(B: int, Hkv: int, N: int, d: int = 128) -> int:
    return int(_ffi.lib().attn_fwd_fp8_workspace_bytes(B, Hkv, N, d))


def _e4m3(t: torch.Tensor, name: str):
    """Accept float8_e4m3fn or uint8 (raw E4M3 codes) contiguous CUDA tensors."""
    if not (t.is_cuda and t.dtype in (torch.float8_e4m3fn, torch.uint8) and t.is_contiguous() and t.dim() == 4):
        raise ValueError(f"{name} must be a contiguous CUDA float8_e4m3fn (or uint8 code) [B, H, N, d] tensor")


def attn_fwd_fp8(q8, k8, v8, q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                 scale: Optional[float] = None, causal: bool = False, block_mask: Optional[torch.Tensor] = None,
                 causal_in_blocks: bool = False, window: Optional[int] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None):
    """Forward on E4M3 operands: ``O = softmax(scale (qd Q8)(kd K8)^T) (vd V8)``.

    Returns ``(O [B,Hq,N,d] bf16, LSE [B,Hq,N] f32)``; ``d`` must be 128.
    ``workspace`` (uint8, >= ``fwd_fp8_workspace_bytes``) receives V^T.
    """
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _e4m3(t, n)
    B, Hq, N, d = q8.shape
    Hkv = k8.shape[1]
    if k8.shape != (B, Hkv, N, d) or v8.shape != k8.shape:
        raise ValueError("k8 and v8 must be [B, Hkv, N, d] matching q8")
    o = torch.empty((B, Hq, N, d), device=q8.device, dtype=torch.bfloat16) if out is None else out
    _contig(o, "out")
    l = torch.empty((B, Hq, N), device=q8.device, dtype=torch.float32) if lse is None else lse
    _contig(l, "lse", torch.float32)
    need = fwd_fp8_workspace_bytes(B, Hkv, N, d)
    ws = torch.empty(max(need, 16), device=q8.device, dtype=torch.uint8) if workspace is None else workspace
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, block_mask, causal_in_blocks, window)
    check(_ffi.lib().attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), float(q_descale), float(k_descale),
                                  float(v_descale), o.data_ptr(), l.data_ptr(), B, Hq, Hkv, N, d, sc, _mp(m),
                                  ws.data_ptr(), ws.numel() * ws.element_size(), _stream(q8)), "attn_fwd_fp8")
    del keep
    return o, l


def attn_partial_fwd(q, k, v, q_offset: int = 0, kv_offset: int = 0, scale: Optional[float] = None,
                     causal: bool = False, block_mask: Optional[torch.Tensor] = None,
                     causal_in_blocks: bool = False, o_part: Optional[torch.Tensor] = None,
                     lse_part: Optional[torch.Tensor] = None, window: Optional[int] = None):
    """Attention of one query chunk against one key/value chunk.

    ``q`` ``[B,Hq,Nq,d]`` and ``k``/``v`` ``[B,Hkv,Nk,d]`` may be row-slices of
    larger tensors (rows contiguous, heads evenly strided).  Returns the fp32
    partial ``O_c [B,Hq,Nq,d]`` normalised over this chunk's keys and
    ``LSE_c [B,Hq,Nq]``.
    """
    qhs = _rows_view(q, "q")
    khs = _rows_view(k, "k")
    vhs = _rows_view(v, "v")
    if vhs != khs or v.shape != k.shape or k.stride() != v.stride():
        raise ValueError("k and v must share shape and strides")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = torch.empty((B, Hq, Nq, d), device=q.device, dtype=torch.float32) if o_part is None else o_part
    l = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32) if lse_part is None else lse_part
    _contig(o, "o_part", torch.float32)
    _contig(l, "lse_part", torch.float32)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, block_mask, causal_in_blocks, window)
    check(_ffi.lib().attn_partial_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                                      B, Hq, Hkv, Nq, Nk, d, sc, _mp(m), int(q_offset), int(kv_offset),
                                      qhs, khs, _stream(q)), "attn_partial_fwd")
    del keep
    return o, l


def attn_merge_lse(o_parts: Sequence[torch.Tensor], lse_parts: Sequence[torch.Tensor],
                   out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                   lse_out: Optional[torch.Tensor] = None):
    """Log-sum-exp merge of partial results over disjoint key sets.

    ``out`` (and ``lse_out``) may be row-slices of larger tensors with the same
    head stride.  Returns ``(O, LSE)``.
    """
    n = len(o_parts)
    if n != len(lse_parts) or n < 1:
        raise ValueError("need matching, non-empty part lists")
    for i, (o, l) in enumerate(zip(o_parts, lse_parts)):
        _contig(o, f"o_parts[{i}]", torch.float32)
        _contig(l, f"lse_parts[{i}]", torch.float32)
    B, Hq, Nq, d = o_parts[0].shape
    for o in o_parts:
        if o.shape != (B, Hq, Nq, d):
            raise ValueError("all parts must share one shape")
    dt = out.dtype if out is not None else out_dtype
    o_out = torch.empty((B, Hq, Nq, d), device=o_parts[0].device, dtype=dt) if out is None else out
    hs = _rows_view(o_out, "out", dt)
    l_out = torch.empty((B, Hq, Nq), device=o_parts[0].device, dtype=torch.float32) if lse_out is None else lse_out
    if l_out.dtype != torch.float32 or l_out.stride(-1) != 1 or (Hq > 1 and l_out.stride(1) != hs):
        raise ValueError("lse_out must be f32 with the same head stride (in rows) as out")
    optrs = (C.c_void_p * n)(*[o.data_ptr() for o in o_parts])
    lptrs = (C.c_void_p * n)(*[l.data_ptr() for l in lse_parts])
    code = _ffi.DTYPE_F32 if dt == torch.float32 else _ffi.DTYPE_BF16
    check(_ffi.lib().attn_merge_lse(optrs, lptrs, n, o_out.data_ptr(), code, l_out.data_ptr(), B, Hq, Nq, d, hs,
                                    _stream(o_parts[0])), "attn_merge_lse")
    return o_out, l_out


def bwd_workspace_bytes(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(_ffi.lib().attn_bwd_workspace_bytes(B, Hq, Hkv, N, d))


def attn_bwd(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False,
             block_mask: Optional[torch.Tensor] = None, causal_in_blocks: bool = False,
             workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None,
             window: Optional[int] = None):
    """Exact backward pass; returns ``(dQ, dK, dV)`` in bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _contig(t, n)
    _contig(lse, "lse", torch.float32)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    need = bwd_workspace_bytes(B, Hq, Hkv, N, d)
    ws = torch.empty(need, device=q.device, dtype=torch.uint8) if workspace is None else workspace
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, block_mask, causal_in_blocks, window)
    check(_ffi.lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                              ws.numel() * ws.element_size(), B, Hq, Hkv, N, d, sc, _mp(m), _stream(q)),
          "attn_bwd")
    del keep
    return dq, dk, dv


def attn_bwd_preprocess(o, lse, do, workspace: Optional[torch.Tensor] = None):
    """Backward step 1 for one query chunk: ``D = rowsum(dO * O)`` and ``LSE * log2 e``.

    ``o``, ``do`` ``[B,Hq,Nq,d]`` bf16 and ``lse`` ``[B,Hq,Nq]`` f32 may be
    row-slices of longer tensors (rows contiguous, one head stride for all
    three).  Pass the MERGED O and LSE of the chunk.  Returns the workspace
    (uint8) that ``attn_partial_bwd`` reads.
    """
    hs = _rows_view(o, "o")
    if _rows_view(do, "do") != hs or do.shape != o.shape:
        raise ValueError("do must match o's shape and head stride")
    B, Hq, Nq, d = o.shape
    if (lse.dtype != torch.float32 or not lse.is_cuda or lse.shape != (B, Hq, Nq) or lse.stride(-1) != 1
            or (Hq > 1 and lse.stride(1) != hs) or (B > 1 and lse.stride(0) != Hq * hs)):
        raise ValueError("lse must be f32 [B, Hq, Nq] with o's head stride (in rows)")
    need = bwd_workspace_bytes(B, Hq, Hq, Nq, d)
    ws = torch.empty(need, device=o.device, dtype=torch.uint8) if workspace is None else workspace
    check(_ffi.lib().attn_bwd_preprocess(o.data_ptr(), do.data_ptr(), lse.data_ptr(), B, Hq, Nq, d, hs,
                                         ws.data_ptr(), ws.numel() * ws.element_size(), _stream(o)),
          "attn_bwd_preprocess")
    return ws


def attn_partial_bwd(q, k, v, do, workspace, dq, dk, dv, q_offset: int = 0, kv_offset: int = 0,
                     scale: Optional[float] = None, causal: bool = False,
                     block_mask: Optional[torch.Tensor] = None, causal_in_blocks: bool = False,
                     window: Optional[int] = None, accumulate: bool = True):
    """Gradient terms of one (query chunk, key/value chunk) pair, added to
    (``accumulate``) or stored in the float32 ``dq`` (q's shape and head
    stride) and ``dk``/``dv`` (k's).  ``workspace`` is the query chunk's
    ``attn_bwd_preprocess`` output.  ``q``/``do`` and ``k``/``v`` may be
    row-slices of longer tensors."""
    qhs = _rows_view(q, "q")
    khs = _rows_view(k, "k")
    if _rows_view(v, "v") != khs or v.shape != k.shape or _rows_view(do, "do") != qhs or do.shape != q.shape:
        raise ValueError("v must match k, do must match q (shape and head stride)")
    if _rows_view(dq, "dq", torch.float32) != qhs or dq.shape != q.shape:
        raise ValueError("dq must be f32 with q's shape and head stride")
    for t, n in ((dk, "dk"), (dv, "dv")):
        if _rows_view(t, n, torch.float32) != khs or t.shape != k.shape:
            raise ValueError(f"{n} must be f32 with k's shape and head stride")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, block_mask, causal_in_blocks, window)
    check(_ffi.lib().attn_partial_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(), dq.data_ptr(), dk.data_ptr(),
                                      dv.data_ptr(), B, Hq, Hkv, Nq, Nk, d, sc, _mp(m), int(q_offset),
                                      int(kv_offset), qhs, khs, 1 if accumulate else 0, _stream(q)),
          "attn_partial_bwd")
    del keep
    return dq, dk, dv


def _chunk_pairs(n_chunks: int, causal: bool):
    if causal:
        return build_chunk_schedule(n_chunks)
    return [(a, b) for a in range(n_chunks) for b in range(n_chunks)]


def chunked_fwd(q, k, v, n_chunks: int, scale: Optional[float] = None, causal: bool = True,
                window: Optional[int] = None):
    """Attention of ``q``, ``k``, ``v`` ``[B,H,N,d]`` cut into ``n_chunks`` equal
    sequence chunks, the way chunked (sequence-parallel) attention runs it on
    one GPU: every visible (query chunk, key chunk) pair with
    ``attn_partial_fwd`` (under a causal or sliding-window mask the pairs with
    key chunk <= query chunk, in the load-balanced order of
    ``build_chunk_schedule``), then one ``attn_merge_lse`` per query chunk.
    Returns ``(O bf16, LSE f32)`` of the whole sequence."""
    B, Hq, N, d = q.shape
    if N % n_chunks:
        raise ValueError("N must be a multiple of n_chunks")
    L = N // n_chunks
    local = causal or window is not None
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32)
    parts = {}
    for qc, kc in _chunk_pairs(n_chunks, local):
        parts[(qc, kc)] = attn_partial_fwd(q[:, :, qc * L:(qc + 1) * L], k[:, :, kc * L:(kc + 1) * L],
                                           v[:, :, kc * L:(kc + 1) * L], qc * L, kc * L, scale=scale,
                                           causal=causal and window is None, window=window)
    for qc in range(n_chunks):
        kcs = [kc for kc in range(n_chunks) if (qc, kc) in parts]
        attn_merge_lse([parts[(qc, kc)][0] for kc in kcs], [parts[(qc, kc)][1] for kc in kcs],
                       out=o[:, :, qc * L:(qc + 1) * L], lse_out=lse[:, :, qc * L:(qc + 1) * L])
    return o, lse


def chunked_bwd(q, k, v, o, lse, do, n_chunks: int, scale: Optional[float] = None, causal: bool = True,
                window: Optional[int] = None, n_streams: int = 1, dq=None, dk=None, dv=None):
    """Backward pass of ``chunked_fwd``: one ``attn_bwd_preprocess`` per query
    chunk (with the merged ``o`` and ``lse``), then ``attn_partial_bwd`` of
    every visible chunk pair, in the load-balanced order, adding into float32
    ``dq``, ``dk``, ``dv`` (zeroed here unless given).  With ``n_streams`` > 1
    the pairs are dealt round-robin to that many side streams (the float32
    reductions make concurrent pairs safe); the current stream waits for all
    of them.  Returns ``(dQ, dK, dV)`` in float32."""
    B, Hq, N, d = q.shape
    if N % n_chunks:
        raise ValueError("N must be a multiple of n_chunks")
    L = N // n_chunks
    local = causal or window is not None
    dq = torch.zeros(q.shape, device=q.device, dtype=torch.float32) if dq is None else dq
    dk = torch.zeros(k.shape, device=q.device, dtype=torch.float32) if dk is None else dk
    dv = torch.zeros(v.shape, device=q.device, dtype=torch.float32) if dv is None else dv
    ws = [attn_bwd_preprocess(o[:, :, c * L:(c + 1) * L], lse[:, :, c * L:(c + 1) * L], do[:, :, c * L:(c + 1) * L])
          for c in range(n_chunks)]
    main = torch.cuda.current_stream(q.device)
    streams = [main] if n_streams <= 1 else [torch.cuda.Stream(q.device) for _ in range(n_streams)]
    if n_streams > 1:
        ready = torch.cuda.Event()
        ready.record(main)
        for st in streams:
            st.wait_event(ready)
    for i, (qc, kc) in enumerate(_chunk_pairs(n_chunks, local)):
        qs, ks = slice(qc * L, (qc + 1) * L), slice(kc * L, (kc + 1) * L)
        with torch.cuda.stream(streams[i % len(streams)]):
            attn_partial_bwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], do[:, :, qs], ws[qc], dq[:, :, qs],
                             dk[:, :, ks], dv[:, :, ks], qc * L, kc * L, scale=scale,
                             causal=causal and window is None, window=window, accumulate=True)
    if n_streams > 1:
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            main.wait_event(ev)
        for t in ws + [dq, dk, dv, q, k, v, do]:
            for st in streams:
                t.record_stream(st)
    return dq, dk, dv


def attn_varlen_fwd(q, k, v, cu_seqlens: torch.Tensor, max_len: Optional[int] = None,
                    scale: Optional[float] = None, causal: bool = False, window: Optional[int] = None,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Forward over sequences of different lengths packed back to back.

    ``q`` ``[total, Hq, d]``, ``k``/``v`` ``[total, Hkv, d]`` (token-major);
    ``cu_seqlens`` int32 ``[B + 1]`` token offsets (on the GPU).  Returns
    ``(O [total, Hq, d] bf16, LSE [Hq, total] f32)``.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3):
            raise ValueError(f"{n} must be a contiguous CUDA bf16 [total, heads, d] tensor")
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (total, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [total, Hkv, d] matching q")
    cu = cu_seqlens.to(device=q.device, dtype=torch.int32).contiguous()
    B = cu.numel() - 1
    if B < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    if max_len is None:
        max_len = int((cu[1:] - cu[:-1]).max().item())
    o = torch.empty_like(q) if out is None else out
    _contig(o, "out")
    l = torch.empty((Hq, total), device=q.device, dtype=torch.float32) if lse is None else lse
    _contig(l, "lse", torch.float32)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, None, False, window)
    check(_ffi.lib().attn_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                                     cu.data_ptr(), B, int(max_len), int(total), Hq, Hkv, d, sc, _mp(m), _stream(q)),
          "attn_varlen_fwd")
    del keep
    return o, l


def varlen_bwd_workspace_bytes(B: int, total: int, Hq: int) -> int:
    return int(_ffi.lib().attn_varlen_bwd_workspace_bytes(B, int(total), Hq))


def attn_varlen_bwd(q, k, v, o, lse, do, cu_seqlens: torch.Tensor, max_len: Optional[int] = None,
                    scale: Optional[float] = None, causal: bool = False, window: Optional[int] = None,
                    workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None):
    """Backward of ``attn_varlen_fwd``: returns ``(dQ [total,Hq,d], dK, dV [total,Hkv,d])`` in bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3):
            raise ValueError(f"{n} must be a contiguous CUDA bf16 [total, heads, d] tensor")
    _contig(lse, "lse", torch.float32)
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = cu_seqlens.to(device=q.device, dtype=torch.int32).contiguous()
    B = cu.numel() - 1
    if max_len is None:
        max_len = int((cu[1:] - cu[:-1]).max().item())
    need = varlen_bwd_workspace_bytes(B, total, Hq)
    ws = torch.empty(need, device=q.device, dtype=torch.uint8) if workspace is None else workspace
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m, keep = mask_desc(causal, None, False, window)
    check(_ffi.lib().attn_varlen_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu.data_ptr(), B,
                                     int(max_len), int(total), Hq, Hkv, d, sc, _mp(m), ws.data_ptr(),
                                     ws.numel() * ws.element_size(), _stream(q)), "attn_varlen_bwd")
    del keep
    return dq, dk, dv


def decode_splits(B: int, Hkv: int, Nk: int) -> int:
    return int(_ffi.lib().attn_decode_splits(B, Hkv, Nk))


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, n_splits: int = 0) -> int:
    return int(_ffi.lib().attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, n_splits))


def attn_decode(q, k_cache, v_cache, seq_lens: Optional[torch.Tensor] = None, causal: bool = True,
                scale: Optional[float] = None, n_splits: int = 0, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """One decoding step against a KV cache, split over the cache.

    ``q`` ``[B, Hq, Nq, d]`` holds the newest ``Nq`` positions of each
    sequence; ``k_cache``/``v_cache`` ``[B, Hkv, Nk, d]`` of which sequence ``b``
    uses the first ``seq_lens[b]`` positions (int32 CUDA tensor, or None for
    all ``Nk``).  Returns ``(O [B,Hq,Nq,d] bf16, LSE [B,Hq,Nq] f32)``.
    """
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _contig(t, n)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Hkv, Nk, d) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must be [B, Hkv, Nk, d] matching q")
    sl = None
    if seq_lens is not None:
        sl = seq_lens.to(device=q.device, dtype=torch.int32).contiguous()
        if sl.shape != (B,):
            raise ValueError("seq_lens must have shape [B]")
    o = torch.empty_like(q) if out is None else out
    _contig(o, "out")
    l = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32) if lse is None else lse
    _contig(l, "lse", torch.float32)
    need = decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, n_splits)
    ws = torch.empty(need, device=q.device, dtype=torch.uint8) if workspace is None else workspace
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(_ffi.lib().attn_decode_fwd(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     sl.data_ptr() if sl is not None else None, o.data_ptr(), l.data_ptr(),
                                     B, Hq, Hkv, Nq, Nk, d, sc, 1 if causal else 0, int(n_splits),
                                     ws.data_ptr(), ws.numel() * ws.element_size(), _stream(q)), "attn_decode_fwd")
    return o, l


def build_schedule(mask_kind: int, B: int, Hq: int, Nq: int, Nk: int, q_offset: int = 0,
                   kv_offset: int = 0, host_block_mask: Optional[np.ndarray] = None,
                   causal_in_blocks: bool = False, Hkv: Optional[int] = None, d: int = 128,
                   window: int = 0) -> np.ndarray:
    """Forward work units in launch order, ``[n, 3]`` int32 (bh, query chunk, key tiles)."""
    L = _ffi.lib()
    hkv = Hq if Hkv is None else Hkv
    n = C.c_size_t(0)
    bm = None
    if host_block_mask is not None:
        bm = np.ascontiguousarray(host_block_mask, dtype=np.uint8)
    bmp = bm.ctypes.data if bm is not None else None
    L.attn_build_schedule(mask_kind, int(causal_in_blocks), bmp, int(window), B, Hq, hkv, Nq, Nk, d, q_offset,
                          kv_offset, None, 0, C.byref(n))
    out = np.zeros(3 * n.value, dtype=np.int32)
    check(L.attn_build_schedule(mask_kind, int(causal_in_blocks), bmp, int(window), B, Hq, hkv, Nq, Nk, d,
                                q_offset, kv_offset, out.ctypes.data_as(C.POINTER(C.c_int32)), out.size,
                                C.byref(n)),
          "attn_build_schedule")
    return out.reshape(-1, 3)


def build_chunk_schedule(n_chunks: int, n_lanes: int = 0):
    """Load-balanced order of causal (q-chunk, kv-chunk) pairs."""
    L = _ffi.lib()
    n = C.c_size_t(0)
    L.attn_build_chunk_schedule(n_chunks, n_lanes, None, 0, C.byref(n))
    out = np.zeros(2 * n.value, dtype=np.int32)
    check(L.attn_build_chunk_schedule(n_chunks, n_lanes, out.ctypes.data_as(C.POINTER(C.c_int32)), out.size,
                                      C.byref(n)), "attn_build_chunk_schedule")
    return [tuple(int(x) for x in p) for p in out.reshape(-1, 2)]


def get_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    s = torch.cuda.current_stream(device).cuda_stream
    return int(_ffi.lib().attn_get_status(s))


def set_wait_limit_ns(limit_ns: int) -> None:
    _ffi.lib().attn_set_wait_limit_ns(int(limit_ns))


def debug_set_tile_counts(counts=None) -> None:
    """Record, per CTA of every later launch, the work it did (8 int32 per CTA,
    fields as attn.h lists them) into ``counts``, a contiguous int32 CUDA
    tensor; ``None`` turns recording off.  The caller keeps ``counts`` alive
    while recording is on."""
    if counts is None:
        check(_ffi.lib().attn_debug_set_tile_counts(None, 0), "attn_debug_set_tile_counts")
        return
    if counts.dtype != torch.int32 or not counts.is_cuda or not counts.is_contiguous():
        raise ValueError("counts must be a contiguous int32 CUDA tensor")
    check(_ffi.lib().attn_debug_set_tile_counts(counts.data_ptr(), counts.numel()), "attn_debug_set_tile_counts")


def selftest_wait_timeout(limit_ns: int, device=None) -> None:
    s = torch.cuda.current_stream(device).cuda_stream
    check(_ffi.lib().attn_selftest_wait_timeout(int(limit_ns), s), "attn_selftest_wait_timeout")


def trace_enable(capacity: int = 4096) -> None:
    """Record CUDA events around every kernel the library launches from now on."""
    check(_ffi.lib().attn_trace_enable(int(capacity)), "attn_trace_enable")


def trace_disable() -> None:
    _ffi.lib().attn_trace_disable()


def trace_read(capacity: int = 1 << 16):
    """Return ``(records, n_launched)``: records are ``(kernel_name, ms)`` in launch order."""
    buf = (_ffi.attn_trace_record_t * capacity)()
    n = C.c_int(0)
    check(_ffi.lib().attn_trace_read(buf, capacity, C.byref(n)), "attn_trace_read")
    recs = [(_ffi.KERNEL_NAMES.get(buf[i].kernel, str(buf[i].kernel)), float(buf[i].ms))
            for i in range(min(n.value, capacity))]
    return recs, n.value

"""Helpers shared by the GPU parity tests (seeded inputs, oracle comparison)."""
import numpy as np
import torch

import oracle
from io_aware_exact_attn_gb300 import inputs

# tolerances for bf16 inputs with fp32 accumulation
O_ATOL = 1e-2          # max |O_gpu - O_ref|
LSE_ATOL = 2e-3        # max |LSE_gpu - LSE_ref|
GRAD_RTOL = 3e-2       # max |g_gpu - g_ref| <= GRAD_RTOL * max |g_ref|


def make(B, Hq, Hkv, N, d, seed=inputs.SEED, k_mul=1.0, Nk=None):
    q, k, v, do = inputs.make_qkvdo(B, Hq, Hkv, N, N if Nk is None else Nk, d, seed, k_mul)
    return [t.cuda() for t in (q, k, v, do)]


def f64(t):
    return inputs.to_f64(t)


def mask_spec(kind, bm=None, cib=False, window=0):
    if kind == "block_sparse":
        return oracle.MaskSpec("block_sparse", np.asarray(bm, bool), 128, cib)
    if kind == "sliding_window":
        return oracle.MaskSpec("sliding_window", window=window)
    return oracle.MaskSpec(kind)


def max_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0


def assert_o_lse(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    eo = max_err(o_gpu, o_ref)
    el = max_err(lse_gpu, lse_ref)
    assert eo <= O_ATOL, f"{what} O max-abs error {eo:.3e} > {O_ATOL}"
    assert el <= LSE_ATOL, f"{what} LSE max-abs error {el:.3e} > {LSE_ATOL}"
    return eo, el


ZERO_GRAD_ATOL = 1e-4  # when the exact gradient is identically 0 (e.g. one key)


def assert_grad(g_gpu, g_ref, what=""):
    ref = np.asarray(g_ref, np.float64)
    scale = float(np.abs(ref).max())
    if scale == 0.0:
        e = max_err(g_gpu, ref)
        assert e <= ZERO_GRAD_ATOL, f"{what} max error {e:.3e} against an exactly-zero gradient"
        return e
    e = max_err(g_gpu, ref) / scale
    assert e <= GRAD_RTOL, f"{what} relative max error {e:.3e} > {GRAD_RTOL}"
    return e

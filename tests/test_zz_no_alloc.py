"""attn_bwd_static_scratch: the backward pass for callers that cannot allocate
device memory (for example code that runs under an allocator or runtime that
owns every device allocation, or a process whose memory was reserved up
front).  It runs the same kernels as attn_bwd on the same inputs, so it must
give bit-identical dQ, dK and dV, including when it is called twice in a row
and the second call reuses the one static scratch area; a wait that runs out
in it would show in attn_get_status, which reads the one status word every
entry point reports to.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test."""
import ctypes as C

import pytest
import torch

from io_aware_exact_attn_gb300 import _ffi, api
from _gpu_helpers import assert_grad, f64, make


def test_static_scratch_rejects_oversized_problem_without_a_gpu():
    lib = _ffi.lib()
    p = C.c_void_p(4096)
    # 2 * 32 * 65536 query rows = 2^22 > 2^20: refused before any device work
    rc = lib.attn_bwd_static_scratch(p, p, p, p, p, p, p, p, p, 2, 32, 32, 65536, 128, 0.088, None, None)
    assert rc == -6
    assert b"static scratch" in lib.attn_last_error_message()


@pytest.mark.gpu
def test_static_scratch_backward_matches_attn_bwd(cuda_lib):
    lib = cuda_lib
    cases = [(1, 4, 2, 700, 128, True), (2, 2, 2, 384, 64, False)]   # two calls in a row
    for B, Hq, Hkv, N, d, causal in cases:
        q, k, v, do = make(B, Hq, Hkv, N, d)
        o, lse = api.attn_fwd(q, k, v, causal=causal)
        ref = api.attn_bwd(q, k, v, o, lse, do, causal=causal)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        m, _ = api.mask_desc(causal=causal)
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.attn_bwd_static_scratch(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N,
                                         d, 1.0 / d ** 0.5, C.byref(m) if m is not None else None, stream)
        assert rc == 0, lib.attn_last_error_message()
        torch.cuda.synchronize()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.equal(got, want), f"{name} B{B} H{Hq}/{Hkv} N{N} d{d}"
            assert_grad(f64(got), f64(want), f"{name} B{B} H{Hq}/{Hkv} N{N} d{d}")
        assert api.get_status() == 0


@pytest.mark.gpu
def test_static_scratch_at_its_row_limit(cuda_lib):
    """The largest call the static scratch takes (B*Hq*ceil(N/128)*128 = 2^20
    query rows, so the statistics operand ends at the array's last byte) gives
    the same gradients as attn_bwd; one row tile more is refused."""
    lib = cuda_lib
    B, Hq, Hkv, N, d = 1, 16, 4, 65536, 64
    q, k, v, do = make(B, Hq, Hkv, N, d)
    o, lse = api.attn_fwd(q, k, v, causal=True)
    ref = api.attn_bwd(q, k, v, o, lse, do, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    m, _ = api.mask_desc(causal=True)
    stream = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr())
    rc = lib.attn_bwd_static_scratch(*args, B, Hq, Hkv, N, d, 1.0 / d ** 0.5, C.byref(m), stream)
    assert rc == 0, lib.attn_last_error_message()
    torch.cuda.synchronize()
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert torch.equal(got, want), name
    assert api.get_status() == 0
    # 2^20 + 128 rows: refused before any device work
    rc = lib.attn_bwd_static_scratch(*args, B, Hq, Hkv, N + 8, d, 1.0 / d ** 0.5, C.byref(m), stream)
    assert rc == -6

"""Exact attention for GB300 (sm_103a): a C-ABI CUDA library plus thin PyTorch bindings.

The compute path is ``libattn.so`` (hand-written tcgen05/TMA kernels); this
package only marshals arguments.  If the library has not been built, every
entry point raises.
"""
from .api import (  # noqa: F401
    attn_fwd,
    attn_fwd_fp8,
    fwd_fp8_workspace_bytes,
    attn_partial_fwd,
    attn_merge_lse,
    attn_bwd,
    bwd_workspace_bytes,
    build_schedule,
    build_chunk_schedule,
    get_status,
    set_wait_limit_ns,
    selftest_wait_timeout,
    mask_desc,
    trace_enable,
    trace_disable,
    trace_read,
)

__version__ = "0.1.0"

"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library under ``io_aware_exact_attn_gb300/``.

What it computes is the plain definition of exact attention,
``O = softmax(scale * Q K^T) V`` with the per-row log-sum-exp, its exact
gradient, and the log-sum-exp merge of partial results, written out with full
``N x N`` score matrices in float64 (no online softmax, no tiling over keys).
Sources, by page and section:

* DISTFLASHATTN reviews (arXiv 2310.03294), first review summary: attention is
  ``softmax(QK^T) V``; the backward pass needs no stored ``N x N`` matrix.
* FlashAttention: Fast and Memory-Efficient Exact Attention with IO-Awareness,
  abstract: the method is *exact* attention; block-sparse attention is the
  same computation with a block mask.
* FlashAttention-2 reviews, second review, items 1-2: deferred rescaling and
  a saved log-sum-exp per row; first review, questions: online-softmax
  equations and the GQA paragraph of the backward section.
* BurstAttention author responses: local attention results are combined
  across devices with online-softmax statistics (the merge); sparse attention
  only changes the attention mask matrix.
* FlashAttention (IO-Awareness) page, related papers, FlashAttention-3:
  attention on FP8 operands (``fp8.py``: E4M3 codes with per-tensor scales).

Every function here is pinned by tests in ``tests/test_oracle_pins.py`` to
something other than itself (closed forms, finite differences, library
softmax, invariants).  No function is "parity unpinned".
"""
from .attention import (  # noqa: F401
    MaskSpec,
    visible,
    head_forward,
    head_backward,
    attention_forward,
    attention_backward,
    attention_backward_dq_rows,
    partial_backward,
    decode_forward,
    varlen_forward,
    varlen_backward,
    merge_partials,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_decode,
    fp8_forward,
    fp8_error_model,
)
from .schedule import (  # noqa: F401
    chunk_pair_lanes,
    chunk_pair_schedule,
    fwd_work_units,
    kv_tile_range_causal,
)

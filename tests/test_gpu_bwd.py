"""GPU backward parity: attn_bwd through the C ABI against the fp64 oracle's
exact gradient on the same seeded bf16 inputs (O and LSE from attn_fwd)."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_grad, assert_o_lse, f64, make, mask_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def run(B, Hq, Hkv, N, d, kind, bm=None, cib=False, k_mul=1.0):
    q, k, v, do = make(B, Hq, Hkv, N, d, k_mul=k_mul)
    bmt = torch.as_tensor(bm, dtype=torch.uint8).cuda() if bm is not None else None
    causal = kind == "causal"
    o, lse = api.attn_fwd(q, k, v, causal=causal, block_mask=bmt, causal_in_blocks=cib)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do, causal=causal, block_mask=bmt, causal_in_blocks=cib)
    torch.cuda.synchronize()
    return (q, k, v, do), (dq, dk, dv)


def check_full(B, Hq, Hkv, N, d, kind, bm=None, cib=False, k_mul=1.0):
    (q, k, v, do), (dq, dk, dv) = run(B, Hq, Hkv, N, d, kind, bm, cib, k_mul)
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), 1 / np.sqrt(d),
                                           mask_spec(kind, bm, cib))
    tag = f"{kind} B{B} H{Hq}/{Hkv} N{N} d{d}"
    return (assert_grad(f64(dq), gq, "dQ " + tag), assert_grad(f64(dk), gk, "dK " + tag),
            assert_grad(f64(dv), gv, "dV " + tag))


@pytest.mark.parametrize("kind", ["none", "causal"])
def test_tiny_exact_attention_grad(kind):
    check_full(1, 2, 2, 128, 64, kind)


SHAPES = [
    (1, 2, 2, 300, 64, "none"), (1, 2, 2, 300, 128, "causal"), (2, 4, 2, 520, 128, "causal"),
    (1, 3, 1, 129, 64, "causal"), (1, 1, 1, 1, 128, "none"), (1, 1, 1, 1, 64, "causal"),
    (1, 2, 2, 1000, 64, "none"), (1, 2, 1, 777, 128, "causal"), (1, 4, 1, 256, 64, "none"),
    (2, 2, 2, 384, 128, "none"), (1, 2, 2, 17, 128, "causal"),
    (1, 8, 1, 300, 128, "causal"),   # dK/dV sum over eight query heads
    (2, 12, 3, 200, 64, "none"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_H{}-{}_N{}_d{}_{}".format(*s))
def test_bwd_shapes(shape):
    check_full(*shape)


def test_bwd_peaked_rows():
    check_full(1, 2, 2, 640, 128, "causal", k_mul=4.0)
    check_full(1, 2, 2, 500, 64, "none", k_mul=4.0)


@pytest.mark.parametrize("cib", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_block_sparse(cib, d):
    N = 900
    nb = -(-N // 128)
    bm = inputs.block_sparse_mask(nb, nb, 0.3, seed=11)
    check_full(1, 2, 2, N, d, "block_sparse", bm, cib)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_empty_block_row_and_column(d):
    """A query tile that sees no key tile (its dQ rows, staged at d = 128 where
    its Q copy lands, are 0) and a key tile nobody sees (dK, dV = 0)."""
    N = 512
    bm = np.ones((4, 4), bool)
    bm[1, :] = False          # rows 128..255 see nothing
    bm[:, 2] = False          # keys 256..383 seen by nobody
    (q, k, v, do), (dq, dk, dv) = run(1, 2, 2, N, d, "block_sparse", bm)
    assert torch.all(dq[:, :, 128:256] == 0)
    assert torch.all(dk[:, :, 256:384] == 0) and torch.all(dv[:, :, 256:384] == 0)
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), 1 / np.sqrt(d),
                                           mask_spec("block_sparse", bm))
    assert_grad(f64(dq), gq)
    assert_grad(f64(dk), gk)
    assert_grad(f64(dv), gv)


def test_bwd_bert_large_shape():
    """B=8, H=16, N=512, d=64 non-causal: the forward's O and LSE and the
    three gradients against the full oracle over all heads."""
    B, H, N, d = 8, 16, 512, 64
    q, k, v, do = make(B, H, H, N, d)
    o, lse = api.attn_fwd(q, k, v)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    scale = 1 / np.sqrt(d)
    o_ref, l_ref = oracle.attention_forward(f64(q), f64(k), f64(v), scale)
    assert_o_lse(f64(o), f64(lse), o_ref, l_ref, "BERT-shaped forward")
    gq, gk, gv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), scale)
    assert_grad(f64(dq), gq, "dQ BERT-shaped")
    assert_grad(f64(dk), gk, "dK BERT-shaped")
    assert_grad(f64(dv), gv, "dV BERT-shaped")


def test_bwd_is_deterministic():
    a = run(1, 4, 2, 700, 128, "causal")[1]
    b = run(1, 4, 2, 700, 128, "causal")[1]
    for x, y in zip(a, b):
        assert torch.equal(x, y)

"""GPU parity for split-KV decoding (attn_decode_fwd through the C ABI) against
the fp64 oracle's decoding step on the same seeded bf16 inputs: per-sequence
cache lengths (including empty and one-token sequences), causal multi-token
queries, GQA groups packing one or two 128-row tiles, both head sizes, and
explicit and automatic split counts."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_attn_gb300 import api, inputs
from _gpu_helpers import assert_o_lse, f64, make

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    assert api.get_status() == 0


def run_case(B, Hq, Hkv, Nq, Nk, d, causal, lens, n_splits, seed=inputs.SEED):
    q, k, v, _ = inputs.make_qkvdo(B, Hq, Hkv, Nq, Nk, d, seed)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    o, lse = api.attn_decode(q, k, v, seq_lens=sl, causal=causal, n_splits=n_splits)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode_forward(f64(q), f64(k), f64(v), 1 / math.sqrt(d), lens, causal)
    return assert_o_lse(f64(o), f64(lse), o_ref, l_ref, f"decode B{B} H{Hq}/{Hkv} Nq{Nq} Nk{Nk} d{d}")


def _lens(B, Nk, seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, Nk + 1, B)]


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal, lens, n_splits
    (4, 32, 8, 1, 4096, 128, True, "rand", 0),
    (4, 32, 8, 4, 4096, 128, True, "rand", 0),
    (2, 8, 8, 1, 1000, 64, False, None, 3),
    (3, 16, 2, 2, 2048, 128, True, [2048, 1, 700], 64),
    (2, 32, 1, 8, 1500, 64, True, [1500, 129], 5),         # 256 rows: two query tiles
    (3, 4, 4, 3, 600, 128, True, [0, 3, 600], 2),          # an empty cache and one as long as the queries
    (2, 8, 2, 1, 129, 64, True, None, 0),
    (1, 16, 16, 16, 333, 128, True, None, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_Nq{}_Nk{}_d{}_{}".format(*c[:7]))
def test_decode_matches_oracle(case):
    B, Hq, Hkv, Nq, Nk, d, causal, lens, ns = case
    if lens == "rand":
        lens = _lens(B, Nk, 17)
    run_case(B, Hq, Hkv, Nq, Nk, d, causal, lens, ns)


def test_decode_split_count_does_not_matter():
    B, Hq, Hkv, Nq, Nk, d = 2, 16, 4, 2, 3000, 128
    q, k, v, _ = inputs.make_qkvdo(B, Hq, Hkv, Nq, Nk, d, inputs.SEED)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    sl = torch.tensor([3000, 1234], dtype=torch.int32, device="cuda")
    outs = [api.attn_decode(q, k, v, seq_lens=sl, n_splits=n) for n in (1, 2, 7, 24)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert float((o.float() - outs[0][0].float()).abs().max()) <= 1e-2
        assert float((l - outs[0][1]).abs().max()) <= 2e-3


def test_decode_equals_last_rows_of_forward():
    """The decoding step over the whole cache gives the last Nq rows of causal
    attn_fwd over the full sequence (two independent GPU paths)."""
    B, Hq, Hkv, N, d, Nq = 2, 8, 2, 1024, 128, 4
    q, k, v, _ = inputs.make_qkvdo(B, Hq, Hkv, N, N, d, inputs.SEED)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o_f, l_f = api.attn_fwd(q, k, v, causal=True)
    o_d, l_d = api.attn_decode(q[:, :, N - Nq:].contiguous(), k, v, causal=True)
    torch.cuda.synchronize()
    assert float((o_d.float() - o_f[:, :, N - Nq:].float()).abs().max()) <= 1e-2
    assert float((l_d - l_f[:, :, N - Nq:]).abs().max()) <= 2e-3


def test_out_of_range_seq_lens_are_clamped_and_reported():
    """Device-side bounds check: a cached length outside [0, Nk] is clamped into
    the cache and reported by attn_get_status as ATTN_ERR_DEVICE_BOUNDS."""
    B, Hq, Hkv, Nq, Nk, d = 3, 8, 2, 1, 640, 128
    q, k, v, _ = make(B, Hq, Hkv, Nq, d, Nk=Nk)
    bad = torch.tensor([700, 640, -5], dtype=torch.int32).cuda()
    o_bad, l_bad = api.attn_decode(q, k, v, bad)
    assert api.get_status() == -8
    o_ok, l_ok = api.attn_decode(q, k, v, torch.tensor([640, 640, 0], dtype=torch.int32).cuda())
    assert api.get_status() == 0
    assert torch.equal(o_bad, o_ok) and torch.equal(l_bad, l_ok)

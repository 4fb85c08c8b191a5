"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws random tensors and
block masks.  Both the CUDA path and the fp64 oracle receive exactly the
tensors produced here (the oracle gets their bf16 values widened to float64).

Recipe: a torch CPU generator seeded with ``seed + offset`` per tensor
(Q: 0, K: 1, V: 2, dO: 3), standard-normal float32 draws rounded to bfloat16
(round-to-nearest-even).  Block masks use NumPy ``default_rng(seed + 4)``.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

SEED = 1234
OFFSET = {"q": 0, "k": 1, "v": 2, "do": 3, "mask": 4}
TILE = 128


def randn_bf16(shape, seed: int, mul: float = 1.0) -> torch.Tensor:
    """float32 N(0,1) draw from a seeded CPU generator, times ``mul``, rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if mul != 1.0:
        x = x * mul
    return x.to(torch.bfloat16)


def make_qkvdo(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
               seed: int = SEED, k_mul: float = 1.0):
    """Q ``[B,Hq,Nq,d]``, K/V ``[B,Hkv,Nk,d]``, dO ``[B,Hq,Nq,d]`` as CPU bf16 tensors."""
    q = randn_bf16((B, Hq, Nq, d), seed + OFFSET["q"])
    k = randn_bf16((B, Hkv, Nk, d), seed + OFFSET["k"], k_mul)
    v = randn_bf16((B, Hkv, Nk, d), seed + OFFSET["v"])
    do = randn_bf16((B, Hq, Nq, d), seed + OFFSET["do"])
    return q, k, v, do


def make_qkv_e4m3(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int = SEED):
    """E4M3 Q ``[B,Hq,N,d]``, K/V ``[B,Hkv,N,d]`` as uint8 CPU code tensors, with
    per-tensor dequantisation factors ``(qd, kd, vd)``.

    Each tensor is the float32 N(0,1) draw of ``randn_bf16``'s generator (same
    seeds) divided by ``amax / 448`` (its largest magnitude mapped to the
    largest finite E4M3 value) and rounded to E4M3 by torch's conversion; the
    factor is ``amax / 448``.
    """
    out, desc = [], []
    for shape, name in (((B, Hq, N, d), "q"), ((B, Hkv, N, d), "k"), ((B, Hkv, N, d), "v")):
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed + OFFSET[name]))
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        f = float(x.abs().max()) / 448.0
        out.append((x / f).to(torch.float8_e4m3fn).view(torch.uint8))
        desc.append(f)
    return out[0], out[1], out[2], tuple(desc)


def block_sparse_mask(nqb: int, nkb: int, density: float = 1.0 / 8.0,
                      seed: int = SEED) -> np.ndarray:
    """Boolean ``[nqb, nkb]`` block mask: every diagonal block kept, plus exactly
    ``round(density * #off-diagonal)`` off-diagonal blocks drawn uniformly
    without replacement."""
    rng = np.random.default_rng(seed + OFFSET["mask"])
    m = np.zeros((nqb, nkb), dtype=bool)
    nd = min(nqb, nkb)
    m[np.arange(nd), np.arange(nd)] = True
    off = np.flatnonzero(~m.reshape(-1))
    n_keep = int(round(density * off.size))
    if n_keep:
        pick = rng.choice(off, size=n_keep, replace=False)
        m.reshape(-1)[pick] = True
    return m


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a (bf16) tensor to a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()


@dataclass(frozen=True)
class Workload:
    """One synthetic attention workload (shape, mask, value distribution)."""

    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    mask: str = "none"            # "none" | "causal" | "block_sparse" | "sliding_window"
    density: float = 1.0
    window: int = 0               # sliding_window: positions a query looks back, its own included
    k_mul: float = 1.0
    chunks: int = 0               # >0: chunked causal (partial fwd + merge)
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def block_mask(self) -> Optional[np.ndarray]:
        if self.mask != "block_sparse":
            return None
        nb = -(-self.N // TILE)
        return block_sparse_mask(nb, nb, self.density)

    def tensors(self, seed: int = SEED):
        return make_qkvdo(self.B, self.Hq, self.Hkv, self.N, self.N, self.d, seed, self.k_mul)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 128, 64, note="both causal and non-causal"),
    "tiny_causal": Workload("tiny_causal", 1, 2, 2, 128, 64, "causal"),
    "bert_large": Workload("bert_large", 8, 16, 16, 512, 64),
    "gpt_causal": Workload("gpt_causal", 2, 32, 32, 8192, 128, "causal"),
    "gpt_causal_peaked": Workload("gpt_causal_peaked", 2, 32, 32, 8192, 128, "causal", k_mul=4.0),
    "gpt_noncausal": Workload("gpt_noncausal", 2, 32, 32, 8192, 128, "none"),
    "chunked_gqa": Workload("chunked_gqa", 1, 32, 8, 32768, 128, "causal", chunks=8),
    "block_sparse": Workload("block_sparse", 1, 16, 16, 16384, 64, "block_sparse", density=1.0 / 8.0),
    # local attention over the last 4096 positions (a Mistral-style sliding window) at the GPT shape
    "gpt_sliding_window": Workload("gpt_sliding_window", 2, 32, 32, 8192, 128, "sliding_window", window=4096),
    # the GPT shape with e4m3 Q, K, V and per-tensor scales (make_qkv_e4m3)
    "gpt_causal_fp8": Workload("gpt_causal_fp8", 2, 32, 32, 8192, 128, "causal"),
}

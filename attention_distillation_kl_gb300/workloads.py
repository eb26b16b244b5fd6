"""Seeded synthetic workloads for the attention-KL path.

This module only draws inputs; it holds none of the method's arithmetic, so
both the CUDA path and the float64 oracle (used by the tests) can take their
inputs from it.

The pages name no dataset: their workloads are long-context distillation at
64K-512K tokens, 32 heads, BF16 (StreamKL article on agidaily.cc, intro and
"Results").  Each named workload below is a synthetic stand-in with those
shapes.  Draws are made per (batch, head) slice from a numpy PCG64 stream
seeded by (workload seed, b, h), in float32, and rounded to bf16 once, so any
subset of heads can be regenerated on its own.
"""

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    NQ: int
    NK: int
    d1: int
    d2: int
    causal: bool
    scale: float
    # "perturbed": Q1,K1 ~ N(0, sd1^2); Q2 = Q1 + sigma N, K2 = K1 + sigma N
    # "independent": Q1,K1 ~ N(0, sd1^2); Q2,K2 ~ N(0, 1), drawn independently
    kind: str
    sigma: float
    sd1: float
    seed: int

    @property
    def pairs(self) -> int:
        """Unmasked (query, key) pairs over all heads."""
        if not self.causal:
            per = self.NQ * self.NK
        else:
            off = self.NK - self.NQ
            # row i sees keys 0..i+off, i.e. i + off + 1 keys (NQ <= NK)
            per = self.NQ * (off + 1) + self.NQ * (self.NQ - 1) // 2
        return self.B * self.H * per

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # small reference case: the oracle finishes it in well under a second
    "pr1": Workload("pr1", 1, 2, 256, 256, 64, 64, False, 1.0 / 8.0, "perturbed", 0.5, 1.0, 1000),
    "c2": Workload("c2", 2, 32, 4096, 4096, 128, 128, True, 1.0 / math.sqrt(128), "perturbed", 0.3, 1.0, 1001),
    "c3": Workload("c3", 1, 32, 16384, 16384, 128, 128, False, 1.0 / math.sqrt(128), "independent", 0.0, 1.5, 1002),
    # c3 at 2048 tokens with unit scale: peaky rows whose probabilities underflow fp32
    "c3u": Workload("c3u", 1, 32, 2048, 2048, 128, 128, False, 1.0, "independent", 0.0, 1.5, 1003),
    # headline: 64K context x 32 heads, d = 128, causal
    "c4": Workload("c4", 1, 32, 65536, 65536, 128, 128, True, 1.0 / math.sqrt(128), "perturbed", 0.3, 1.0, 1004),
    # key-split stress: 128K context, d1 = 128 teacher, d2 = 64 indexer-style student
    "c5": Workload("c5", 1, 4, 131072, 131072, 128, 64, True, 1.0 / math.sqrt(128), "independent", 0.0, 1.0, 1005),
}


def _rng(w: Workload, b: int, h: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, b, h]))


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def generate_head(w: Workload, b: int, h: int):
    """(q1, k1, q2, k2) bf16 CPU tensors [N, d] for one (batch, head) slice.

    Draw order: Q1, K1, then the student draws (noise for Q2, noise for K2 in
    the perturbed kind; Q2, K2 in the independent kind).
    """
    g = _rng(w, b, h)
    q1 = g.standard_normal((w.NQ, w.d1), dtype=np.float32) * np.float32(w.sd1)
    k1 = g.standard_normal((w.NK, w.d1), dtype=np.float32) * np.float32(w.sd1)
    if w.kind == "perturbed":
        if w.d1 != w.d2:
            raise ValueError("perturbed workloads need d1 == d2")
        nq = g.standard_normal((w.NQ, w.d2), dtype=np.float32)
        nk = g.standard_normal((w.NK, w.d2), dtype=np.float32)
        q2 = q1 + np.float32(w.sigma) * nq
        k2 = k1 + np.float32(w.sigma) * nk
    elif w.kind == "independent":
        q2 = g.standard_normal((w.NQ, w.d2), dtype=np.float32)
        k2 = g.standard_normal((w.NK, w.d2), dtype=np.float32)
    elif w.kind == "same":
        q2, k2 = q1.copy(), k1.copy()
    else:
        raise ValueError(f"unknown workload kind {w.kind}")
    return _bf16(q1), _bf16(k1), _bf16(q2), _bf16(k2)


def generate(w: Workload, heads=None):
    """Full [B, H, N, d] bf16 CPU tensors (q1, k1, q2, k2).

    ``heads``: optional list of (b, h) to fill; other slices stay zero (used
    to build large workloads whose checked heads are exact and cheap).
    """
    q1 = torch.zeros((w.B, w.H, w.NQ, w.d1), dtype=torch.bfloat16)
    k1 = torch.zeros((w.B, w.H, w.NK, w.d1), dtype=torch.bfloat16)
    q2 = torch.zeros((w.B, w.H, w.NQ, w.d2), dtype=torch.bfloat16)
    k2 = torch.zeros((w.B, w.H, w.NK, w.d2), dtype=torch.bfloat16)
    todo = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.H)]
    for b, h in todo:
        a, bb, c, d = generate_head(w, b, h)
        q1[b, h], k1[b, h], q2[b, h], k2[b, h] = a, bb, c, d
    return q1, k1, q2, k2


def generate_gqa(w: Workload, hk1: int, hk2: int, sd: float = 1.2):
    """Inputs with grouped key heads: q1 [B, H, NQ, d1], k1 [B, hk1, NK, d1],
    q2 [B, H, NQ, d2], k2 [B, hk2, NK, d2], every element N(0, sd^2) drawn
    independently from a generator seeded with w.seed (bf16 CPU tensors)."""
    g = torch.Generator().manual_seed(w.seed)
    shapes = ((w.H, w.NQ, w.d1), (hk1, w.NK, w.d1), (w.H, w.NQ, w.d2), (hk2, w.NK, w.d2))
    return [(sd * torch.randn((w.B,) + s, generator=g)).to(torch.bfloat16) for s in shapes]


def generate_dkl(w: Workload, kind: str = "ones", seed: int = 0) -> torch.Tensor:
    """Upstream gradient dL/dKL, fp32 [B, H, NQ]: all ones (the gradient of
    sum(KL)), U(0.5, 1.5) to exercise per-row indexing ("uniform"), or
    U(-1.5, 1.5) with every fifth row exactly 0 ("signed": a loss that weights
    some rows negatively or not at all), or magnitudes 10^U(-40, 30) with random
    signs and every seventh row 0 ("wide": per-row weights over the whole fp32
    range, subnormals included)."""
    if kind == "ones":
        return torch.ones((w.B, w.H, w.NQ), dtype=torch.float32)
    g = np.random.Generator(np.random.PCG64([w.seed, 7919, seed]))
    if kind == "signed":
        v = g.uniform(-1.5, 1.5, size=(w.B, w.H, w.NQ))
        v[..., ::5] = 0.0
        return torch.from_numpy(v.astype(np.float32))
    if kind == "wide":
        shape = (w.B, w.H, w.NQ)
        v = np.power(10.0, g.uniform(-40.0, 30.0, size=shape)) * np.where(g.random(shape) < 0.5, -1.0, 1.0)
        v[..., ::7] = 0.0
        return torch.from_numpy(v.astype(np.float32))
    return torch.from_numpy(g.uniform(0.5, 1.5, size=(w.B, w.H, w.NQ)).astype(np.float32))


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16/fp32 tensor (for the oracle)."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)

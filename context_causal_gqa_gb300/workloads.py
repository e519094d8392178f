"""Seeded synthetic workloads: shapes and inputs, no attention arithmetic.

This module is the one place that both the CUDA path's tests/bench and the
FP64 oracle get their inputs from.  It holds the five workload shapes (packed
THD causal GQA attention at the sizes the TransformerEngine context-parallel
pull request measures) and a seeded generator of BF16 N(0,1) q, k, v, dO.
It computes nothing of the method itself.

Recipe: seed = 1000 + workload index (1-based); a torch generator on the
target device draws q, k, v, dO in that order as float32 N(0,1), each
converted with round-to-nearest-even to BF16.  Padding rows are drawn like
any other row.  Large tensors are drawn in fixed slabs of 2^26 elements so
that no float32 copy of a whole tensor is ever held.
"""

from dataclasses import dataclass, field
from typing import List

import numpy as np

SLAB = 1 << 26


@dataclass
class Workload:
    name: str
    index: int
    seqlens: List[int]          # logical lengths S_b
    hq: int
    hkv: int
    head_dim: int
    cp: int
    pad_to: int = 1
    pack_roundtrip: bool = False
    padded: List[int] = field(default_factory=list)

    def __post_init__(self):
        if not self.padded:
            m = self.pad_to
            self.padded = [((s + m - 1) // m) * m for s in self.seqlens]

    @property
    def batch(self):
        return len(self.seqlens)

    @property
    def seed(self):
        return 1000 + self.index

    @property
    def cu_seqlens(self):
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int32)

    @property
    def cu_seqlens_padded(self):
        return np.concatenate([[0], np.cumsum(self.padded)]).astype(np.int32)

    @property
    def total_tokens(self):
        return int(sum(self.padded))

    def flops_fwd(self):
        """Causal-adjusted algorithmic forward FLOPs: 4*D*Hq*sum S(S+1)/2."""
        return 4.0 * self.head_dim * self.hq * sum(s * (s + 1) / 2 for s in self.seqlens)

    def flops_fwd_bwd(self):
        """Forward + backward algorithmic FLOPs (backward = 2.5 x forward)."""
        return 3.5 * self.flops_fwd()

    def describe(self):
        return {"workload": self.name, "batch": self.batch, "total_tokens": self.total_tokens,
                "hq": self.hq, "hkv": self.hkv, "head_dim": self.head_dim, "cp": self.cp,
                "max_seqlen": max(self.seqlens), "pack_roundtrip": self.pack_roundtrip}


def _unequal_lengths(seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(512, 4097, size=8)]


WORKLOADS = {
    "tiny": Workload("tiny", 1, [512], 4, 1, 128, 2),
    "uniform": Workload("uniform", 2, [2048] * 4, 16, 4, 128, 4),
    "unequal": Workload("unequal", 3, _unequal_lengths(1003), 32, 8, 128, 4, pad_to=64),
    "d256": Workload("d256", 4, [8192] * 8, 32, 8, 256, 8),
    "large": Workload("large", 5, [8192] * 64, 32, 8, 256, 8, pack_roundtrip=True),
}


def custom_workload(name, seqlens, hq, hkv, head_dim, cp, pad_to=1, padded=None, index=0,
                    pack_roundtrip=False):
    return Workload(name, index, list(seqlens), hq, hkv, head_dim, cp, pad_to=pad_to,
                    pack_roundtrip=pack_roundtrip, padded=list(padded) if padded is not None else [])


def _randn_bf16(shape, gen, device):
    import torch
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, SLAB):
        e = min(n, s + SLAB)
        out[s:e] = torch.randn(e - s, generator=gen, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def make_inputs(w: Workload, device="cpu", seed=None):
    """Seeded BF16 q, k, v, dO plus int32 cu_seqlens / cu_seqlens_padded."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    T = w.total_tokens
    q = _randn_bf16((T, w.hq, w.head_dim), gen, device)
    k = _randn_bf16((T, w.hkv, w.head_dim), gen, device)
    v = _randn_bf16((T, w.hkv, w.head_dim), gen, device)
    do = _randn_bf16((T, w.hq, w.head_dim), gen, device)
    cu = torch.from_numpy(w.cu_seqlens).to(device)
    cu_pad = torch.from_numpy(w.cu_seqlens_padded).to(device)
    return {"q": q, "k": k, "v": v, "do": do, "cu_seqlens": cu, "cu_seqlens_padded": cu_pad}


def sample_pairs(w: Workload, n_pairs, seed=None):
    """Seeded (sequence, q head) pairs for sampled oracle comparisons."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 7)
    seqs = rng.choice(w.batch, size=min(n_pairs, w.batch), replace=False)
    heads = rng.integers(0, w.hq, size=len(seqs))
    return [(int(b), int(h)) for b, h in zip(seqs, heads)]

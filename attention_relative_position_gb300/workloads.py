"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module only draws random inputs with the shapes and distributions of the FAT5 report's
attention benchmark (T5 encoder/decoder self-attention, head_dim 64/128, sequence 128 to 16384)
and of padding-free packing (concatenated documents with cu_seqlens boundaries). It holds none
of the attention arithmetic: the CUDA path and the oracle each do their own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seqlens: Tuple[int, ...]
    num_heads: int
    head_dim: int
    qkv_std: float = 1.0
    t5: Optional[Tuple[int, int, bool]] = None  # (num_buckets, max_distance, bidirectional)
    alibi: bool = False
    causal: bool = False
    scale: float = 1.0
    seed: int = 0
    table_std: float = 0.5
    description: str = ""

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens)) if self.seqlens else 0

    def fwd_flops(self) -> float:
        """4 * L^2 * d per head per document, halved when causal."""
        f = sum(4.0 * L * L * self.head_dim for L in self.seqlens) * self.num_heads
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def lognormal_lengths(total: int, mu: float, sigma: float, lo: int, hi: int, seed: int):
    """Document lengths round(lognormal(mu, sigma)) clipped to [lo, hi], drawn until their sum
    reaches `total`; the last one is truncated so the sum is exactly `total`."""
    rng = np.random.default_rng(seed)
    out = []
    s = 0
    while s < total:
        L = int(np.clip(round(float(rng.lognormal(mu, sigma))), lo, hi))
        L = min(L, total - s)
        out.append(L)
        s += L
    return tuple(out)


def alibi_slopes(num_heads: int) -> np.ndarray:
    """The ALiBi paper's geometric slopes 2^(-8(h+1)/H), h = 0..H-1 (caller-provided input)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / num_heads) for h in range(num_heads)], np.float32)


# The five benchmark workloads. Index 0 is the small case the oracle finishes in seconds;
# index 1 (T5 encoder, batch 8 x seq 1024) is the headline benchmark line; indices 3 and 4 are
# the long-sequence cases (seq >= 4096).
WORKLOADS = (
    Workload("t5enc_b1_h2_s128_d64", (128,), 2, 64, 1.0, (32, 128, True), False, False, 1.0,
             seed=1001, description="T5 encoder, batch 1, 2 heads, seq 128, head_dim 64"),
    Workload("t5enc_b8_h8_s1024_d64", (1024,) * 8, 8, 64, 1.0 / math.sqrt(8.0), (32, 128, True),
             False, False, 1.0, seed=1002,
             description="T5 encoder, batch 8, 8 heads, seq 1024, head_dim 64"),
    Workload("t5dec_causal_varlen_16k_h12_d64",
             lognormal_lengths(16384, 5.8, 0.8, 16, 2048, seed=1003), 12, 64, 1.0,
             (32, 128, False), False, True, 1.0, seed=1003,
             description="T5 decoder causal, varlen packed 16384 tokens, lognormal(5.8,0.8) "
                         "lengths in [16,2048], 12 heads, head_dim 64"),
    Workload("alibi_causal_b2_h16_s8192_d128", (8192,) * 2, 16, 128, 1.0, None, True, True,
             1.0 / math.sqrt(128.0), seed=1004,
             description="causal ALiBi, batch 2, 16 heads, seq 8192, head_dim 128"),
    Workload("t5enc_long_b1_h12_s16384_d64", (16384,), 12, 64, 1.0, (64, 1024, True), False,
             False, 1.0, seed=1005,
             description="long-context T5 encoder, batch 1, 12 heads, seq 16384, head_dim 64"),
)


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def make_inputs(w: Workload, device: str = "cpu", with_dout: bool = True) -> dict:
    """Draw the inputs of workload `w` on the CPU (torch generator seeded with w.seed) and move
    them to `device`. bf16 tensors are fp32 normals rounded to nearest-even bf16."""
    g = torch.Generator().manual_seed(w.seed)
    T, H, d = w.total_tokens, w.num_heads, w.head_dim

    def normal(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, dtype=torch.float32) * std)

    q = normal(T, H, d, std=w.qkv_std).to(torch.bfloat16)
    k = normal(T, H, d, std=w.qkv_std).to(torch.bfloat16)
    v = normal(T, H, d, std=w.qkv_std).to(torch.bfloat16)
    table = None
    if w.t5 is not None:
        table = normal(w.t5[0], H, std=w.table_std)
    dout = normal(T, H, d).to(torch.bfloat16) if with_dout else None
    slopes = torch.from_numpy(alibi_slopes(H)) if w.alibi else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(w.seqlens)]).astype(np.int32))
    out = dict(q=q, k=k, v=v, table=table, slopes=slopes, dout=dout, cu_seqlens=cu)
    if device != "cpu":
        out = {key: (t.to(device) if t is not None else None) for key, t in out.items()}
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 tensor as numpy uint16 (exact, no conversion)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class XWorkload:
    """A problem with its own query and key lengths per document (cross-attention, or queries
    over a longer key cache) and grouped-query heads."""
    name: str
    qlens: Tuple[int, ...]
    klens: Tuple[int, ...]
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    qkv_std: float = 1.0
    t5: Optional[Tuple[int, int, bool]] = None
    alibi: bool = False
    causal: bool = False
    scale: float = 1.0
    seed: int = 0
    table_std: float = 0.5

    @property
    def total_q(self) -> int:
        return int(sum(self.qlens))

    @property
    def total_k(self) -> int:
        return int(sum(self.klens))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.qlens)) if self.qlens else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.klens)) if self.klens else 0

    def fwd_flops(self) -> float:
        """4 * Lq * Lk * d per query head and document (the attention products a dense kernel
        computes), halved when causal only for square documents (the diagonal mask)."""
        f = sum(4.0 * a * b * self.head_dim for a, b in zip(self.qlens, self.klens))
        f *= self.num_heads_q
        return f / 2 if (self.causal and self.qlens == self.klens) else f


def make_xinputs(w: XWorkload, device: str = "cpu") -> dict:
    """Seeded inputs of an XWorkload (torch CPU generator, then moved to `device`): q, dout
    [Tq, Hq, d], k, v [Tk, Hkv, d] as bf16-rounded normals, the table [nb, Hq] and the ALiBi
    slopes [Hq] when asked for, and both cu_seqlens."""
    g = torch.Generator().manual_seed(w.seed)
    Tq, Tk, Hq, Hkv, d = w.total_q, w.total_k, w.num_heads_q, w.num_heads_kv, w.head_dim

    def normal(*shape, std=1.0):
        return torch.randn(*shape, generator=g, dtype=torch.float32) * std

    q = normal(Tq, Hq, d, std=w.qkv_std).to(torch.bfloat16)
    k = normal(Tk, Hkv, d, std=w.qkv_std).to(torch.bfloat16)
    v = normal(Tk, Hkv, d, std=w.qkv_std).to(torch.bfloat16)
    table = normal(w.t5[0], Hq, std=w.table_std) if w.t5 is not None else None
    dout = normal(Tq, Hq, d).to(torch.bfloat16)
    slopes = torch.from_numpy(alibi_slopes(Hq)) if w.alibi else None
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(w.qlens)]).astype(np.int32))
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(w.klens)]).astype(np.int32))
    out = dict(q=q, k=k, v=v, table=table, slopes=slopes, dout=dout, cu_seqlens_q=cu_q,
               cu_seqlens_k=cu_k)
    if device != "cpu":
        out = {key: (t.to(device) if t is not None else None) for key, t in out.items()}
    return out


def make_norm_inputs(rows: int, dim: int, seed: int, device: str = "cpu"):
    """RMSNorm inputs: x bf16 [rows, dim] ~ N(0, s_r^2) with a per-row scale s_r in [0.1, 4],
    the weight fp32 [dim] ~ 1 + 0.1 N(0, 1), and dy bf16 [rows, dim] ~ N(0, 1)."""
    g = torch.Generator().manual_seed(seed)
    s = 0.1 + 3.9 * torch.rand(rows, 1, generator=g)
    x = (torch.randn(rows, dim, generator=g) * s).to(torch.bfloat16)
    w = 1.0 + 0.1 * torch.randn(dim, generator=g)
    dy = torch.randn(rows, dim, generator=g).to(torch.bfloat16)
    return x.to(device), w.to(device), dy.to(device)


def make_ce_inputs(rows: int, vocab: int, seed: int, device: str = "cpu"):
    """Cross-entropy inputs: logits bf16 [rows, vocab] ~ N(0, 2^2), and int32 targets uniform
    over the vocabulary with about one row in eight ignored (-100)."""
    g = torch.Generator().manual_seed(seed)
    z = (2.0 * torch.randn(rows, vocab, generator=g)).to(torch.bfloat16)
    t = torch.randint(0, vocab, (rows,), generator=g, dtype=torch.int32)
    drop = torch.rand(rows, generator=g) < 0.125
    t[drop] = -100
    return z.to(device), t.to(device)

"""Seeded synthetic inputs for the attention forward.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds shapes, seeds and random numbers only -- none of the
attention arithmetic.

Recipe (after "[BUG] CuTe DSL 4.7/4.8 regression: FlashAttention-4 SM100
forward kernel spills registers", section "Steps/Code to reproduce bug"):
seed 0, then q, k, v drawn in that order as standard-normal bf16 tensors of
shape [total_tokens, heads, head_dim]; sequence boundaries
cu_seqlens = round(linspace(0, total, docs + 1)) as int32; max_seqlen = the
longest sequence; scale = 1/sqrt(head_dim).  Draws use a CPU torch generator,
so the same bytes feed the oracle and the GPU.

The dense workloads (batch, seq, heads, head_dim) follow the shape flags of
"[BUG] Unexpected Slower Performance in C++ CuTe (77_blackwell_fmha) vs Python
CuTe DSL (fmha.py) on Jetson Thor", section "Test Commands": the [b, s, h, d]
tensor is the same memory as [b * s, h, d] with implicit equal-length
sequences.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """Shape description of one attention forward problem."""

    name: str
    description: str
    heads: int
    head_dim: int
    seqlens_q: tuple
    seqlens_k: tuple
    causal: bool
    dense: bool = False  # True: equal lengths, passed without cu_seqlens
    scale: Optional[float] = None  # None -> 1/sqrt(head_dim)
    kv_heads: Optional[int] = None  # grouped K/V heads; None -> heads (multi-head)

    @property
    def n_kv_heads(self) -> int:
        return self.heads if self.kv_heads is None else int(self.kv_heads)

    @property
    def batch(self) -> int:
        return len(self.seqlens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.seqlens_k))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.seqlens_q)) if self.seqlens_q else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.seqlens_k)) if self.seqlens_k else 0

    @property
    def softmax_scale(self) -> float:
        return (1.0 / math.sqrt(self.head_dim)) if self.scale is None else float(self.scale)

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs that attend, summed over sequences (one head)."""
        total = 0
        for lq, lk in zip(self.seqlens_q, self.seqlens_k):
            if not self.causal:
                total += lq * lk
            else:
                off = lk - lq
                for_rows = 0
                # row i sees min(lk, max(0, i + off + 1)) keys
                lo = max(0, -off)  # first row with any visible key (if lk > 0)
                for i in range(lo, lq):
                    for_rows += min(lk, i + off + 1)
                total += for_rows
        return total

    def flops(self) -> float:
        """Algorithmic FLOPs: 2 GEMMs x 2 FLOP per MAC x head_dim per visible pair."""
        return 4.0 * self.head_dim * self.heads * self.visible_pairs()

    def cu_seqlens(self):
        cq = np.concatenate([[0], np.cumsum(self.seqlens_q)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(self.seqlens_k)]).astype(np.int32)
        return cq, ck


def linspace_docs(total: int, docs: int) -> tuple:
    """Document lengths from cu = round(linspace(0, total, docs + 1))."""
    cu = np.rint(np.linspace(0, total, docs + 1)).astype(np.int64)
    return tuple(int(x) for x in np.diff(cu))


def dense(name, batch, seqlen_q, heads, head_dim=128, causal=False, seqlen_k=None,
          description="", scale=None, kv_heads=None) -> Workload:
    seqlen_k = seqlen_q if seqlen_k is None else seqlen_k
    return Workload(name, description, heads, head_dim, (seqlen_q,) * batch,
                    (seqlen_k,) * batch, causal, dense=True, scale=scale, kv_heads=kv_heads)


def varlen(name, seqlens_q: Sequence[int], heads, head_dim=128, causal=True,
           seqlens_k: Optional[Sequence[int]] = None, description="", scale=None,
           kv_heads=None) -> Workload:
    seqlens_k = seqlens_q if seqlens_k is None else seqlens_k
    if len(seqlens_k) != len(seqlens_q):
        raise ValueError("seqlens_q and seqlens_k must have the same number of sequences")
    return Workload(name, description, heads, head_dim, tuple(int(x) for x in seqlens_q),
                    tuple(int(x) for x in seqlens_k), causal, dense=False, scale=scale,
                    kv_heads=kv_heads)


# The five named workloads.
C1 = dense("dense_b1_h2_s128", 1, 128, 2,
           description="Dense non-causal, batch 1, heads 2, seq 128, head_dim 128")
C2 = dense("dense_b1_h16_s2225", 1, 2225, 16,
           description="Dense non-causal, batch 1, heads 16, seq 2225, head_dim 128")
C3 = varlen("varlen_causal_t8192_h32_docs4", linspace_docs(8192, 4), 32,
            description="Varlen causal, 8192 packed tokens, 32 heads, 4 docs")
C4 = varlen("varlen_causal_t32768_h32_docs8", linspace_docs(32768, 8), 32,
            description="Varlen causal, 32768 packed tokens, 32 heads, 8 docs")
C5 = varlen("causal_t32768_h16_docs1", linspace_docs(32768, 1), 16,
            description="Single-document causal, 32768 tokens, 16 heads")

CONFIGS = {w.name: w for w in (C1, C2, C3, C4, C5)}

# Grouped K/V heads on the varlen causal 8192-token shape: 32 query heads on 8
# K/V heads (not one of the five named workloads; measured as an extension).
GQA_C3 = varlen("gqa_varlen_causal_t8192_h32_kv8_docs4", linspace_docs(8192, 4), 32, kv_heads=8,
                description="Varlen causal, 8192 packed tokens, 32 query heads on 8 K/V heads, 4 docs")
# head_dim 64 on the single-document causal 32768-token shape with 32 heads
D64_C5 = varlen("d64_causal_t32768_h32_docs1", linspace_docs(32768, 1), 32, head_dim=64,
                description="Single-document causal, 32768 tokens, 32 heads, head_dim 64")
# head_dim 256 (one 128-row query tile per CTA) on the dense h16 s2225 shape
# and on the varlen causal 8192-token shape
D256_C2 = dense("d256_dense_b1_h16_s2225", 1, 2225, 16, head_dim=256,
                description="Dense non-causal, batch 1, heads 16, seq 2225, head_dim 256")
D256_C3 = varlen("d256_varlen_causal_t8192_h32_docs4", linspace_docs(8192, 4), 32, head_dim=256,
                 description="Varlen causal, 8192 packed tokens, 32 heads, 4 docs, head_dim 256")
EXTRA = {GQA_C3.name: GQA_C3, D64_C5.name: D64_C5, D256_C2.name: D256_C2, D256_C3.name: D256_C3}


@dataclass
class Inputs:
    workload: Workload
    q: torch.Tensor  # [total_q, heads, head_dim] bf16, CPU
    k: torch.Tensor  # [total_k, heads, head_dim] bf16, CPU
    v: torch.Tensor
    cu_seqlens_q: Optional[torch.Tensor]  # int32 [batch + 1] or None (dense)
    cu_seqlens_k: Optional[torch.Tensor]
    extra: dict = field(default_factory=dict)

    def oracle_args(self):
        """Arguments in the order oracle_fwd / brute_force_fwd take them."""
        w = self.workload
        cq = None if self.cu_seqlens_q is None else self.cu_seqlens_q.numpy()
        ck = None if self.cu_seqlens_k is None else self.cu_seqlens_k.numpy()
        return (self.q, self.k, self.v, cq, ck, w.batch, w.max_seqlen_q, w.max_seqlen_k,
                w.softmax_scale, w.causal)


def make_inputs(w: Workload, seed: int = 0, dist: str = "randn") -> Inputs:
    """Seeded q, k, v (drawn in that order) for workload w, on the CPU.

    dist: "randn" (standard normal, the recipe above) or "uniform" (U[-1, 1)),
    both rounded to bf16.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shapes = [(w.total_q, w.heads, w.head_dim), (w.total_k, w.n_kv_heads, w.head_dim),
              (w.total_k, w.n_kv_heads, w.head_dim)]
    out = []
    for shp in shapes:
        if dist == "randn":
            t = torch.randn(shp, generator=g, dtype=torch.float32)
        elif dist == "uniform":
            t = torch.rand(shp, generator=g, dtype=torch.float32) * 2.0 - 1.0
        else:
            raise ValueError(dist)
        out.append(t.to(torch.bfloat16))
    q, k, v = out
    if w.dense:
        cq = ck = None
    else:
        a, b = w.cu_seqlens()
        cq, ck = torch.from_numpy(a), torch.from_numpy(b)
    return Inputs(w, q, k, v, cq, ck)


def make_dout(w: Workload, seed: int = 0) -> torch.Tensor:
    """Seeded upstream gradient dO for the backward pass: standard-normal bf16
    [total_q, heads, head_dim] on the CPU, from its own generator (seeded with
    seed + 0x5EED, so q, k, v of make_inputs keep their bytes)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 0x5EED)
    return torch.randn((w.total_q, w.heads, w.head_dim), generator=g, dtype=torch.float32).to(torch.bfloat16)


def sample_keys(w: Workload, n_random: int, seed: int = 2, edge_rows: int = 2) -> np.ndarray:
    """Flattened (token * kv_heads + kv_head) key indices for a seeded sample:
    every sequence's first and last ``edge_rows`` keys for every K/V head plus
    ``n_random`` uniformly drawn (token, K/V head) pairs."""
    rng = np.random.default_rng(seed)
    picks = []
    _, ck = w.cu_seqlens()
    hk = w.n_kv_heads
    for b in range(w.batch):
        lo, hi = int(ck[b]), int(ck[b + 1])
        toks = set(range(lo, min(hi, lo + edge_rows))) | set(range(max(lo, hi - edge_rows), hi))
        for t in sorted(toks):
            for h in range(hk):
                picks.append(t * hk + h)
    if w.total_k > 0 and n_random > 0:
        toks = rng.integers(0, w.total_k, size=n_random)
        hs = rng.integers(0, hk, size=n_random)
        picks.extend((toks * hk + hs).tolist())
    return np.unique(np.asarray(picks, dtype=np.int64))


def sample_rows(w: Workload, n_random: int, seed: int = 1, edge_rows: int = 2) -> np.ndarray:
    """Flattened (token * heads + head) indices for a seeded row sample.

    Per sequence: its first and last ``edge_rows`` rows for every head, plus
    ``n_random`` uniformly drawn (token, head) pairs over the whole batch.
    """
    rng = np.random.default_rng(seed)
    picks = []
    cq, _ = w.cu_seqlens()
    for b in range(w.batch):
        lo, hi = int(cq[b]), int(cq[b + 1])
        toks = set(range(lo, min(hi, lo + edge_rows))) | set(range(max(lo, hi - edge_rows), hi))
        for t in sorted(toks):
            for h in range(w.heads):
                picks.append(t * w.heads + h)
    if w.total_q > 0 and n_random > 0:
        toks = rng.integers(0, w.total_q, size=n_random)
        hs = rng.integers(0, w.heads, size=n_random)
        picks.extend((toks * w.heads + hs).tolist())
    return np.unique(np.asarray(picks, dtype=np.int64))

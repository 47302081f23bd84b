"""Seeded synthetic workloads for context-parallel prefill attention.

This module holds shapes, seeds and random-number generation only -- none of
the attention arithmetic -- so that both the CUDA path's tests and the oracle's
tests can draw the same inputs from it.

Shapes follow the long-context prefill workloads the article "Scaling LLM
Inference: Innovations in Tensor Parallelism, Context Parallelism, and Expert
Parallelism" discusses (sections "Context Parallelism for Million-Token
Contexts" and "The communication bottleneck across all three axes": Llama 3
405B at 128K tokens, 1M-token contexts): GQA head counts of one TP-8 shard of a
405B-shaped layer (16 q heads, 1 kv head), a Llama-3-8B-shaped layer (32/8), a
partial prefill against a cached context, and a 1M-token case.  The pages name
no dataset; Q, K, V are i.i.d. N(0, 1) drawn with torch's generator on the
target device and rounded to the compute dtype (round-to-nearest-even).
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED_Q, SEED_K, SEED_V = 1, 2, 3
SAMPLE_SEED = 20251017
SAMPLE_ROWS = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    hq: int
    hkv: int
    head_dim: int
    sq: int            # query rows
    skv: int           # key/value rows
    q_base: int        # absolute position of query row 0
    n_chunks: int      # CP chunks (ranks)
    dtype: str         # "bf16" or "fp32"
    k_scale: float = 1.0
    causal: bool = True

    @property
    def chunk_q(self) -> int:
        return self.sq // self.n_chunks if self.sq >= self.n_chunks else self.sq

    @property
    def chunk_kv(self) -> int:
        return self.skv // self.n_chunks

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the causal mask keeps, per (batch, head)."""
        p = self.q_base + np.arange(self.sq, dtype=np.int64)
        if not self.causal:
            return int(self.sq * self.skv)
        return int(np.minimum(p + 1, self.skv).clip(min=0).sum())

    def causal_flops(self) -> float:
        """Causal-effective FLOPs of one layer: QK^T and PV, 2 FLOPs per MAC each,
        over the visible pairs only."""
        return 4.0 * self.head_dim * self.hq * self.batch * self.visible_pairs()


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 64, 256, 256, 0, 4, "fp32"),
    "llama3-8b": Workload("llama3-8b", 1, 32, 8, 128, 8192, 8192, 0, 8, "bf16", k_scale=0.5),
    "partial-32k": Workload("partial-32k", 1, 16, 1, 128, 2048, 32768, 30720, 8, "bf16"),
    "128k": Workload("128k", 1, 16, 1, 128, 131072, 131072, 0, 16, "bf16"),
    "1m": Workload("1m", 1, 8, 1, 128, 1048576, 1048576, 0, 8, "bf16"),
    # Decode-shaped Pass-Q: one new token per sequence against a 128K-token
    # cache sharded over 16 CP ranks, 8 sequences (405B TP-8 shard heads).
    "decode-128k-b8": Workload("decode-128k-b8", 8, 16, 1, 128, 1, 131072, 131071, 16, "bf16"),
}


def make_qkv(w: Workload, device="cpu", seeds=(SEED_Q, SEED_K, SEED_V)):
    """Q [B,Sq,Hq,D], K/V [B,Skv,Hkv,D], i.i.d. N(0,1) in w.dtype on ``device``."""
    import torch

    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = []
    for seed, shape, scale in ((seeds[0], (w.batch, w.sq, w.hq, w.head_dim), 1.0),
                               (seeds[1], (w.batch, w.skv, w.hkv, w.head_dim), w.k_scale),
                               (seeds[2], (w.batch, w.skv, w.hkv, w.head_dim), 1.0)):
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        t = torch.empty(shape, dtype=dt, device=device)
        # Draw in slabs so the fp32 temporary stays small at 1M tokens.
        flat = t.view(shape[0] * shape[1], -1)
        step = max(1, (1 << 27) // flat.shape[1])
        for r0 in range(0, flat.shape[0], step):
            r1 = min(flat.shape[0], r0 + step)
            x = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                            dtype=torch.float32)
            flat[r0:r1] = x.to(dt)
        if scale != 1.0:
            t.mul_(scale)  # a power of two: exact after the cast
        out.append(t)
    return tuple(out)


def sample_rows(w: Workload, n: int = SAMPLE_ROWS, seed: int = SAMPLE_SEED) -> np.ndarray:
    """Sorted distinct query-row indices: the first and last row of every chunk,
    the rest uniform without replacement from ``default_rng(seed)``."""
    if w.sq <= n:
        return np.arange(w.sq, dtype=np.int64)
    cq = w.chunk_q
    forced = set()
    for c in range(w.n_chunks):
        forced.add(c * cq)
        forced.add(c * cq + cq - 1)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(w.sq, dtype=np.int64), np.fromiter(forced, dtype=np.int64))
    pick = rng.choice(rest, size=n - len(forced), replace=False)
    return np.sort(np.concatenate([np.fromiter(forced, dtype=np.int64), pick]))

"""Brute-force attention over the full masked score matrix -- TEST INFRASTRUCTURE.

Used only to pin the C oracle on tiny inputs.  It takes a different route from
``cpattn_oracle.c``: it builds the whole [nq, Skv] logit matrix with one matmul
per head, masks it with -inf, and normalises with ``numpy`` reductions over the
full matrix, so an index or masking slip in either one shows up as a mismatch.
Definition followed: causal softmax attention, the result the article "Scaling
LLM Inference ..." (section "Context Parallelism for Million-Token Contexts")
says every CP rank obtains over the full context.
"""
from __future__ import annotations

import numpy as np


def attention(q, k, v, *, q_pos=None, kv_pos0=0, causal=True, scale=None):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, nq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    g = Hq // Hkv
    if q_pos is None:
        q_pos = np.arange(nq)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kv_abs = kv_pos0 + np.arange(Skv)
    visible = np.ones((nq, Skv), dtype=bool)
    if causal:
        visible = kv_abs[None, :] <= q_pos[:, None]
    o = np.zeros((B, nq, Hq, D))
    lse = np.full((B, Hq, nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            kh = k[b, :, h // g, :]
            vh = v[b, :, h // g, :]
            logits = scale * (q[b, :, h, :] @ kh.T)          # [nq, Skv]
            logits = np.where(visible, logits, -np.inf)
            for i in range(nq):
                row = logits[i]
                if not visible[i].any():
                    continue
                m = row.max()
                e = np.exp(row - m)                           # masked -> 0
                z = e.sum()
                o[b, i, h] = (e / z) @ vh
                lse[b, h, i] = m + np.log(z)
    return o, lse

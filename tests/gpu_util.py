"""Helpers for the GPU parity tests: run the oracle on host copies of exactly
the inputs the GPU saw and compare element by element."""
from __future__ import annotations

import numpy as np

import oracle

# Max-abs-error bounds on O and LSE (bf16 inputs / fp32 inputs).
TOL = {"bf16": (2e-2, 1e-3), "fp32": (1e-4, 1e-5)}


def host_f32(t):
    return t.detach().float().cpu().numpy()


def oracle_rows(q, k, v, rows, *, q_base=0, kv_pos0=0, causal=True, scale=None):
    """Oracle (O, LSE) for the listed query rows of q (torch tensors, any device)."""
    import torch

    rows_t = torch.as_tensor(np.asarray(rows), device=q.device, dtype=torch.long)
    qs = host_f32(q.index_select(1, rows_t))
    return oracle.attention(qs, host_f32(k), host_f32(v), q_pos=q_base + np.asarray(rows),
                            kv_pos0=kv_pos0, causal=causal, scale=scale)


def compare(o_gpu, lse_gpu, rows, ref_o, ref_l, tol, what=""):
    """Max-abs errors of GPU rows against the oracle; asserts the bounds."""
    import torch

    rows_t = torch.as_tensor(np.asarray(rows), device=o_gpu.device, dtype=torch.long)
    go = o_gpu.index_select(1, rows_t).float().cpu().numpy().astype(np.float64)
    gl = lse_gpu.index_select(2, rows_t).float().cpu().numpy().astype(np.float64)
    assert np.isfinite(go).all(), f"{what}: non-finite O"
    assert not np.isnan(gl).any(), f"{what}: NaN LSE"
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(gl), empty), f"{what}: empty-row mismatch"
    e_o = float(np.abs(go - ref_o).max()) if go.size else 0.0
    fin = ~empty
    e_l = float(np.abs(gl[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert e_o <= tol[0], f"{what}: max |dO| = {e_o:.3g} > {tol[0]}"
    assert e_l <= tol[1], f"{what}: max |dLSE| = {e_l:.3g} > {tol[1]}"
    return e_o, e_l

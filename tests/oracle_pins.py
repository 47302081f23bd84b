"""Pins for the fp64 oracle, written against any ``attention(q, k, v, ...)`` callable.

Each pin checks the oracle against something other than itself: a brute-force
evaluation over the full score matrix, a hand-derived worked example, a closed
form, a textbook library routine, or an invariant of the definition.  The same
pins are run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show that a plausible slip fails at least one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_examples.json")

_CONST = {"0": 0.0, "1": 1.0, "ln2": math.log(2.0), "ln3": math.log(3.0),
          "ln4": math.log(4.0), "ln3/2": math.log(3.0) / 2.0, "-inf": -math.inf}


def _num(x):
    if isinstance(x, str):
        return _CONST[x]
    if isinstance(x, list):
        return [_num(y) for y in x]
    return float(x)


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(rng, shape, lo=-2, hi=2):
    # Multiples of 1/8 in a small range: exact in fp32, so shifts stay exact.
    return (rng.integers(lo * 8, hi * 8 + 1, size=shape) / 8.0).astype(np.float32)


def pin_golden_attention(attn):
    for ex in golden()["attention"]:
        q, k, v = (np.array(ex[n], dtype=np.float32) for n in ("q", "k", "v"))
        o, lse = attn(q, k, v, q_pos=np.array(ex["q_pos"]), kv_pos0=ex["kv_pos0"],
                      causal=ex["causal"], scale=_num(ex["scale"]))
        np.testing.assert_allclose(o, np.array(ex["o"]), rtol=0, atol=1e-12, err_msg=ex["name"])
        np.testing.assert_allclose(lse, np.array(_num(ex["lse"])), rtol=0, atol=1e-12,
                                   err_msg=ex["name"])


def pin_bruteforce(attn, seed=0):
    rng = np.random.default_rng(seed)
    for S, D, (hq, hkv), causal in [(1, 1, (1, 1), True), (2, 8, (2, 1), True),
                                    (3, 64, (4, 2), True), (17, 8, (4, 1), False),
                                    (64, 128, (2, 2), True), (40, 64, (6, 3), True)]:
        B = 2 if S <= 17 else 1
        q = rng.standard_normal((B, S, hq, D)).astype(np.float32)
        skv = S + 5
        k = rng.standard_normal((B, skv, hkv, D)).astype(np.float32)
        v = rng.standard_normal((B, skv, hkv, D)).astype(np.float32)
        q_pos = rng.integers(0, skv + 3, size=S)          # arbitrary positions
        kv_pos0 = int(rng.integers(0, 3))
        o, lse = attn(q, k, v, q_pos=q_pos, kv_pos0=kv_pos0, causal=causal)
        ob, lb = brute.attention(q, k, v, q_pos=q_pos, kv_pos0=kv_pos0, causal=causal)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-11)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lb))
        fin = np.isfinite(lb)
        np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-11)


def pin_library_softmax(attn, seed=1):
    """Non-causal single query: attention is softmax-weighted averaging, which
    scipy's softmax / logsumexp compute independently."""
    from scipy.special import logsumexp, softmax

    rng = np.random.default_rng(seed)
    D, skv = 16, 33
    q = rng.standard_normal((1, 1, 1, D)).astype(np.float32)
    k = rng.standard_normal((1, skv, 1, D)).astype(np.float32)
    v = rng.standard_normal((1, skv, 1, D)).astype(np.float32)
    scale = 0.37
    o, lse = attn(q, k, v, q_pos=[0], causal=False, scale=scale)
    s = scale * (k[0, :, 0, :].astype(np.float64) @ q[0, 0, 0].astype(np.float64))
    np.testing.assert_allclose(o[0, 0, 0], softmax(s) @ v[0, :, 0, :].astype(np.float64),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], logsumexp(s), rtol=0, atol=1e-12)


def pin_constant_v(attn, seed=2):
    rng = np.random.default_rng(seed)
    B, S, hq, hkv, D = 1, 23, 4, 2, 8
    q = rng.standard_normal((B, S, hq, D)).astype(np.float32)
    k = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    c = _rand(rng, (D,))
    v = np.broadcast_to(c, (B, S, hkv, D)).copy()
    o, _ = attn(q, k, v, causal=True)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def pin_zero_q(attn, seed=3):
    """Q = 0: every visible logit is 0, so O is the mean of the visible V rows and
    LSE = ln(number of visible keys)."""
    rng = np.random.default_rng(seed)
    B, S, hq, hkv, D = 1, 19, 2, 1, 8
    kv_pos0 = 4
    q = np.zeros((B, S, hq, D), dtype=np.float32)
    k = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    v = _rand(rng, (B, S, hkv, D))
    q_pos = np.arange(S) + 6        # row i sees keys 0..min(i+2, S-1)
    o, lse = attn(q, k, v, q_pos=q_pos, kv_pos0=kv_pos0, causal=True)
    for i in range(S):
        n = min(q_pos[i] - kv_pos0 + 1, S)
        for h in range(hq):
            np.testing.assert_allclose(o[0, i, h], v[0, :n, 0].astype(np.float64).mean(0),
                                       rtol=0, atol=1e-12)
            assert abs(lse[0, h, i] - math.log(n)) < 1e-12


def pin_single_visible_key(attn, seed=4):
    """A row whose position equals the first key's position sees only that key:
    O = v_0 exactly and LSE = scale * q . k_0."""
    rng = np.random.default_rng(seed)
    D, S = 32, 9
    q = _rand(rng, (1, 1, 3, D))
    k = _rand(rng, (1, S, 3, D))
    v = _rand(rng, (1, S, 3, D))
    scale = 0.25
    o, lse = attn(q, k, v, q_pos=[7], kv_pos0=7, causal=True, scale=scale)
    for h in range(3):
        np.testing.assert_array_equal(o[0, 0, h], v[0, 0, h].astype(np.float64))
        expect = scale * float(np.dot(q[0, 0, h].astype(np.float64), k[0, 0, h].astype(np.float64)))
        assert abs(lse[0, h, 0] - expect) < 1e-12


def pin_key_shift(attn, seed=5):
    """Adding u to every key adds scale*q.u to every logit of a row: O is
    unchanged and LSE shifts by scale*q.u."""
    rng = np.random.default_rng(seed)
    B, S, hq, hkv, D = 1, 21, 4, 2, 16
    q = _rand(rng, (B, S, hq, D))
    k = _rand(rng, (B, S, hkv, D))
    v = _rand(rng, (B, S, hkv, D))
    u = _rand(rng, (D,))
    scale = 0.5
    o0, l0 = attn(q, k, v, causal=True, scale=scale)
    o1, l1 = attn(q, (k + u).astype(np.float32), v, causal=True, scale=scale)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-11)
    shift = scale * np.einsum("bihd,d->bhi", q.astype(np.float64), u.astype(np.float64))
    np.testing.assert_allclose(l1 - l0, shift, rtol=0, atol=1e-11)


def pin_empty_rows(attn):
    q = np.ones((1, 3, 2, 4), dtype=np.float32)
    k = np.ones((1, 5, 1, 4), dtype=np.float32)
    v = np.ones((1, 5, 1, 4), dtype=np.float32)
    o, lse = attn(q, k, v, q_pos=[0, 9, 10], kv_pos0=10, causal=True)
    assert np.all(np.isneginf(lse[0, :, :2])) and np.all(o[0, :2] == 0)
    assert np.all(np.isfinite(lse[0, :, 2]))


def pin_chunking_invariance(attn, merge, seed=6):
    """Any split of the keys into disjoint contiguous parts, each attended
    separately at its own offset and merged by LSE, equals the unsplit result
    (the claim that CP ranks reach attention over the full context)."""
    rng = np.random.default_rng(seed)
    B, S, hq, hkv, D = 1, 50, 4, 2, 16
    q = rng.standard_normal((B, S, hq, D)).astype(np.float32)
    k = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    ref_o, ref_l = attn(q, k, v, causal=True)
    for cuts in ([25], [1, 2, 49], sorted(rng.choice(np.arange(1, S), 6, replace=False))):
        bounds = [0] + list(cuts) + [S]
        parts_o, parts_l = [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            o, lse = attn(q, k[:, a:b], v[:, a:b], kv_pos0=a, causal=True)
            parts_o.append(o)
            parts_l.append(np.transpose(lse, (0, 2, 1)))   # [B, S, Hq] like o
        mo, ml = merge(np.stack(parts_o), np.stack(parts_l))
        np.testing.assert_allclose(mo, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(np.transpose(ml, (0, 2, 1)), ref_l, rtol=0, atol=1e-12)


def pin_golden_merge(merge):
    for ex in golden()["merge"]:
        o, lse = merge(np.array(ex["o_parts"], dtype=np.float64),
                       np.array(_num(ex["lse_parts"]), dtype=np.float64))
        np.testing.assert_allclose(o, np.array(ex["o"]), rtol=0, atol=1e-12, err_msg=ex["name"])
        np.testing.assert_allclose(lse, np.array(_num(ex["lse"])), rtol=0, atol=1e-12,
                                   err_msg=ex["name"])
        assert not np.isnan(o).any()


ATTENTION_PINS = [pin_golden_attention, pin_bruteforce, pin_library_softmax, pin_constant_v,
                  pin_zero_q, pin_single_visible_key, pin_key_shift, pin_empty_rows]

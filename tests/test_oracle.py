"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ATTENTION_PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    pin(oracle.attention)


def test_chunking_invariance():
    pins.pin_chunking_invariance(oracle.attention, oracle.merge)


def test_golden_merge():
    pins.pin_golden_merge(oracle.merge)


def test_merge_commutes_and_identity():
    rng = np.random.default_rng(11)
    o = rng.standard_normal((3, 7, 5))
    lse = rng.standard_normal((3, 7)) * 3
    a, la = oracle.merge(o, lse)
    b, lb = oracle.merge(o[::-1].copy(), lse[::-1].copy())
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-14)
    one, lone = oracle.merge(np.stack([o[0], np.zeros_like(o[0])]),
                             np.stack([lse[0], np.full_like(lse[0], -np.inf)]))
    np.testing.assert_allclose(one, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lone, lse[0], rtol=0, atol=1e-15)


def test_ring_schedules_equal_unchunked():
    """Pass-KV order (ring steps j = i, i-1, ...) and Pass-Q order (j ascending),
    both merging per-pair partials, give the unchunked result."""
    rng = np.random.default_rng(12)
    B, S, hq, hkv, D, N = 1, 48, 2, 1, 8, 4
    C = S // N
    q = rng.standard_normal((B, S, hq, D)).astype(np.float32)
    k = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, S, hkv, D)).astype(np.float32)
    ref_o, ref_l = oracle.attention(q, k, v, causal=True)
    for order in ("kv", "q"):
        for i in range(N):
            js = [(i - t) % N for t in range(N)] if order == "kv" else list(range(N))
            parts_o, parts_l = [], []
            for j in js:
                if j * C > i * C + C - 1:
                    continue       # fully masked pair
                o, lse = oracle.attention(q[:, i * C:(i + 1) * C], k[:, j * C:(j + 1) * C],
                                          v[:, j * C:(j + 1) * C],
                                          q_pos=np.arange(i * C, (i + 1) * C), kv_pos0=j * C)
                parts_o.append(o)
                parts_l.append(np.transpose(lse, (0, 2, 1)))
            mo, ml = oracle.merge(np.stack(parts_o), np.stack(parts_l))
            np.testing.assert_allclose(mo, ref_o[:, i * C:(i + 1) * C], rtol=0, atol=1e-12)
            np.testing.assert_allclose(np.transpose(ml, (0, 2, 1)),
                                       ref_l[:, :, i * C:(i + 1) * C], rtol=0, atol=1e-12)

"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one: evidence that the pins constrain the oracle."""
import functools
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "cpattn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("n_vis = last + 1;", "n_vis = last;"),
    "gqa_mapping": ("const int64_t hk = h / g;", "const int64_t hk = h % Hkv;"),
    "dropped_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "lse_missing_max": ("const double L = m + log(sum);\n      /* Pass 2",
                        "const double L = log(sum);\n      /* Pass 2"),
    "merge_missing_max": ("const double L = m + log(sum);\n    for (int64_t t = 0; t < D; ++t) orow",
                          "const double L = log(sum);\n    for (int64_t t = 0; t < D; ++t) orow"),
    "k_and_v_swapped": ("const float *kj = k + ", "const float *kj = v + "),
    "kv_offset_sign": ("q_pos[i] - kv_pos0", "q_pos[i] + kv_pos0"),
    "unnormalised_weights": ("const double w = exp(s[j] - L);", "const double w = exp(s[j] - m);"),
    "empty_row_lse": ("*li = -INFINITY;", "*li = 0.0;"),
    "query_head_index": ("const float *qi = q + ((b * nq + i) * Hq + h) * D;",
                         "const float *qi = q + ((b * nq + i) * Hq + hk) * D;"),
    "merge_weight_max": ("const double w = exp(lse_parts[p * rows + r] - L);",
                         "const double w = exp(lse_parts[p * rows + r] - m);"),
    "merge_lse_drop_max": ("lse[r] = L;", "lse[r] = log(sum);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(path),
                    "-o", str(so), "-lm"], check=True)
    lib = oracle.bind_variant(str(so))
    attn = functools.partial(oracle.attention, _lib=lib)
    merge = functools.partial(oracle.merge, _lib=lib)
    checks = [functools.partial(p, attn) for p in pins.ATTENTION_PINS]
    checks += [functools.partial(pins.pin_chunking_invariance, attn, merge),
               functools.partial(pins.pin_golden_merge, merge)]
    caught = []
    for c in checks:
        try:
            c()
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(c.func.__name__)
    assert caught, f"no pin caught mutant {name}"

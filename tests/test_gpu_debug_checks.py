"""The small parity cases again, against a library built with -DCPATTN_DEBUG:
every kernel then checks each destination row, workspace slot, partial-slot
range and progress counter it touches, skips an out-of-range access and sets
a device status bit instead of trapping.  The run must stay parity-green and
leave every status word clear (checked after each test)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Small cases only: every kernel and launch mode, none of the full-size workloads.
SELECT = " or ".join([
    "test_prefill_edge_cases",
    "test_prefill_odd_groups_all_launch_modes",
    "test_prefill_batch_strides_and_mask",
    "test_prefill_workload and (tiny or llama3)",
    "test_prefill_launch_modes_match and llama3",
    "test_partial_bf16_vs_oracle",
    "test_partial_batch_and_strides",
    "test_partial_simt_vs_oracle",
    "test_partial_growing_logits_rescale",
    "test_merge_pairwise_vs_oracle",
    "test_merge_identity_commutes_and_empty",
    "test_decode_vs_oracle",
    "test_decode_no_visible_key",
])


def test_small_parity_cases_under_debug_checks():
    pytest.importorskip("torch")
    from context_ring_attention_cpattn_gb300 import build

    lib = build.build(debug=True)
    env = dict(os.environ, CPATTN_LIBRARY=lib, CPATTN_CHECK_DEVICE_STATUS="1")
    files = ["tests/test_gpu_prefill.py", "tests/test_gpu_partial.py", "tests/test_gpu_decode.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-q", "-x", "-m", "gpu", "-k", SELECT,
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in tail and " failed" not in tail, tail

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """With CPATTN_CHECK_DEVICE_STATUS=1 every GPU test must leave the
    library's device status words clear (no timed-out wait, and in a
    -DCPATTN_DEBUG library no failed kernel bounds check)."""
    yield
    if os.environ.get("CPATTN_CHECK_DEVICE_STATUS") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    if request.node.name.startswith("test_single_launch_wait_runs_out"):
        return  # that test makes a wait run out on purpose and clears the word itself
    from context_ring_attention_cpattn_gb300 import binding

    assert binding.device_status(clear=True) == 0, "device status word set"

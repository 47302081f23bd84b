"""cpattn_prefill_noalloc: the entry point for callers that cannot allocate
device memory (a framework whose own pool owns all device memory, or a
latency-critical loop that cannot take cudaMalloc's implicit synchronisation).
Its workspace is a static buffer inside the library; its results must match
cpattn_prefill with a caller-allocated workspace.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.  It must also pass on its own in a
fresh process (the first call on the device sets the buffer up)."""
import ctypes

import pytest

from tests.gpu_util import TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from context_ring_attention_cpattn_gb300 import binding, build

    build.build()
    return binding


def inputs(seed, sq=4096, skv=4096, hq=8, hkv=2, d=128):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    mk = lambda s, h: torch.randn((1, s, h, d), generator=g, device="cuda").to(torch.bfloat16)
    return mk(sq, hq), mk(skv, hkv), mk(skv, hkv)


@pytest.mark.parametrize("mode", [1, 2])
def test_noalloc_matches_prefill_on_two_calls(B, mode):
    n_chunks = 4
    for call, seed in enumerate((101, 202)):  # two calls in a row, different inputs
        q, k, v = inputs(seed)
        assert B.workspace_size(q, k, n_chunks, mode) <= (64 << 20)
        ref_o, ref_l = B.prefill(q, k, v, n_chunks, mode)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((1, q.shape[2], q.shape[1]), float("nan"), device="cuda")
        qv, kv, vv, ov = B.view(q), B.view(k), B.view(v), B.view(o)
        status = B.lib().cpattn_prefill_noalloc(
            ctypes.byref(qv), ctypes.byref(kv), ctypes.byref(vv), 0, n_chunks, mode, 1, 0.0,
            ctypes.byref(ov), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert status == 0, B.lib().cpattn_status_string(status)
        torch.cuda.synchronize()
        d_o = (o.float() - ref_o.float()).abs().max().item()
        d_l = (lse - ref_l).abs().max().item()
        assert d_o <= TOL["bf16"][0] and d_l <= TOL["bf16"][1], (call, d_o, d_l)


def test_noalloc_rejects_problems_beyond_its_buffer(B):
    q, k, v = inputs(7, sq=65536, skv=65536, hq=4, hkv=1)   # Pass-Q: fp32 partials, > 64 MiB
    assert B.workspace_size(q, k, 8, 2) > (64 << 20)
    with pytest.raises(B.CpattnError) as err:
        B.prefill_noalloc(q, k, v, 8, 2)
    assert err.value.status == 2   # CPATTN_ERR_UNSUPPORTED, nothing enqueued

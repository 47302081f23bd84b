"""Pass-Q decode (cpattn_decode): a few query tokens against a CP-sharded KV
cache, split into pieces per chunk and merged by LSE, against the fp64 oracle."""
import numpy as np
import pytest

from tests.gpu_util import TOL, compare, oracle_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from context_ring_attention_cpattn_gb300 import binding, build

    build.build()
    return binding


# (n_tok, hq, hkv, skv, n_chunks, q_base, causal, batch, dtype, d)
CASES = [
    (1, 16, 1, 8192, 4, 8191, True, 1, "bf16", 128),      # one token, GQA 16:1 packed
    (8, 16, 1, 8192, 4, 8184, True, 1, "bf16", 128),      # 8 tokens fill the packed tile
    (4, 32, 8, 4096, 8, 3000, True, 2, "bf16", 128),      # GQA 4:1, later chunks invisible, batch 2
    (1, 8, 8, 2048, 2, 2047, True, 1, "bf16", 128),       # no GQA (group of 1)
    (3, 16, 1, 6144, 3, 5000, True, 1, "bf16", 128),      # ragged piece ends
    (16, 16, 1, 4096, 4, 4080, True, 1, "bf16", 128),     # 256 packed rows: one tile per head
    (2, 4, 2, 1024, 4, 1000, False, 1, "bf16", 128),      # no mask
    (2, 4, 1, 512, 2, 500, True, 1, "fp32", 64),          # fp32 kernel
    (1, 16, 1, 131072, 16, 131071, True, 1, "bf16", 128),  # long cache, many pieces
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_decode_vs_oracle(B, case):
    n_tok, hq, hkv, skv, n, q_base, causal, bsz, dt, d = case
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device="cuda")
    g.manual_seed(n_tok * 1000 + skv)
    q = torch.randn((bsz, n_tok, hq, d), generator=g, device="cuda").to(dtype)
    k = torch.randn((bsz, skv, hkv, d), generator=g, device="cuda").to(dtype)
    v = torch.randn((bsz, skv, hkv, d), generator=g, device="cuda").to(dtype)
    o, lse = B.decode(q, k, v, n, q_base=q_base, causal=causal)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    rows = np.arange(n_tok)
    for b in range(bsz):
        ref_o, ref_l = oracle_rows(q[b:b + 1], k[b:b + 1], v[b:b + 1], rows, q_base=q_base,
                                   causal=causal)
        compare(o[b:b + 1], lse[b:b + 1], rows, ref_o, ref_l, TOL[dt], f"decode {case} b{b}")
    # Bitwise reproducible.
    o2, lse2 = B.decode(q, k, v, n, q_base=q_base, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_decode_no_visible_key(B):
    """Tokens before every cached key: O = 0, LSE = -inf, no workspace needed."""
    q = torch.randn((1, 2, 4, 128), device="cuda").to(torch.bfloat16)
    k = torch.randn((1, 256, 1, 128), device="cuda").to(torch.bfloat16)
    assert B.decode_workspace_size(q, k, 2, q_base=-10) == 0
    o, lse = B.decode(q, k, k, 2, q_base=-10)
    torch.cuda.synchronize()
    assert torch.isneginf(lse).all() and (o == 0).all()


def test_decode_bench_workload(B):
    """The benchmark's decode workload (8 sequences x 1 token vs 128K cached keys,
    16 CP ranks), every output row against the oracle."""
    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS["decode-128k-b8"]
    q, k, v = make_qkv(w, device="cuda")
    o, lse = B.decode(q, k, v, w.n_chunks, q_base=w.q_base, causal=w.causal)
    torch.cuda.synchronize()
    rows = np.arange(w.sq)
    for b in range(w.batch):
        ref_o, ref_l = oracle_rows(q[b:b + 1], k[b:b + 1], v[b:b + 1], rows, q_base=w.q_base)
        compare(o[b:b + 1], lse[b:b + 1], rows, ref_o, ref_l, TOL["bf16"], f"decode bench b{b}")

"""cpattn_partial and cpattn_merge on the GPU against the fp64 oracle."""
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


def rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * scale
    return x.to(dtype)


# (sq, skv, hq, hkv, d, q_off, kv_off, causal)
TC_CASES = [
    (128, 128, 2, 1, 128, 0, 0, True),          # one tile, diagonal
    (512, 512, 4, 1, 128, 0, 0, True),          # several tiles, GQA 4:1
    (300, 700, 4, 2, 128, 400, 0, True),        # ragged tails, unaligned offset
    (256, 384, 2, 2, 128, 77, 13, True),        # Hq == Hkv (one tile per CTA)
    (200, 333, 16, 1, 128, 1000, 500, True),    # GQA 16:1, fully visible keys
    (257, 129, 6, 3, 128, 5, 60, True),         # odd group size, rows with no key
    (384, 640, 8, 2, 128, 0, 0, False),         # no mask
    (130, 1000, 2, 1, 128, 20, 900, True),      # most rows empty (keys in the future)
    (1, 1, 2, 1, 128, 0, 0, True),              # single row and key
    (64, 0, 2, 1, 128, 0, 0, True),             # no keys at all
    (700, 700, 3, 3, 128, 0, 0, True),          # MHA: two row blocks of one head per CTA
    (300, 500, 6, 2, 128, 100, 0, True),        # odd group size 3, ragged row pair
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_partial_bf16_vs_oracle(B, case, out_dtype):
    sq, skv, hq, hkv, d, q_off, kv_off, causal = case
    q = rand((1, sq, hq, d), torch.bfloat16, 1)
    k = rand((1, skv, hkv, d), torch.bfloat16, 2)
    v = rand((1, skv, hkv, d), torch.bfloat16, 3)
    od = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    o, lse = B.partial(q, k, v, q_off, kv_off, causal, out_dtype=od)
    torch.cuda.synchronize()
    rows = np.arange(sq)
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=q_off, kv_pos0=kv_off, causal=causal)
    compare(o, lse, rows, ref_o, ref_l, TOL["bf16"], f"partial {case}")
    assert B.device_status() == 0


def test_partial_batch_and_strides(B):
    """Batch 2 and a non-contiguous q (a slice of a wider buffer)."""
    base = rand((2, 300, 4, 256), torch.bfloat16, 4)
    q = base[..., 64:192]
    k = rand((2, 500, 2, 128), torch.bfloat16, 5)
    v = rand((2, 500, 2, 128), torch.bfloat16, 6)
    o, lse = B.partial(q, k, v, 250, 0, True)
    torch.cuda.synchronize()
    for b in range(2):
        rows = np.arange(300)
        ref_o, ref_l = oracle_rows(q[b:b + 1], k[b:b + 1], v[b:b + 1], rows, q_base=250)
        compare(o[b:b + 1], lse[b:b + 1], rows, ref_o, ref_l, TOL["bf16"], f"batch {b}")


SIMT_CASES = [
    ("fp32", 64, 256, 256, 1, 1, 0, 0, True),
    ("fp32", 64, 100, 333, 4, 2, 250, 10, True),
    ("fp32", 128, 65, 190, 2, 1, 3, 0, True),
    ("fp32", 128, 70, 90, 2, 2, 0, 0, False),
    ("bf16", 64, 200, 300, 4, 1, 120, 0, True),
]


@pytest.mark.parametrize("case", SIMT_CASES, ids=lambda c: "x".join(map(str, c)))
def test_partial_simt_vs_oracle(B, case):
    dt, d, sq, skv, hq, hkv, q_off, kv_off, causal = case
    dtype = torch.float32 if dt == "fp32" else torch.bfloat16
    q = rand((1, sq, hq, d), dtype, 7)
    k = rand((1, skv, hkv, d), dtype, 8)
    v = rand((1, skv, hkv, d), dtype, 9)
    o, lse = B.partial(q, k, v, q_off, kv_off, causal)
    torch.cuda.synchronize()
    rows = np.arange(sq)
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=q_off, kv_pos0=kv_off, causal=causal)
    compare(o, lse, rows, ref_o, ref_l, TOL[dt], f"simt {case}")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_merge_pairwise_vs_oracle(B, dtype):
    """Merging the partials of two disjoint key ranges gives the full result."""
    import oracle

    dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    sq, skv, hq, d = 333, 600, 4, 128
    q = rand((1, sq, hq, d), torch.bfloat16, 10)
    k = rand((1, skv, 1, d), torch.bfloat16, 11)
    v = rand((1, skv, 1, d), torch.bfloat16, 12)
    cut = 250
    oa, la = B.partial(q, k[:, :cut], v[:, :cut], 300, 0, True, out_dtype=dt)
    ob, lb = B.partial(q, k[:, cut:], v[:, cut:], 300, cut, True, out_dtype=dt)
    B.merge_(oa, la, ob, lb)
    torch.cuda.synchronize()
    rows = np.arange(sq)
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=300)
    compare(oa, la, rows, ref_o, ref_l, TOL["bf16"], "merge")
    # Against the oracle's own merge of the same GPU partials (fp32 inputs).
    if dtype == "fp32":
        oa2, la2 = B.partial(q, k[:, :cut], v[:, :cut], 300, 0, True, out_dtype=dt)
        pa = (oa2.double().cpu().numpy(), la2.double().cpu().numpy().transpose(0, 2, 1))
        pb = (ob.double().cpu().numpy(), lb.double().cpu().numpy().transpose(0, 2, 1))
        mo, ml = oracle.merge(np.stack([pa[0], pb[0]]), np.stack([pa[1], pb[1]]))
        np.testing.assert_allclose(oa.double().cpu().numpy(), mo, rtol=0, atol=1e-5)
        fin = np.isfinite(ml)
        np.testing.assert_allclose(la.double().cpu().numpy().transpose(0, 2, 1)[fin], ml[fin],
                                   rtol=0, atol=1e-5)


def test_merge_identity_commutes_and_empty(B):
    shape = (1, 257, 3, 128)
    o1 = rand(shape, torch.float32, 13)
    l1 = rand((1, 3, 257), torch.float32, 14) * 5
    o2 = rand(shape, torch.float32, 15)
    l2 = rand((1, 3, 257), torch.float32, 16) * 5
    # identity: merging an empty partial (-inf, 0) changes nothing
    a, la = o1.clone(), l1.clone()
    B.merge_(a, la, torch.zeros_like(o1), torch.full_like(l1, -float("inf")))
    torch.testing.assert_close(a, o1, rtol=0, atol=1e-6)
    torch.testing.assert_close(la, l1, rtol=0, atol=1e-6)
    # commutativity, bitwise
    x, lx = o1.clone(), l1.clone()
    y, ly = o2.clone(), l2.clone()
    B.merge_(x, lx, o2, l2)
    B.merge_(y, ly, o1, l1)
    assert torch.equal(x, y) and torch.equal(lx, ly)
    # both sides empty: no NaN
    e, le = torch.zeros_like(o1), torch.full_like(l1, -float("inf"))
    B.merge_(e, le, torch.zeros_like(o1), torch.full_like(l1, -float("inf")))
    torch.cuda.synchronize()
    assert torch.isneginf(le).all() and (e == 0).all()


def test_argument_errors_do_not_launch(B):
    q = rand((1, 64, 4, 96), torch.bfloat16, 1)
    with pytest.raises(B.CpattnError) as err:
        B.partial(q, q[:, :, :1], q[:, :, :1])
    assert err.value.status == 2   # head_dim 96 unsupported


@pytest.mark.parametrize("hq,hkv", [(4, 1), (3, 3)], ids=["head_pairs", "row_pairs"])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_partial_growing_logits_rescale(B, hq, hkv, out_dtype):
    """Keys whose scale grows along the sequence make every row's running
    maximum grow by more than the lazy-rescale threshold again and again, so
    O is rescaled in TMEM at many KV steps (the softmax then waits for the
    previous step's PV MMA): every row against the oracle."""
    sq, skv = 640, 1536
    q = rand((1, sq, hq, 128), torch.bfloat16, 41)
    ramp = (1.0 + torch.arange(skv, device="cuda", dtype=torch.float32) / 48.0).view(1, skv, 1, 1)
    k = (rand((1, skv, hkv, 128), torch.float32, 42) * ramp).to(torch.bfloat16)
    v = rand((1, skv, hkv, 128), torch.bfloat16, 43)
    od = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    o, lse = B.partial(q, k, v, skv - sq, 0, True, out_dtype=od)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    rows = np.arange(sq)
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=skv - sq)
    compare(o, lse, rows, ref_o, ref_l, TOL["bf16"], f"growing logits {hq}/{hkv}")


def test_profile_records_work_and_time(B):
    """cpattn_profile_begin/end: one record per library launch, with the
    kernel kind, a positive CUDA-event time and the launch's algorithmic work
    (causal-effective FLOPs for attention, bytes for a merge)."""
    q = rand((1, 256, 4, 128), torch.bfloat16, 31)
    k = rand((1, 256, 2, 128), torch.bfloat16, 32)
    v = rand((1, 256, 2, 128), torch.bfloat16, 33)
    B.profile_begin(8)
    try:
        oa, la = B.partial(q, k, v, 0, 0, True, out_dtype=torch.float32)
        ob, lb = B.partial(q, k, v, 0, 0, True, out_dtype=torch.float32)
        B.merge_(oa, la, ob, lb)
    finally:
        recs = B.profile_end(8)
    assert [r[0] for r in recs] == ["attn_tc", "attn_tc", "merge2"]
    assert all(r[1] > 0.0 for r in recs)
    flops = 4.0 * 128 * 4 * (256 * 257 / 2)   # 4 d hq x visible (query, key) pairs
    assert abs(recs[0][2] - flops) <= 1e-9 * flops and abs(recs[1][2] - flops) <= 1e-9 * flops
    merge_bytes = 3 * 256 * 4 * (128 * 4 + 4)  # read both sides, write one (fp32 O + LSE)
    assert abs(recs[2][2] - merge_bytes) <= 1e-9 * merge_bytes

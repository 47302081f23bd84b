"""CP prefill (Pass-KV and Pass-Q) on the five long-context workloads against
the fp64 oracle: every row for the small ones, a seeded sample of query rows
(first and last row of every chunk included) for the large ones.  Pass-KV and
Pass-Q must also agree with each other on every element, and each schedule
must be bitwise reproducible."""
import os

import numpy as np
import pytest

from tests.gpu_util import TOL, compare, oracle_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N_SAMPLE = int(os.environ.get("CPATTN_SAMPLE_ROWS", "4096"))


@pytest.fixture(scope="module")
def B():
    from context_ring_attention_cpattn_gb300 import binding, build

    build.build()
    return binding


@pytest.mark.parametrize("name", ["tiny", "llama3-8b", "partial-32k", "128k", "1m"])
def test_prefill_workload(B, name):
    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv, sample_rows

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    tol = TOL[w.dtype]
    outs = {}
    for mode in (B.PASS_KV, B.PASS_Q):
        o, lse = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        outs[mode] = (o, lse)
    rows = sample_rows(w, n=min(N_SAMPLE, w.sq))
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=w.q_base, causal=w.causal)
    for mode, (o, lse) in outs.items():
        compare(o, lse, rows, ref_o, ref_l, tol, f"{name} mode {mode}")
    # Pass-KV and Pass-Q agree on every element.
    (o1, l1), (o2, l2) = outs[B.PASS_KV], outs[B.PASS_Q]
    d_o = (o1.float() - o2.float()).abs().max().item()
    d_l = (l1 - l2).abs().max().item()
    assert d_o <= tol[0] and d_l <= tol[1], (d_o, d_l)
    # Bitwise reproducible: no atomics, fixed merge order.
    for mode in (B.PASS_KV, B.PASS_Q):
        o, lse = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal)
        torch.cuda.synchronize()
        assert torch.equal(o, outs[mode][0]) and torch.equal(lse, outs[mode][1])
    del outs, q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", [
    # (sq, skv, hq, hkv, n_chunks, q_base, dtype)
    (1000, 1000, 4, 2, 8, 0, "bf16"),       # chunks of 125 rows: ragged tiles everywhere
    (384, 768, 4, 1, 3, 384, "bf16"),       # more keys than queries, partial prefill
    (192, 192, 2, 1, 6, -64, "bf16"),       # first chunks see no key at all
    (240, 240, 2, 2, 5, 0, "fp32"),         # fp32 path, hq == hkv
    (32, 4096, 2, 1, 32, 8192, "bf16"),     # one row per chunk, 32 partials per row
    (640, 640, 3, 3, 5, 0, "bf16"),         # MHA, 128-row chunks (second row block empty)
    (1000, 1000, 6, 2, 8, 0, "bf16"),       # odd group size 3, ragged row pairs
])
def test_prefill_edge_cases(B, case, mode):
    sq, skv, hq, hkv, n, q_base, dt = case
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device="cuda")
    g.manual_seed(sq + skv + n)
    q = torch.randn((1, sq, hq, 128), generator=g, device="cuda").to(dtype)
    k = torch.randn((1, skv, hkv, 128), generator=g, device="cuda").to(dtype)
    v = torch.randn((1, skv, hkv, 128), generator=g, device="cuda").to(dtype)
    o, lse = B.prefill(q, k, v, n, mode, q_base=q_base)
    torch.cuda.synchronize()
    rows = np.arange(sq)
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=q_base)
    compare(o, lse, rows, ref_o, ref_l, TOL[dt], f"edge {case} mode {mode}")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("name,batch", [("llama3-8b", 1), ("partial-32k", 1), ("partial-32k", 2)])
def test_prefill_host_entry_point(B, mode, name, batch):
    """The host-buffer entry point (output rows copied back piece by piece as
    the ring finalises them) gives the same result as the device one."""
    import dataclasses

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv

    w = dataclasses.replace(WORKLOADS[name], batch=batch)
    q, k, v = make_qkv(w, device="cuda")
    o_ref, l_ref = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base)
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.full_like(qh, float("nan")).pin_memory()
    lh = torch.full((batch, w.hq, w.sq), float("nan"), dtype=torch.float32).pin_memory()
    scratch = torch.empty(B.host_scratch_size(qh, kh, w.n_chunks, mode, q_base=w.q_base),
                          dtype=torch.uint8, device="cuda")
    B.prefill_host(qh, kh, vh, w.n_chunks, mode, oh, lh, scratch, q_base=w.q_base)
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())


@pytest.mark.parametrize("mode", [1, 2])
def test_prefill_host_groups_long_items(B, mode):
    """Long items (65536 causal tokens, 8 chunks of 8192, 16/1 heads): the
    host-buffer call works through consecutive groups of Q pieces ({0},
    {1, 2}, {3, 4}, {5, 6}, {7}) so that copies overlap the work -- Pass-KV as
    five on-chip launches, Pass-Q as the ring's pairs grouped by Q piece with
    each group's merge before the next group's pairs -- and gives the device
    call's result bit for bit."""
    g = torch.Generator(device="cuda")
    g.manual_seed(65536)
    sq, n = 65536, 8
    q = torch.randn((1, sq, 16, 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((1, sq, 1, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((1, sq, 1, 128), generator=g, device="cuda").to(torch.bfloat16)
    o_ref, l_ref = B.prefill(q, k, v, n, mode)
    o_ref, l_ref = o_ref.cpu(), l_ref.cpu()
    torch.cuda.empty_cache()
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.full_like(qh, float("nan")).pin_memory()
    lh = torch.full((1, 16, sq), float("nan"), dtype=torch.float32).pin_memory()
    scratch = torch.empty(B.host_scratch_size(qh, kh, n, mode), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    B.profile_begin(256)
    try:
        B.prefill_host(qh, kh, vh, n, mode, oh, lh, scratch)
    finally:
        recs = B.profile_end(256)
    kinds = [r[0] for r in recs if r[0] != "table"]
    if mode == B.PASS_KV:
        assert B.launch_mode(q, k, n, mode) == B.LAUNCH_SINGLE_ONCHIP
        assert kinds == ["attn_tc_onchip"] * 5
    else:
        assert B.launch_mode(q, k, n, mode) == B.LAUNCH_PER_STEP
        # five groups, each: its pairs, then the merge of its pieces (piece 0
        # has one pair, stored directly)
        assert kinds == ["attn_tc"] + ["attn_tc", "mergeN"] * 4
    assert torch.equal(oh, o_ref) and torch.equal(lh, l_ref)


@pytest.mark.parametrize("name", ["tiny", "llama3-8b", "partial-32k", "128k"])
def test_prefill_zigzag_assignment(B, name):
    """Zigzag chunk-to-rank assignment (rank r holds pieces r and 2N-1-r) gives
    the same attention as the contiguous one, for both schedules."""
    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv, sample_rows

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    tol = TOL[w.dtype]
    rows = sample_rows(w, n=min(N_SAMPLE, w.sq, 1024))
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=w.q_base, causal=w.causal)
    base = B.prefill(q, k, v, w.n_chunks, B.PASS_KV, q_base=w.q_base, causal=w.causal)
    for mode in (B.PASS_KV, B.PASS_Q):
        o, lse = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal,
                           assignment=B.ASSIGN_ZIGZAG)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        compare(o, lse, rows, ref_o, ref_l, tol, f"zigzag {name} mode {mode}")
        d_o = (o.float() - base[0].float()).abs().max().item()
        d_l = (lse - base[1]).abs().max().item()
        assert d_o <= tol[0] and d_l <= tol[1], (d_o, d_l)
    del q, k, v, base
    torch.cuda.empty_cache()


@pytest.mark.parametrize("launch", [1, 2, 4], ids=["persistent_step", "single_launch", "single_onchip"])
@pytest.mark.parametrize("name,assignment", [("llama3-8b", 0), ("partial-32k", 0), ("128k", 0),
                                             ("llama3-8b", 1), ("128k", 1)])
def test_prefill_launch_modes_match(B, name, assignment, launch):
    """Persistent CTAs per ring step, and one persistent launch for all ring
    steps (with Pass-KV accumulator updates ordered by progress counters), give
    bitwise the same result as one CTA per work item.  The single launch with
    an on-chip Pass-KV accumulator merges in TMEM instead of through fp32 HBM
    partials, so its Pass-KV result agrees within the tolerance (Pass-Q runs
    as the single launch: bitwise)."""
    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv, sample_rows

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    rows = sample_rows(w, n=min(N_SAMPLE, w.sq, 512))
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=w.q_base, causal=w.causal)
    for mode in (B.PASS_KV, B.PASS_Q):
        o0, l0 = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal,
                           assignment=assignment, launch=B.LAUNCH_PER_STEP)
        o1, l1 = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal,
                           assignment=assignment, launch=launch)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        if launch == B.LAUNCH_SINGLE_ONCHIP and mode == B.PASS_KV:
            tol = TOL[w.dtype]
            assert (o0.float() - o1.float()).abs().max().item() <= tol[0], (name, mode)
            assert (l0 - l1).abs().max().item() <= tol[1], (name, mode)
            o2, l2 = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal,
                               assignment=assignment, launch=launch)
            assert torch.equal(o1, o2) and torch.equal(l1, l2), "on-chip launch not reproducible"
        else:
            assert torch.equal(o0, o1) and torch.equal(l0, l1), (name, mode)
        compare(o1, l1, rows, ref_o, ref_l, TOL[w.dtype], f"{name} launch {launch} mode {mode}")
    del q, k, v
    torch.cuda.empty_cache()


def test_single_launch_wait_runs_out(B):
    """Failure detection without a device fault: with hold_ordered_waits every
    ordered Pass-KV accumulator update of a single launch waits for a progress
    count that nothing reaches.  The bounded wait gives up, the host reads
    CPATTN_ERR_TIMEOUT from cpattn_device_status, and the context stays usable:
    the next call is correct and reports no error."""
    import time

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS["llama3-8b"]
    q, k, v = make_qkv(w, device="cuda")
    o_ref, l_ref = B.prefill(q, k, v, w.n_chunks, B.PASS_KV, launch=B.LAUNCH_SINGLE)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    t0 = time.time()
    B.prefill(q, k, v, w.n_chunks, B.PASS_KV, launch=B.LAUNCH_SINGLE, hold_ordered_waits=True)
    assert B.device_status() == 5   # CPATTN_ERR_TIMEOUT; synchronizes first
    elapsed = time.time() - t0
    assert 1.0 < elapsed < 60.0, elapsed
    assert B.device_status() == 0   # cleared by the previous read
    o, lse = B.prefill(q, k, v, w.n_chunks, B.PASS_KV, launch=B.LAUNCH_SINGLE)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("assignment", [0, 1])
def test_prefill_batch_strides_and_mask(B, mode, causal, assignment):
    """Batch 2, a Q that is a head-dim slice of a wider buffer (row and head
    strides of the view, not of a dense tensor), with and without the causal
    mask, both chunk assignments: every row against the oracle."""
    g = torch.Generator(device="cuda")
    g.manual_seed(4242 + mode)
    base = torch.randn((2, 1024, 8, 256), generator=g, device="cuda").to(torch.bfloat16)
    q = base[..., 128:]
    k = torch.randn((2, 1024, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((2, 1024, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    o, lse = B.prefill(q, k, v, 4, mode, causal=causal, assignment=assignment)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    rows = np.arange(1024)
    for b in range(2):
        ref_o, ref_l = oracle_rows(q[b:b + 1], k[b:b + 1], v[b:b + 1], rows, causal=causal)
        compare(o[b:b + 1], lse[b:b + 1], rows, ref_o, ref_l, TOL["bf16"],
                f"batch {b} mode {mode} causal {causal} assignment {assignment}")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("hkv", [4, 2])
def test_prefill_odd_groups_all_launch_modes(B, mode, hkv):
    """MHA (group size 1) and an odd group size run as row-pair work items: every
    launch mode -- including the single launch, whose Pass-KV ordering counters
    are indexed by 128-row tile -- gives bitwise the same result, and it
    matches the oracle."""
    g = torch.Generator(device="cuda")
    g.manual_seed(77 + hkv)
    hq = 4 if hkv == 4 else 6
    q = torch.randn((1, 2048, hq, 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((1, 2048, hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((1, 2048, hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    outs = []
    for launch in (0, 1, 2):
        o, lse = B.prefill(q, k, v, 4, mode, launch=launch)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    rows = np.arange(2048)
    ref_o, ref_l = oracle_rows(q, k, v, rows)
    compare(outs[0][0], outs[0][1], rows, ref_o, ref_l, TOL["bf16"], f"odd group hkv {hkv} mode {mode}")
    # The on-chip single launch (multi-segment row-pair items) against the oracle.
    o, lse = B.prefill(q, k, v, 4, mode, launch=B.LAUNCH_SINGLE_ONCHIP)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    compare(o, lse, rows, ref_o, ref_l, TOL["bf16"], f"odd group hkv {hkv} mode {mode} on chip")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("name", ["llama3-8b", "partial-32k"])
def test_prefill_graph_capture_replay(B, mode, name):
    """The default launch mode (AUTO; a single persistent launch for these
    short-item workloads -- Pass-KV with its accumulator on chip -- whose pair
    table is uploaded by fill kernels rather than a host copy) can be captured into a CUDA graph: replays on new input
    values give the same bits as eager calls, and match the oracle."""
    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv, sample_rows

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    assert B.launch_mode(q, k, w.n_chunks, mode, w.q_base, w.causal) == (
        B.LAUNCH_SINGLE_ONCHIP if mode == B.PASS_KV else B.LAUNCH_SINGLE)
    o = torch.empty_like(q)
    lse = torch.empty((w.batch, w.hq, w.sq), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, B.workspace_size(q, k, w.n_chunks, mode, w.q_base, w.causal)),
                     dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager warm-up on the capture stream
        B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, out=o, lse=lse, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, out=o, lse=lse, workspace=ws)
    q2, k2, v2 = make_qkv(w, device="cuda", seeds=(11, 12, 13))
    for src_, dst in ((q2, q), (k2, k), (v2, v)):
        dst.copy_(src_)
    o.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert B.device_status() == 0
    o_ref, l_ref = B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    rows = sample_rows(w, n=min(N_SAMPLE, w.sq, 512))
    ref_o, ref_l = oracle_rows(q, k, v, rows, q_base=w.q_base, causal=w.causal)
    compare(o, lse, rows, ref_o, ref_l, TOL[w.dtype], f"graph {name} mode {mode}")
    del graph

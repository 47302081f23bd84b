"""Host-side checks of libcpattn.so that need no GPU: the library loads, it
exports every function include/cpattn.h declares, argument errors come back
as status codes before any CUDA call, and the ring plan -- driven through the
fp64 oracle on the CPU -- reproduces unchunked causal attention."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from context_ring_attention_cpattn_gb300 import binding as B
from context_ring_attention_cpattn_gb300 import build as pkg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(B.EXPORTED)


def declared_struct_fields(name):
    """Field names of a typedef'd struct in the header, in order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*" + name + ";", text).group(1)
    fields = []
    for decl in filter(None, (d.strip() for d in body.split(";"))):
        names = decl.split(None, 1)[1]          # drop the type
        fields += [re.sub(r"[*\s]|\[\d+\]", "", n) for n in names.split(",")]
    return fields


@pytest.mark.parametrize("cname,pyname", [("cpattn_tensor", "CpattnTensor"),
                                          ("cpattn_plan_entry", "PlanEntry"),
                                          ("cpattn_prefill_options", "PrefillOptions"),
                                          ("cpattn_profile_record", "ProfileRecord")])
def test_binding_structs_match_header(cname, pyname):
    fields = [f[0] for f in getattr(B, pyname)._fields_]
    assert declared_struct_fields(cname) == fields


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def T(data=0x10000, dtype=B.BF16, b=1, s=256, h=4, d=128, stride=None):
    if stride is None:
        stride = (s * h * d, h * d, d)
    return B.CpattnTensor(data, dtype, 0, b, s, h, d, *stride)


def call_partial(lib, q, k, v, o, lse=0x20000, q_off=0, kv_off=0):
    return lib.cpattn_partial(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), q_off, kv_off, 1,
                              0.0, ctypes.byref(o), lse, None)


INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.mark.parametrize("case,expect", [
    ("null_q", INVALID), ("bad_dtype", INVALID), ("mixed_dtype", INVALID), ("gqa_indivisible", INVALID),
    ("head_dim_96", UNSUPPORTED), ("misaligned_ptr", INVALID), ("misaligned_stride", INVALID),
    ("kv_len_mismatch", INVALID), ("out_shape", INVALID), ("null_lse", INVALID),
    ("null_data", INVALID), ("batch_mismatch", INVALID)])
def test_partial_argument_errors(lib, case, expect):
    q, k, v, o = T(h=8), T(h=2), T(h=2), T(h=8)
    lse = 0x20000
    if case == "null_q":
        assert lib.cpattn_partial(None, ctypes.byref(k), ctypes.byref(v), 0, 0, 1, 0.0,
                                  ctypes.byref(o), lse, None) == expect
        return
    if case == "bad_dtype":
        q.dtype = 7
    elif case == "mixed_dtype":
        k.dtype = B.FP32
    elif case == "gqa_indivisible":
        q.h, o.h = 6, 6
        k.h, v.h = 4, 4
    elif case == "head_dim_96":
        for t in (q, k, v, o):
            t.d = 96
    elif case == "misaligned_ptr":
        q.data = 0x10008
    elif case == "misaligned_stride":
        k.stride_s = 2 * 128 + 4
    elif case == "kv_len_mismatch":
        v.s = 128
    elif case == "out_shape":
        o.s = 255
    elif case == "null_lse":
        lse = None
    elif case == "null_data":
        q.data = None
    elif case == "batch_mismatch":
        k.b = 2
    assert call_partial(lib, q, k, v, o, lse) == expect


def test_prefill_argument_errors(lib):
    q, k, v, o = T(h=8, s=1024), T(h=1, s=1024), T(h=1, s=1024), T(h=8, s=1024)
    size = ctypes.c_size_t()
    # n_chunks must divide both lengths, lie in 1..64; mode must be 1 or 2.
    for n, mode in ((3, 1), (0, 1), (65, 1), (4, 3)):
        assert lib.cpattn_prefill_workspace_size(ctypes.byref(q), ctypes.byref(k), 0, n, mode, 1,
                                                 ctypes.byref(size)) == INVALID
    per_step = ctypes.byref(B.PrefillOptions(0, B.LAUNCH_PER_STEP))
    assert lib.cpattn_prefill_workspace_size_ex(ctypes.byref(q), ctypes.byref(k), 0, 4, 1, 1,
                                                per_step, ctypes.byref(size)) == 0
    assert size.value == 1024 * 8 * 128 * 4 + 1024 * 8 * 4   # the fp32 accumulator and its LSE
    assert lib.cpattn_prefill_workspace_size(ctypes.byref(q), ctypes.byref(k), 0, 4, 1, 1,
                                             ctypes.byref(size)) == 0
    need = size.value  # the default (AUTO) adds the single launch's pair table and counters
    # Missing / short / misaligned workspace is rejected before any launch.
    args = lambda ws, n: (ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 0, 4, 1, 1, 0.0,
                          ctypes.byref(o), 0x20000, ws, n, None)
    assert lib.cpattn_prefill(*args(None, 0)) == WORKSPACE
    assert lib.cpattn_prefill(*args(0x40000, need - 1)) == WORKSPACE
    assert lib.cpattn_prefill(*args(0x40010, need)) == WORKSPACE


def test_workspace_sizes(lib):
    # Pass-Q keeps one fp32 partial per visible pair of chunks reached more than once.
    q, k = T(h=16, s=4096), T(h=1, s=4096)
    size = ctypes.c_size_t()
    per_step = ctypes.byref(B.PrefillOptions(0, B.LAUNCH_PER_STEP))
    assert lib.cpattn_prefill_workspace_size_ex(ctypes.byref(q), ctypes.byref(k), 0, 4, 2, 1,
                                                per_step, ctypes.byref(size)) == 0
    slots = 2 + 3 + 4   # chunks 1..3 reach 2, 3, 4 KV chunks; chunk 0 reaches one
    per_slot_o, per_slot_l = 1024 * 16 * 128 * 4, 16 * 1024 * 4
    align = lambda x: (x + 255) // 256 * 256
    assert size.value == align(slots * per_slot_o) + align(slots * per_slot_l)


@pytest.mark.parametrize("shape,dtype,want_kv,want_q", [
    ((8192, 8192, 32, 8, 8), B.BF16, B.LAUNCH_SINGLE_ONCHIP, B.LAUNCH_SINGLE),   # 8-tile items
    ((2048, 32768, 16, 1, 8), B.BF16, B.LAUNCH_SINGLE_ONCHIP, B.LAUNCH_SINGLE),  # 32-tile items
    ((131072, 131072, 16, 1, 16), B.BF16, B.LAUNCH_SINGLE_ONCHIP, B.LAUNCH_PER_STEP),  # ~60-tile, K/V in L2
    ((1048576, 1048576, 8, 1, 8), B.BF16, B.LAUNCH_PER_STEP, B.LAUNCH_PER_STEP),  # long items, K/V 512 MiB
    ((8192, 8192, 32, 8, 8), B.FP32, B.LAUNCH_PER_STEP, B.LAUNCH_PER_STEP),      # no tensor cores
])
def test_auto_launch_mode(lib, shape, dtype, want_kv, want_q):
    """CPATTN_LAUNCH_AUTO (the default) resolves, with the tensor-core kernel,
    for Pass-KV to one launch with the accumulator on chip when work items
    are short or K and V fit in L2, and for Pass-Q to one launch for all ring
    steps when work items are short; otherwise, and without the tensor-core
    kernel, to one launch per step.  The default workspace size is the
    resolved mode's."""
    sq, skv, hq, hkv, n = shape
    q_base = skv - sq
    q, k = T(dtype=dtype, s=sq, h=hq), T(dtype=dtype, s=skv, h=hkv)
    for mode, want in ((1, want_kv), (2, want_q)):
        got = ctypes.c_int(-1)
        assert lib.cpattn_prefill_launch_mode(ctypes.byref(q), ctypes.byref(k), q_base, n, mode, 1,
                                              None, ctypes.byref(got)) == 0
        assert got.value == want
        explicit = ctypes.byref(B.PrefillOptions(0, B.LAUNCH_PERSISTENT_STEP))
        assert lib.cpattn_prefill_launch_mode(ctypes.byref(q), ctypes.byref(k), q_base, n, mode, 1,
                                              explicit, ctypes.byref(got)) == 0
        assert got.value == B.LAUNCH_PERSISTENT_STEP
        a, b = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.cpattn_prefill_workspace_size(ctypes.byref(q), ctypes.byref(k), q_base, n, mode, 1,
                                                 ctypes.byref(a)) == 0
        resolved = ctypes.byref(B.PrefillOptions(0, want))
        assert lib.cpattn_prefill_workspace_size_ex(ctypes.byref(q), ctypes.byref(k), q_base, n,
                                                    mode, 1, resolved, ctypes.byref(b)) == 0
        assert a.value == b.value


def test_host_call_takes_the_device_launch_mode(lib):
    """The host-buffer entry point runs the launch mode AUTO picks for the
    device call (at the 128K shape it splits the on-chip Pass-KV launch into
    groups of Q pieces, which needs no more workspace): its scratch is the
    staging buffers plus the device call's workspace, the pair table only, with
    no fp32 accumulator, for long (128K) and short (Llama-3-8B) items alike."""
    align = lambda x: (x + 255) // 256 * 256
    for sq, hq, hkv, n in ((131072, 16, 1, 16), (8192, 32, 8, 8)):
        q, k = T(dtype=B.BF16, s=sq, h=hq), T(dtype=B.BF16, s=sq, h=hkv)
        scratch, auto, launch = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
        assert lib.cpattn_prefill_host_scratch_size(ctypes.byref(q), ctypes.byref(k), 0, n, 1, 1,
                                                    B.BF16, ctypes.byref(scratch)) == 0
        assert lib.cpattn_prefill_workspace_size(ctypes.byref(q), ctypes.byref(k), 0, n, 1, 1,
                                                 ctypes.byref(auto)) == 0
        assert lib.cpattn_prefill_launch_mode(ctypes.byref(q), ctypes.byref(k), 0, n, 1, 1, None,
                                              ctypes.byref(launch)) == 0
        assert launch.value == B.LAUNCH_SINGLE_ONCHIP
        staging = (align(sq * hq * 128 * 2) + 2 * align(sq * hkv * 128 * 2) +
                   align(sq * hq * 128 * 2) + align(hq * sq * 4))
        assert scratch.value == staging + auto.value
        assert auto.value < sq * hq * 128 * 4   # no accumulator


def test_onchip_workspace_has_no_accumulator(lib):
    """SINGLE_ONCHIP Pass-KV keeps the accumulator on chip: its workspace is
    the pair table alone, SINGLE's adds progress counters and the fp32
    accumulator (O and LSE); an unknown launch mode is an argument error."""
    sq, hq, hkv, n = 8192, 32, 8, 8
    q, k = T(dtype=B.BF16, s=sq, h=hq), T(dtype=B.BF16, s=sq, h=hkv)
    sizes = {}
    for launch in (B.LAUNCH_SINGLE, B.LAUNCH_SINGLE_ONCHIP):
        size = ctypes.c_size_t()
        assert lib.cpattn_prefill_workspace_size_ex(ctypes.byref(q), ctypes.byref(k), 0, n, 1, 1,
                                                    ctypes.byref(B.PrefillOptions(0, launch)),
                                                    ctypes.byref(size)) == 0
        sizes[launch] = size.value
    align = lambda x: (x + 255) // 256 * 256
    acc = align(sq * hq * 128 * 4) + align(hq * sq * 4)
    assert sizes[B.LAUNCH_SINGLE] - sizes[B.LAUNCH_SINGLE_ONCHIP] >= acc
    assert sizes[B.LAUNCH_SINGLE_ONCHIP] < 64 * 1024
    size = ctypes.c_size_t()
    assert lib.cpattn_prefill_workspace_size_ex(ctypes.byref(q), ctypes.byref(k), 0, n, 1, 1,
                                                ctypes.byref(B.PrefillOptions(0, 7)),
                                                ctypes.byref(size)) == 1


def test_status_strings(lib):
    for code in range(7):
        assert lib.cpattn_status_string(code).decode().startswith("CPATTN")


# --------------------------------------------------------------------- the ring plan
def plan_cases():
    return [(256, 256, 0, 4, True), (256, 256, 0, 4, False), (2048, 32768, 30720, 8, True),
            (96, 192, 40, 3, True), (64, 64, 0, 1, True), (120, 120, -50, 5, True),
            (64, 64, 500, 8, True)]


@pytest.mark.parametrize("sq,skv,q_base,n,causal", plan_cases())
@pytest.mark.parametrize("mode", [B.PASS_KV, B.PASS_Q])
def test_plan_structure(lib, sq, skv, q_base, n, causal, mode):
    plan = B.prefill_plan(sq, skv, n, mode, q_base, causal)
    cq, c = sq // n, skv // n
    visible = {(i, j) for i in range(n) for j in range(n)
               if (not causal) or j * c <= q_base + i * cq + cq - 1}
    assert sorted((e[1], e[2]) for e in plan) == sorted(visible)
    steps = [e[0] for e in plan]
    assert steps == sorted(steps)
    for step, i, j, role, slot in plan:
        if mode == B.PASS_KV:
            assert j == (i - step) % n      # rank i holds Q chunk i, K/V travel
        else:
            assert i == (j - step) % n      # rank j holds K/V chunk j, Q travel
    for t in set(steps):
        ranks = [e[1] if mode == B.PASS_KV else e[2] for e in plan if e[0] == t]
        assert len(ranks) == len(set(ranks))  # one pair per rank per step
    slots = [e[4] for e in plan if e[3] == 4]
    assert len(slots) == len(set(slots))


def emulate_plan(q, k, v, n, mode, q_base, causal, assignment=B.ASSIGN_CONTIGUOUS):
    """Run the library's plan on the CPU with oracle partials and merges."""
    Bsz, sq, hq, d = q.shape
    skv = k.shape[1]
    pieces = 2 * n if assignment == B.ASSIGN_ZIGZAG else n
    cq, c = sq // pieces, skv // pieces
    plan = B.prefill_plan(sq, skv, n, mode, q_base, causal, assignment)
    out_o = np.full((Bsz, sq, hq, d), np.nan)
    out_l = np.full((Bsz, hq, sq), np.nan)
    acc = {}
    slots = {}
    for step, i, j, role, slot in plan:
        o, lse = oracle.attention(q[:, i * cq:(i + 1) * cq], k[:, j * c:(j + 1) * c],
                                  v[:, j * c:(j + 1) * c],
                                  q_pos=q_base + np.arange(i * cq, (i + 1) * cq), kv_pos0=j * c,
                                  causal=causal)
        lse_t = np.transpose(lse, (0, 2, 1))
        name = B.ROLE_NAMES[role]
        if name == "store":
            out_o[:, i * cq:(i + 1) * cq], out_l[:, :, i * cq:(i + 1) * cq] = o, lse
        elif name == "acc_init":
            acc[i] = (o, lse_t)
        elif name in ("acc_merge", "acc_final"):
            mo, ml = oracle.merge(np.stack([acc[i][0], o]), np.stack([acc[i][1], lse_t]))
            acc[i] = (mo, ml)
            if name == "acc_final":
                out_o[:, i * cq:(i + 1) * cq] = mo
                out_l[:, :, i * cq:(i + 1) * cq] = np.transpose(ml, (0, 2, 1))
        else:
            slots[slot] = (i, j, o, lse_t)
    for i in range(pieces):
        parts = sorted((s, val) for s, val in slots.items() if val[0] == i)
        if parts:
            assert [val[1] for _, val in parts] == sorted(val[1] for _, val in parts)
            mo, ml = oracle.merge(np.stack([val[2] for _, val in parts]),
                                  np.stack([val[3] for _, val in parts]))
            out_o[:, i * cq:(i + 1) * cq] = mo
            out_l[:, :, i * cq:(i + 1) * cq] = np.transpose(ml, (0, 2, 1))
        elif np.isnan(out_l[:, :, i * cq:(i + 1) * cq]).all():
            out_o[:, i * cq:(i + 1) * cq] = 0.0         # no key reaches this chunk
            out_l[:, :, i * cq:(i + 1) * cq] = -np.inf
    return out_o, out_l


@pytest.mark.parametrize("sq,skv,q_base,n,causal", plan_cases())
@pytest.mark.parametrize("mode", [B.PASS_KV, B.PASS_Q])
def test_plan_reproduces_full_attention(lib, sq, skv, q_base, n, causal, mode):
    if skv > 4096:
        sq, skv, q_base = sq // 16, skv // 16, q_base // 16
    rng = np.random.default_rng(sq + skv + n)
    q = rng.standard_normal((1, sq, 2, 8)).astype(np.float32)
    k = rng.standard_normal((1, skv, 1, 8)).astype(np.float32)
    v = rng.standard_normal((1, skv, 1, 8)).astype(np.float32)
    o, lse = emulate_plan(q, k, v, n, mode, q_base, causal)
    ref_o, ref_l = oracle.attention(q, k, v, q_pos=q_base + np.arange(sq), causal=causal)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=0, atol=1e-12)


def test_decode_workspace_sizes(lib):
    size = ctypes.c_size_t()
    # One token at the end of a 131072-key cache, 16 q heads on 1 kv head, 16 chunks:
    # pieces of 256 keys (total keys / 1024 CTAs, at least 256) -> 512 fp32 partials.
    q, k = T(s=1, h=16), T(s=131072, h=1)
    assert lib.cpattn_decode_workspace_size(ctypes.byref(q), ctypes.byref(k), 131071, 16, 1,
                                            ctypes.byref(size)) == 0
    align = lambda x: (x + 255) // 256 * 256
    assert size.value == align(512 * 16 * 128 * 4) + align(512 * 16 * 4)
    # A token at position 1000 sees only the first chunk's first 1001 keys: 4 pieces.
    assert lib.cpattn_decode_workspace_size(ctypes.byref(q), ctypes.byref(k), 1000, 16, 1,
                                            ctypes.byref(size)) == 0
    assert size.value == align(4 * 16 * 128 * 4) + align(4 * 16 * 4)
    # n_chunks must divide the cache length.
    assert lib.cpattn_decode_workspace_size(ctypes.byref(q), ctypes.byref(k), 0, 3, 1,
                                            ctypes.byref(size)) == INVALID


# --------------------------------------------------------------------- zigzag assignment
@pytest.mark.parametrize("sq,skv,q_base,n,causal", [(256, 256, 0, 4, True), (240, 240, 0, 3, True),
                                                    (160, 320, 160, 4, True), (128, 128, 0, 2, False)])
@pytest.mark.parametrize("mode", [B.PASS_KV, B.PASS_Q])
def test_zigzag_plan_reproduces_full_attention(lib, sq, skv, q_base, n, causal, mode):
    rng = np.random.default_rng(sq + n)
    q = rng.standard_normal((1, sq, 2, 8)).astype(np.float32)
    k = rng.standard_normal((1, skv, 1, 8)).astype(np.float32)
    v = rng.standard_normal((1, skv, 1, 8)).astype(np.float32)
    o, lse = emulate_plan(q, k, v, n, mode, q_base, causal, B.ASSIGN_ZIGZAG)
    ref_o, ref_l = oracle.attention(q, k, v, q_pos=q_base + np.arange(sq), causal=causal)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", [B.PASS_KV, B.PASS_Q])
def test_zigzag_plan_structure(lib, mode):
    n = 4
    plan = B.prefill_plan(512, 512, n, mode, 0, True, B.ASSIGN_ZIGZAG, full=True)
    owner = lambda piece: piece if piece < n else 2 * n - 1 - piece
    seen = set()
    for step, qp, kp, role, slot, launch, rank in plan:
        # Pass-KV: the rank owns the Q piece and receives K/V of rank (r - t) mod n;
        # Pass-Q: the rank owns the K/V piece and receives Q of rank (r - t) mod n.
        if mode == B.PASS_KV:
            assert owner(qp) == rank and owner(kp) == (rank - step) % n
        else:
            assert owner(kp) == rank and owner(qp) == (rank - step) % n
        seen.add((qp, kp))
    assert seen == {(i, j) for i in range(2 * n) for j in range(2 * n) if j <= i}
    # No Q piece is written twice by one launch (accumulator updates stay ordered).
    per_launch = {}
    for step, qp, kp, role, slot, launch, rank in plan:
        if role != 4:
            assert (launch, qp) not in per_launch
            per_launch[(launch, qp)] = True


def test_critical_path_balance(lib):
    """Contiguous chunks leave the causal ring about half idle (each step waits
    for the rank with the most visible keys); zigzag pieces balance it."""
    n, s = 8, 8192
    for mode in (B.PASS_KV, B.PASS_Q):
        crit_c, tot_c, _ = B.critical_path(s, s, n, mode, 0, True, B.ASSIGN_CONTIGUOUS)
        crit_z, tot_z, steps = B.critical_path(s, s, n, mode, 0, True, B.ASSIGN_ZIGZAG)
        assert tot_c == tot_z == s * (s + 1) / 2
        c = s // n  # closed form for contiguous chunks: one diagonal step, n-1 full steps
        assert crit_c == c * (c + 1) / 2 + (n - 1) * c * c
        assert tot_c / (n * crit_c) < 0.55
        assert tot_z / (n * crit_z) > 0.98
        assert len(steps) == n and abs(sum(steps) - crit_z) < 1e-6


def test_choose_mode_traffic_model(lib):
    """Full prefill with GQA 16:1 moves far fewer bytes as K/V; a decode-shaped
    query (a few tokens against a long cache) moves fewer bytes as Q."""
    m, kvb, qb = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    def choose(sq, hq, skv, hkv, n):
        q, k = T(s=sq, h=hq), T(s=skv, h=hkv)
        assert lib.cpattn_prefill_choose_mode(ctypes.byref(q), ctypes.byref(k), n, ctypes.byref(m),
                                              ctypes.byref(kvb), ctypes.byref(qb)) == 0
        return m.value, kvb.value, qb.value
    mode, kv, qq = choose(131072, 16, 131072, 1, 16)
    assert mode == B.PASS_KV and kv == 16 * 15 * 2 * 8192 * 128 * 2
    assert qq == 16 * 15 * 8192 * 16 * (128 * 2 * 2 + 4)
    mode, kv, qq = choose(16, 16, 131072, 1, 16)
    assert mode == B.PASS_Q
    # The 32K partial prefill: 2 MiB of K/V vs ~2 MiB of Q + returned O per hop.
    mode, kv, qq = choose(2048, 16, 32768, 1, 8)
    assert mode == B.PASS_KV and qq > kv


def choose_ex(lib, sq, hq, skv, hkv, n, q_base=0, causal=True, assignment=B.ASSIGN_CONTIGUOUS,
              d=128):
    m, kvb, qb = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    q, k = T(s=sq, h=hq, d=d), T(s=skv, h=hkv, d=d)
    assert lib.cpattn_prefill_choose_mode_ex(ctypes.byref(q), ctypes.byref(k), q_base, n,
                                             int(causal), B._opts(assignment), ctypes.byref(m),
                                             ctypes.byref(kvb), ctypes.byref(qb)) == 0
    return m.value, kvb.value, qb.value


def test_choose_mode_ex_causal_hops(lib):
    """Hand-counted ring traffic.  Causal self-prefill, 4 contiguous chunks:
    K/V chunk j is needed by ranks j+1..3, which the ring reaches first, so
    the chunks make 3 + 2 + 1 + 0 = 6 hops; Q chunk i needs ranks 0..i-1,
    which the ring reaches last, so Q chunks 1, 2, 3 make 3 hops each (9);
    6 remote pairs return a partial.  Without the mask every chunk makes 3
    hops and 12 pairs return."""
    c = 256 // 4
    kv_chunk = 2 * c * 1 * 128 * 2          # K and V of one chunk, 1 kv head, bf16
    q_chunk = c * 4 * 128 * 2               # Q of one chunk, 4 q heads
    ret = c * 4 * (128 * 2 + 4)             # one partial O (bf16) and its LSE
    mode, kv, qq = choose_ex(lib, 256, 4, 256, 1, 4)
    assert kv == 6 * kv_chunk and qq == 9 * q_chunk + 6 * ret and mode == B.PASS_KV
    mode, kv, qq = choose_ex(lib, 256, 4, 256, 1, 4, causal=False)
    assert kv == 12 * kv_chunk and qq == 12 * q_chunk + 12 * ret
    # A single chunk never travels.
    assert choose_ex(lib, 256, 4, 256, 1, 1)[1:] == (0.0, 0.0)


def test_choose_mode_ex_partial_prefill_and_decode(lib):
    """Partial prefill (2048 new tokens at 30720.. against 32768 cached keys,
    8 ranks): every new token sees every cached chunk, so each chunk makes all
    7 hops and all 56 remote pairs return -- the same counts as the unmasked
    model.  A decode-shaped query (16 tokens at the end of a 128K cache)
    travels as Q."""
    mode, kv, qq = choose_ex(lib, 2048, 16, 32768, 1, 8, q_base=30720)
    assert kv == 8 * 7 * 2 * 4096 * 128 * 2
    assert qq == 8 * 7 * 256 * 16 * 128 * 2 + 56 * 256 * 16 * (128 * 2 + 4)
    assert mode == B.PASS_KV
    mode, kv, qq = choose_ex(lib, 16, 16, 131072, 1, 16, q_base=131072 - 16)
    assert mode == B.PASS_Q and qq < kv


def test_choose_mode_ex_zigzag(lib):
    """Zigzag pieces (rank r holds r and 2N-1-r): every rank's Q sees every
    rank's K/V, so both schedules use all N-1 hops per rank, each hop moving
    two pieces."""
    n, s = 4, 512
    p = s // (2 * n)
    mode, kv, qq = choose_ex(lib, s, 4, s, 1, n, assignment=B.ASSIGN_ZIGZAG)
    assert kv == n * (n - 1) * 2 * p * 1 * 128 * 2 * 2
    visible_remote = 0
    pieces = lambda r: (r, 2 * n - 1 - r)
    for r in range(n):
        for t in range(n):
            if r != t:
                visible_remote += sum(1 for a in pieces(r) for b in pieces(t) if b * p <= a * p + p - 1)
    assert qq == n * (n - 1) * 2 * p * 4 * 128 * 2 + visible_remote * p * 4 * (128 * 2 + 4)


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """A plain C11 program includes include/cpattn.h, links libcpattn.so and
    calls the host-only entry points (plan, critical path, launch mode,
    workspace size, schedule choice, status string) without a GPU."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    libdir = os.path.dirname(B.library_path())
    exe = tmp_path / "abi_from_c"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-L", libdir, "-lcpattn",
           "-Wl,-rpath," + libdir, "-o", str(exe)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    env = dict(os.environ)
    cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    env["LD_LIBRARY_PATH"] = cuda_lib + (":" + env["LD_LIBRARY_PATH"] if env.get("LD_LIBRARY_PATH") else "")
    run = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "FAIL" not in run.stdout

"""Thin Python binding of libcpattn.so (argument marshalling only).

Every function here converts torch tensors into ``cpattn_tensor`` views and
calls the C ABI declared in ``include/cpattn.h``; all arithmetic runs in the
library's CUDA kernels.  If the library has not been built the first call
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

PASS_KV = 1
PASS_Q = 2
BF16, FP32 = 0, 1
ROLE_NAMES = {0: "store", 1: "acc_init", 2: "acc_merge", 3: "acc_final", 4: "partial"}
KERNEL_NAMES = {1: "attn_tc", 2: "attn_simt", 3: "merge2", 4: "mergeN", 5: "table", 6: "attn_tc_onchip"}


class CpattnTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("b", ctypes.c_int64), ("s", ctypes.c_int64), ("h", ctypes.c_int64),
                ("d", ctypes.c_int64), ("stride_b", ctypes.c_int64), ("stride_s", ctypes.c_int64),
                ("stride_h", ctypes.c_int64)]


class PlanEntry(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("q_chunk", ctypes.c_int32),
                ("kv_chunk", ctypes.c_int32), ("role", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("launch", ctypes.c_int32), ("rank", ctypes.c_int32)]


class PrefillOptions(ctypes.Structure):
    _fields_ = [("assignment", ctypes.c_int32), ("launch", ctypes.c_int32),
                ("hold_ordered_waits", ctypes.c_int32), ("reserved", ctypes.c_int32 * 5)]


ASSIGN_CONTIGUOUS, ASSIGN_ZIGZAG = 0, 1
LAUNCH_PER_STEP, LAUNCH_PERSISTENT_STEP, LAUNCH_SINGLE, LAUNCH_AUTO, LAUNCH_SINGLE_ONCHIP = 0, 1, 2, 3, 4


def _opts(assignment: int, launch: int = LAUNCH_AUTO, hold_ordered_waits: bool = False):
    return ctypes.byref(PrefillOptions(int(assignment), int(launch), int(bool(hold_ordered_waits))))


class ProfileRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("ms", ctypes.c_float), ("work", ctypes.c_double)]


EXPORTED = ["cpattn_partial", "cpattn_merge", "cpattn_prefill_workspace_size", "cpattn_prefill",
            "cpattn_prefill_launch_mode",
            "cpattn_prefill_plan", "cpattn_prefill_host_scratch_size", "cpattn_prefill_host",
            "cpattn_prefill_noalloc", "cpattn_decode_workspace_size", "cpattn_decode",
            "cpattn_prefill_ex", "cpattn_prefill_workspace_size_ex", "cpattn_prefill_plan_ex",
            "cpattn_prefill_critical_path", "cpattn_prefill_choose_mode",
            "cpattn_prefill_choose_mode_ex",
            "cpattn_status_string", "cpattn_device_status",
            "cpattn_profile_begin", "cpattn_profile_end"]

_lib = None


class CpattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().cpattn_status_string(status).decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


def library_path() -> str:
    """The in-tree libcpattn.so, or the file CPATTN_LIBRARY names (a debug
    build of the same sources, for instance)."""
    return os.environ.get("CPATTN_LIBRARY") or _build.LIB


def lib():
    """Load libcpattn.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libcpattn.so is not built ({path}); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    T = ctypes.POINTER(CpattnTensor)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sz = ctypes.POINTER(ctypes.c_size_t)
    L.cpattn_partial.argtypes = [T, T, T, i64, i64, i32, f32, T, vp, vp]
    L.cpattn_merge.argtypes = [T, vp, T, vp, vp]
    L.cpattn_prefill_workspace_size.argtypes = [T, T, i64, i32, i32, i32, sz]
    L.cpattn_prefill.argtypes = [T, T, T, i64, i32, i32, i32, f32, T, vp, vp, ctypes.c_size_t, vp]
    L.cpattn_prefill_plan.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(PlanEntry), i32,
                                      ctypes.POINTER(ctypes.c_int)]
    L.cpattn_prefill_host_scratch_size.argtypes = [T, T, i64, i32, i32, i32, i32, sz]
    L.cpattn_prefill_host.argtypes = [T, T, T, i64, i32, i32, i32, f32, T, vp, vp, ctypes.c_size_t,
                                      vp]
    L.cpattn_prefill_noalloc.argtypes = [T, T, T, i64, i32, i32, i32, f32, T, vp, vp]
    L.cpattn_decode_workspace_size.argtypes = [T, T, i64, i32, i32, sz]
    O = ctypes.POINTER(PrefillOptions)
    dp = ctypes.POINTER(ctypes.c_double)
    L.cpattn_prefill_ex.argtypes = [T, T, T, i64, i32, i32, i32, f32, T, vp, vp, ctypes.c_size_t, O,
                                    vp]
    L.cpattn_prefill_workspace_size_ex.argtypes = [T, T, i64, i32, i32, i32, O, sz]
    L.cpattn_prefill_plan_ex.argtypes = [i64, i64, i64, i32, i32, i32, O, ctypes.POINTER(PlanEntry),
                                         i32, ctypes.POINTER(ctypes.c_int)]
    L.cpattn_prefill_critical_path.argtypes = [i64, i64, i64, i32, i32, i32, O, dp, dp, dp]
    L.cpattn_prefill_choose_mode.argtypes = [T, T, i32, ctypes.POINTER(ctypes.c_int), dp, dp]
    L.cpattn_prefill_choose_mode_ex.argtypes = [T, T, i64, i32, i32, O, ctypes.POINTER(ctypes.c_int),
                                                dp, dp]
    L.cpattn_prefill_launch_mode.argtypes = [T, T, i64, i32, i32, i32, O,
                                             ctypes.POINTER(ctypes.c_int)]
    L.cpattn_decode.argtypes = [T, T, T, i64, i32, i32, f32, T, vp, vp, ctypes.c_size_t, vp]
    L.cpattn_status_string.argtypes = [i32]
    L.cpattn_status_string.restype = ctypes.c_char_p
    L.cpattn_device_status.argtypes = [i32]
    L.cpattn_profile_begin.argtypes = [i32]
    L.cpattn_profile_end.argtypes = [ctypes.POINTER(ProfileRecord), i32, ctypes.POINTER(ctypes.c_int)]
    for name in EXPORTED:
        if name != "cpattn_status_string":
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status: int, where: str):
    if status != 0:
        raise CpattnError(status, where)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def view(t) -> CpattnTensor:
    """cpattn_tensor view of a 4-D [b, s, h, d] torch tensor (last dim contiguous)."""
    if t.dim() != 4:
        raise ValueError("expected a [b, s, h, d] tensor")
    if t.shape[3] > 1 and t.stride(3) != 1:
        raise ValueError("the d dimension must be contiguous")
    b, s, h, d = t.shape
    sb, ss, sh, _ = t.stride()
    return CpattnTensor(t.data_ptr(), _dtype_code(t), 0, b, s, h, d, sb, ss, sh)


def _stream(stream=None, device=None) -> int:
    """Raw handle of `stream`, else of the current stream of `device` (the
    device of the call's tensors)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _on(t):
    """Context that makes the device of tensor `t` current for a library call
    (the library launches on the current device)."""
    import contextlib

    import torch

    if t.device.type != "cuda":
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def partial(q, k, v, q_off: int = 0, kv_off: int = 0, causal: bool = True, scale=None,
            out_dtype=None, out=None, lse=None, stream=None):
    """(O, LSE) of one (Q-chunk, KV-chunk) pair; see cpattn_partial."""
    import torch

    B, S, H, D = q.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    qv, kv_, vv, ov = view(q), view(k), view(v), view(out)
    with _on(q):
        _check(lib().cpattn_partial(ctypes.byref(qv), ctypes.byref(kv_), ctypes.byref(vv),
                                    int(q_off), int(kv_off), int(bool(causal)),
                                    float(scale or 0.0), ctypes.byref(ov), lse.data_ptr(),
                                    _stream(stream, q.device)), "cpattn_partial")
    return out, lse


def merge_(o_a, lse_a, o_b, lse_b, stream=None):
    """In place: (o_a, lse_a) <- LSE-merge of (o_a, lse_a) and (o_b, lse_b)."""
    av, bv = view(o_a), view(o_b)
    with _on(o_a):
        _check(lib().cpattn_merge(ctypes.byref(av), lse_a.data_ptr(), ctypes.byref(bv),
                                  lse_b.data_ptr(), _stream(stream, o_a.device)), "cpattn_merge")
    return o_a, lse_a


def workspace_size(q, k, n_chunks: int, mode: int, q_base: int = 0, causal: bool = True,
                   assignment: int = ASSIGN_CONTIGUOUS, launch: int = LAUNCH_AUTO) -> int:
    n = ctypes.c_size_t(0)
    qv, kv_ = view(q), view(k)
    _check(lib().cpattn_prefill_workspace_size_ex(ctypes.byref(qv), ctypes.byref(kv_), int(q_base),
                                                  int(n_chunks), int(mode), int(bool(causal)),
                                                  _opts(assignment, launch), ctypes.byref(n)),
           "cpattn_prefill_workspace_size_ex")
    return n.value


def prefill(q, k, v, n_chunks: int, mode: int, q_base: int = 0, causal: bool = True, scale=None,
            out=None, lse=None, workspace=None, out_dtype=None, stream=None,
            assignment: int = ASSIGN_CONTIGUOUS, launch: int = LAUNCH_AUTO,
            hold_ordered_waits: bool = False):
    """CP prefill of one attention layer on one GPU; see cpattn_prefill_ex.
    ``hold_ordered_waits`` exists only to test failure detection."""
    import torch

    B, S, H, D = q.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    need = workspace_size(q, k, n_chunks, mode, q_base, causal, assignment, launch)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    qv, kv_, vv, ov = view(q), view(k), view(v), view(out)
    with _on(q):
        _check(lib().cpattn_prefill_ex(ctypes.byref(qv), ctypes.byref(kv_), ctypes.byref(vv),
                                       int(q_base), int(n_chunks), int(mode), int(bool(causal)),
                                       float(scale or 0.0), ctypes.byref(ov), lse.data_ptr(),
                                       ws_ptr, ws_len, _opts(assignment, launch, hold_ordered_waits),
                                       _stream(stream, q.device)),
               "cpattn_prefill_ex")
    return out, lse


def decode_workspace_size(q, k, n_chunks: int, q_base: int = 0, causal: bool = True) -> int:
    n = ctypes.c_size_t(0)
    qv, kv_ = view(q), view(k)
    _check(lib().cpattn_decode_workspace_size(ctypes.byref(qv), ctypes.byref(kv_), int(q_base),
                                              int(n_chunks), int(bool(causal)), ctypes.byref(n)),
           "cpattn_decode_workspace_size")
    return n.value


def decode(q, k, v, n_chunks: int, q_base: int = 0, causal: bool = True, scale=None, out=None,
           lse=None, workspace=None, out_dtype=None, stream=None):
    """Pass-Q decode of a few query tokens against a CP-sharded KV cache; see cpattn_decode."""
    import torch

    B, S, H, D = q.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    need = decode_workspace_size(q, k, n_chunks, q_base, causal)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    qv, kv_, vv, ov = view(q), view(k), view(v), view(out)
    with _on(q):
        _check(lib().cpattn_decode(ctypes.byref(qv), ctypes.byref(kv_), ctypes.byref(vv),
                                   int(q_base), int(n_chunks), int(bool(causal)),
                                   float(scale or 0.0), ctypes.byref(ov), lse.data_ptr(), ws_ptr,
                                   ws_len, _stream(stream, q.device)),
               "cpattn_decode")
    return out, lse


def prefill_noalloc(q, k, v, n_chunks: int, mode: int, q_base: int = 0, causal: bool = True,
                    scale=None, out=None, lse=None, stream=None):
    """cpattn_prefill with the library's static workspace (no allocation by
    the library); see cpattn_prefill_noalloc."""
    import torch

    B, S, H, D = q.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    qv, kv_, vv, ov = view(q), view(k), view(v), view(out)
    with _on(q):
        _check(lib().cpattn_prefill_noalloc(ctypes.byref(qv), ctypes.byref(kv_), ctypes.byref(vv),
                                            int(q_base), int(n_chunks), int(mode),
                                            int(bool(causal)), float(scale or 0.0),
                                            ctypes.byref(ov), lse.data_ptr(),
                                            _stream(stream, q.device)), "cpattn_prefill_noalloc")
    return out, lse


def host_scratch_size(q, k, n_chunks, mode, q_base=0, causal=True, out_dtype=None) -> int:
    n = ctypes.c_size_t(0)
    qv, kv_ = view(q), view(k)
    code = _dtype_code(q) if out_dtype is None else (BF16 if str(out_dtype).endswith("bfloat16") else FP32)
    _check(lib().cpattn_prefill_host_scratch_size(ctypes.byref(qv), ctypes.byref(kv_), int(q_base),
                                                  int(n_chunks), int(mode), int(bool(causal)),
                                                  code, ctypes.byref(n)),
           "cpattn_prefill_host_scratch_size")
    return n.value


def prefill_host(q, k, v, n_chunks, mode, out, lse, dev_scratch, q_base=0, causal=True,
                 scale=None, stream=None):
    """End to end from host tensors: H2D copies, prefill, D2H copies, sync."""
    qv, kv_, vv, ov = view(q), view(k), view(v), view(out)
    with _on(dev_scratch):
        _check(lib().cpattn_prefill_host(ctypes.byref(qv), ctypes.byref(kv_), ctypes.byref(vv),
                                         int(q_base), int(n_chunks), int(mode), int(bool(causal)),
                                         float(scale or 0.0), ctypes.byref(ov), lse.data_ptr(),
                                         dev_scratch.data_ptr(),
                                         dev_scratch.numel() * dev_scratch.element_size(),
                                         _stream(stream, dev_scratch.device)), "cpattn_prefill_host")
    return out, lse


def prefill_plan(sq: int, skv: int, n_chunks: int, mode: int, q_base: int = 0,
                 causal: bool = True, assignment: int = ASSIGN_CONTIGUOUS, full: bool = False):
    """Launch-order list of (step, q_piece, kv_piece, role, slot) -- plus
    (launch, rank) when full=True -- computed on the host."""
    n = ctypes.c_int(0)
    _check(lib().cpattn_prefill_plan_ex(int(sq), int(skv), int(q_base), int(n_chunks), int(mode),
                                        int(bool(causal)), _opts(assignment), None, 0,
                                        ctypes.byref(n)), "cpattn_prefill_plan_ex")
    arr = (PlanEntry * max(1, n.value))()
    _check(lib().cpattn_prefill_plan_ex(int(sq), int(skv), int(q_base), int(n_chunks), int(mode),
                                        int(bool(causal)), _opts(assignment), arr, n.value,
                                        ctypes.byref(n)), "cpattn_prefill_plan_ex")
    if full:
        return [(e.step, e.q_chunk, e.kv_chunk, e.role, e.slot, e.launch, e.rank)
                for e in arr[:n.value]]
    return [(e.step, e.q_chunk, e.kv_chunk, e.role, e.slot) for e in arr[:n.value]]


def launch_mode(q, k, n_chunks: int, mode: int, q_base: int = 0, causal: bool = True,
                assignment: int = ASSIGN_CONTIGUOUS, launch: int = LAUNCH_AUTO) -> int:
    """The launch mode cpattn_prefill_ex uses for these shapes (AUTO resolved)."""
    out = ctypes.c_int(0)
    qv, kv_ = view(q), view(k)
    _check(lib().cpattn_prefill_launch_mode(ctypes.byref(qv), ctypes.byref(kv_), int(q_base),
                                            int(n_chunks), int(mode), int(bool(causal)),
                                            _opts(assignment, launch), ctypes.byref(out)),
           "cpattn_prefill_launch_mode")
    return out.value


def choose_mode_ex(q, k, n_chunks: int, q_base: int = 0, causal: bool = True,
                   assignment: int = ASSIGN_CONTIGUOUS):
    """(mode, pass_kv_bytes, pass_q_bytes) counting only the ring hops the
    masked ring needs; see cpattn_prefill_choose_mode_ex."""
    m = ctypes.c_int(0)
    kvb, qb = ctypes.c_double(0.0), ctypes.c_double(0.0)
    qv, kv_ = view(q), view(k)
    _check(lib().cpattn_prefill_choose_mode_ex(ctypes.byref(qv), ctypes.byref(kv_), int(q_base),
                                               int(n_chunks), int(bool(causal)), _opts(assignment),
                                               ctypes.byref(m), ctypes.byref(kvb), ctypes.byref(qb)),
           "cpattn_prefill_choose_mode_ex")
    return m.value, kvb.value, qb.value


def choose_mode(q, k, n_chunks: int):
    """(mode, pass_kv_bytes, pass_q_bytes) from the ring traffic model; see
    cpattn_prefill_choose_mode."""
    m = ctypes.c_int(0)
    kvb, qb = ctypes.c_double(0.0), ctypes.c_double(0.0)
    qv, kv_ = view(q), view(k)
    _check(lib().cpattn_prefill_choose_mode(ctypes.byref(qv), ctypes.byref(kv_), int(n_chunks),
                                            ctypes.byref(m), ctypes.byref(kvb), ctypes.byref(qb)),
           "cpattn_prefill_choose_mode")
    return m.value, kvb.value, qb.value


def critical_path(sq: int, skv: int, n_chunks: int, mode: int, q_base: int = 0,
                  causal: bool = True, assignment: int = ASSIGN_CONTIGUOUS):
    """(critical, total, per-step maxima) of the emulated ring, in visible
    (query, key) pairs per (batch, head); see cpattn_prefill_critical_path."""
    crit, tot = ctypes.c_double(0.0), ctypes.c_double(0.0)
    steps = (ctypes.c_double * n_chunks)()
    _check(lib().cpattn_prefill_critical_path(int(sq), int(skv), int(q_base), int(n_chunks),
                                              int(mode), int(bool(causal)), _opts(assignment),
                                              steps, ctypes.byref(crit), ctypes.byref(tot)),
           "cpattn_prefill_critical_path")
    return crit.value, tot.value, list(steps)


def device_status(clear: bool = True) -> int:
    return lib().cpattn_device_status(int(bool(clear)))


def profile_begin(capacity: int):
    _check(lib().cpattn_profile_begin(int(capacity)), "cpattn_profile_begin")


def profile_end(capacity: int):
    recs = (ProfileRecord * capacity)()
    n = ctypes.c_int(0)
    _check(lib().cpattn_profile_end(recs, capacity, ctypes.byref(n)), "cpattn_profile_end")
    return [(KERNEL_NAMES.get(r.kind, str(r.kind)), r.ms, r.work) for r in recs[:min(n.value, capacity)]]

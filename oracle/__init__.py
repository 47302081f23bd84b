"""CPU fp64 oracle for context-parallel causal attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  It shares no code with the CUDA
library.  It restates the definition of causal softmax attention and of the
LSE-weighted merge that the article "Scaling LLM Inference: Innovations in
Tensor Parallelism, Context Parallelism, and Expert Parallelism" relies on when
it says (section "Context Parallelism for Million-Token Contexts", Pass-KV and
Pass-Q bullets) that each CP rank computes attention over the full context.

Two implementations live here:

* ``attention`` / ``merge``: thin ctypes wrappers over ``cpattn_oracle.c``
  (plain two-pass fp64 loops, OpenMP over (batch, row, head)).
* ``brute.py``: a numpy brute force over the full masked score matrix, used
  only to pin the C oracle on tiny inputs.

Parity of the absolute error scale is unpinned by the pages (they print no
numeric example); the formulas are pinned in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libcpattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O3, OpenMP).  Returns the .so path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, ptr = ctypes.c_int64, ctypes.c_void_p
    lib.cpattn_oracle_attention.restype = ctypes.c_int
    lib.cpattn_oracle_attention.argtypes = [
        ptr, ptr, i64, ptr, ptr, i64, i64, i64, i64, i64, i64,
        ctypes.c_int, ctypes.c_double, ptr, ptr, ctypes.c_int]
    lib.cpattn_oracle_merge.restype = ctypes.c_int
    lib.cpattn_oracle_merge.argtypes = [ptr, ptr, i64, i64, i64, ptr, ptr]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def bind_variant(so_path: str):
    """Load another build of the oracle source (used by the tests that plant a
    mistake in a copy of the oracle and check that a pin catches it)."""
    return _bind(so_path)


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def attention(q, k, v, *, q_pos=None, kv_pos0: int = 0, causal: bool = True,
              scale: float | None = None, threads: int | None = None, _lib=None):
    """fp64 attention of query rows ``q`` against keys/values ``k``, ``v``.

    q: [B, nq, Hq, D]; k, v: [B, Skv, Hkv, D] (any float dtype numpy can hold;
    bf16 values must be widened to float32 by the caller, which is exact).
    q_pos: absolute position of each query row (default 0..nq-1); key row j is
    at absolute position kv_pos0 + j.  Returns (O [B,nq,Hq,D] f64, LSE
    [B,Hq,nq] f64), LSE in natural log, empty rows -> (0, -inf).
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    B, nq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    assert v.shape == k.shape and Bk == B and Dk == D and Hq % Hkv == 0
    if q_pos is None:
        q_pos = np.arange(nq, dtype=np.int64)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    assert q_pos.shape == (nq,)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty((B, nq, Hq, D), dtype=np.float64)
    lse = np.empty((B, Hq, nq), dtype=np.float64)
    rc = (_lib or _load()).cpattn_oracle_attention(
        q.ctypes.data, q_pos.ctypes.data, nq, k.ctypes.data, v.ctypes.data,
        int(kv_pos0), Skv, B, Hq, Hkv, D, int(bool(causal)), float(scale),
        o.ctypes.data, lse.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"cpattn_oracle_attention failed: {rc}")
    return o, lse


def merge(o_parts, lse_parts, _lib=None):
    """LSE-weighted merge of partials over disjoint key sets (fp64).

    o_parts: [P, ..., D]; lse_parts: [P, ...] with the same leading shape.
    Returns (O [..., D], LSE [...]).
    """
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    P = o_parts.shape[0]
    D = o_parts.shape[-1]
    row_shape = o_parts.shape[1:-1]
    assert lse_parts.shape == (P,) + row_shape
    rows = int(np.prod(row_shape)) if row_shape else 1
    o = np.empty(row_shape + (D,), dtype=np.float64)
    lse = np.empty(row_shape, dtype=np.float64)
    rc = (_lib or _load()).cpattn_oracle_merge(o_parts.ctypes.data, lse_parts.ctypes.data,
                                     P, rows, D, o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"cpattn_oracle_merge failed: {rc}")
    return o, lse

"""GB300-native context-parallel ring attention (prefill hot path).

The compute lives in ``libcpattn.so`` (hand-written sm_103a CUDA behind a C
ABI declared in ``include/cpattn.h``); :mod:`.binding` marshals torch tensors
into that ABI.  Importing this package does not load the library; the first
call through :mod:`.binding` does, and raises if it is missing.
"""
from .workloads import WORKLOADS, Workload, make_qkv, sample_rows  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_qkv", "sample_rows"]

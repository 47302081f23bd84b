"""Build libcpattn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library links against
the shared CUDA runtime so it uses the same runtime instance as PyTorch.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libcpattn.so")
SOURCES = ["api.cu", "attn_pair.cu", "attn_tc.cu", "attn_simt.cu", "merge.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps(csrc: str) -> list[str]:
    inc = os.path.join(INCLUDE, "cpattn.h")
    files = [os.path.join(csrc, f) for f in os.listdir(csrc)]
    return files + [inc, os.path.abspath(__file__)]


def _stale(lib: str, csrc: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps(csrc))


DEBUG_DIR = os.path.join(PKG, "_build_debug")


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str = OUT_DIR,
          csrc: str = CSRC, debug: bool = False) -> str:
    """Compile the sources in `csrc` into `out_dir`/libcpattn.so (the in-tree
    library by default).  debug=True builds the same sources with
    -DCPATTN_DEBUG (kernel bounds checks) into _build_debug/."""
    if debug:
        extra_flags = (*extra_flags, "-DCPATTN_DEBUG")
        out_dir = DEBUG_DIR if out_dir == OUT_DIR else out_dir
    lib = os.path.join(out_dir, "libcpattn.so")
    if not force and not _stale(lib, csrc):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", csrc, "-I", INCLUDE, "-c",
               os.path.join(csrc, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))

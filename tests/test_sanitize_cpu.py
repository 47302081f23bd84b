"""The host code of the C ABI and the fp64 oracle under AddressSanitizer and
UndefinedBehaviorSanitizer, on the CPU.

api.cu (argument checks, ring plan, workspace layout, schedule choice) is
compiled with -fsanitize=address,undefined and linked with the library's
other objects into tests/c/sanitize_host.c, which sweeps the host-only entry
points and every argument-error path; the oracle is compiled the same way
into tests/c/sanitize_oracle.c.  Any memory error, leak or undefined
behaviour aborts the program."""
import os
import shutil
import subprocess

import pytest

from context_ring_attention_cpattn_gb300 import build as pkg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-omit-frame-pointer",
       "-fno-sanitize-recover=all", "-g"]
ENV = {"ASAN_OPTIONS": "detect_leaks=1:abort_on_error=0:halt_on_error=1",
       "UBSAN_OPTIONS": "halt_on_error=1:print_stacktrace=1"}


def run(cmd, **kw):
    res = subprocess.run(cmd, capture_output=True, text=True, **kw)
    assert res.returncode == 0, " ".join(cmd) + "\n" + res.stdout[-4000:] + res.stderr[-4000:]
    return res


def cuda_lib_dir():
    return os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")


@pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("nvcc") is None
                    and not os.path.exists("/usr/local/cuda/bin/nvcc"), reason="needs gcc and nvcc")
def test_host_abi_under_sanitizers(tmp_path):
    pkg_build.build()  # the kernels' objects (their host stubs are not instrumented)
    nvcc = pkg_build._nvcc()
    obj = tmp_path / "api_san.o"
    run([nvcc, *pkg_build.ARCH, "-O1", "-std=c++17", "--expt-relaxed-constexpr",
         *[f"-Xcompiler={f}" for f in SAN + ["-fPIC"]], "-I", pkg_build.INCLUDE, "-c",
         os.path.join(pkg_build.CSRC, "api.cu"), "-o", str(obj)])
    others = [os.path.join(pkg_build.OUT_DIR, s.replace(".cu", ".o"))
              for s in pkg_build.SOURCES if s != "api.cu"]
    exe = tmp_path / "sanitize_host"
    run(["g++", *SAN, "-I", os.path.join(ROOT, "include"), "-x", "c",
         os.path.join(ROOT, "tests", "c", "sanitize_host.c"), "-x", "none", str(obj), *others,
         "-L", cuda_lib_dir(), "-lcudart", "-Wl,-rpath," + cuda_lib_dir(), "-o", str(exe)])
    env = dict(os.environ, **ENV)
    res = run([str(exe)], env=env, timeout=300)
    assert "FAIL" not in res.stdout and res.stdout.strip().endswith("(0 failures)")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_oracle_under_sanitizers(tmp_path):
    exe = tmp_path / "sanitize_oracle"
    run(["gcc", "-std=c11", "-O1", "-fopenmp", *SAN,
         os.path.join(ROOT, "tests", "c", "sanitize_oracle.c"),
         os.path.join(ROOT, "oracle", "cpattn_oracle.c"), "-lm", "-o", str(exe)])
    env = dict(os.environ, **ENV)
    # libgomp keeps its thread pool alive at exit: not a leak of the oracle's.
    env["ASAN_OPTIONS"] = env["ASAN_OPTIONS"].replace("detect_leaks=1", "detect_leaks=0")
    res = run([str(exe)], env=env, timeout=300)
    assert "FAIL" not in res.stdout and res.stdout.strip().endswith("(0 failures)")

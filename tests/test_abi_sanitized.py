"""The C ABI's host code under AddressSanitizer and UndefinedBehaviorSanitizer.

ccl_api.cu (argument checks, aliasing rules, descriptor building, the
literal engine's host loop) is recompiled with -fsanitize=address,undefined
and linked with the regular kernel objects into a separate library; the
GPU-free ABI tests then run against it in a child process with the ASan
runtime preloaded.  Any sanitizer report fails the test.  No GPU is used:
every call in tests/test_abi.py is rejected on the host or is a no-op.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

import pytest

from conftest import ROOT


def _runtime(name: str) -> str | None:
    gcc = shutil.which("gcc")
    if gcc is None:
        return None
    path = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_abi_checks_are_clean_under_asan_and_ubsan(tmp_path):
    from a2a_ring_ordered_gb300 import build

    asan = _runtime("libasan.so")
    if asan is None or _runtime("libubsan.so") is None:
        pytest.skip("gcc's ASan / UBSan runtimes are not installed")
    build.build()
    objs = [o for o in glob.glob(os.path.join(build.BUILD, "*.o")) if not o.endswith("ccl_api.cu.o")]
    assert objs, "kernel objects missing after build()"
    san = ["-Xcompiler", "-fPIC,-fsanitize=address,-fsanitize=undefined,-fno-omit-frame-pointer,"
           "-fno-sanitize-recover=undefined"]
    api_obj = str(tmp_path / "ccl_api.o")
    lib = str(tmp_path / "libccl_san.so")
    subprocess.run([build.nvcc(), *build.ARCH, "-O1", "-std=c++17", *san, "-I", build.INCLUDE, "-I", build.CSRC,
                    "-c", os.path.join(build.CSRC, "ccl_api.cu"), "-o", api_obj], check=True)
    subprocess.run([build.nvcc(), *build.ARCH, "-shared", "--cudart", "static",
                    "-Xcompiler", "-fsanitize=address,-fsanitize=undefined", "-o", lib, api_obj, *objs], check=True)
    env = dict(os.environ, LD_PRELOAD=asan, CCL_LIBRARY=lib,
               ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_abi.py"), "-q",
                        "-p", "no:cacheprovider", "-k", "not without_library"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "AddressSanitizer" not in out and "runtime error" not in out, out[-4000:]
    assert lib in subprocess.run([sys.executable, "-c", "from a2a_ring_ordered_gb300 import ccl; print(ccl.LIB_PATH)"],
                                 cwd=ROOT, env=env, capture_output=True, text=True).stdout

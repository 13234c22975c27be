"""The C ABI from a plain C program (tests/c_abi/worked_example.c), with no
Python or torch between the caller and libccl.so.  On the CPU: include/ccl.h
compiles as C11 with warnings as errors and the program links.  On a GPU: the
program runs the worked example of "Networks and Collective Communication"
(section 4.1) and every line it prints matches the golden fixture."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "worked_example.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "worked_example_p4.txt")


def golden() -> dict[str, list[float]]:
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            name, vals = line.split(":", 1)
            out[name.strip()] = [float(v) for v in vals.split()]
    return out


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    from a2a_ring_ordered_gb300 import build, ccl

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc is not installed")
    cuda = os.path.dirname(os.path.dirname(build.nvcc()))
    lib = os.path.abspath(ccl.LIB_PATH)
    out = str(tmp_path_factory.mktemp("c_abi") / "worked_example")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", build.INCLUDE, "-I", os.path.join(cuda, "include"), SRC, "-o", out,
           lib, f"-Wl,-rpath,{os.path.dirname(lib)}",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_header_is_c_and_program_links(exe):
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_worked_example_from_c(exe):
    g = golden()
    args = [f"{v:g}" for r in range(4) for v in g[f"input {r}"]]
    r = subprocess.run([exe, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = {}
    for line in r.stdout.splitlines():
        name, vals = line.split(":", 1)
        got[name.strip()] = [float(v) for v in vals.split()]
    assert len(got) == 12
    for name, vals in got.items():
        assert vals == g[name], f"{name}: {vals} != {g[name]}"

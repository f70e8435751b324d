"""The C ABI from plain C: tests/c/abi_smoke.c includes include/c3_api.h and
links libc3.so.  On the CPU it must compile as C99 with warnings as errors and
link with every declared entry point resolved; on a GPU it runs a GEMM, an
all-gather and a concurrent run through the ABI alone and checks them."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "concurrent_communication_overlap_gb300")
LIB = os.path.join(PKG, "libc3.so")
SRC = os.path.join(ROOT, "tests", "c", "abi_smoke.c")
CUDA = "/usr/local/cuda"


def _build(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("CUDA headers not found")
    if not os.path.exists(LIB):
        pytest.skip("libc3.so is not built")
    exe = str(tmp_path / "abi_smoke")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic-errors", "-Wno-cast-function-type",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA, "include"), SRC, "-o", exe,
           "-L", PKG, "-lc3", "-Wl,-rpath," + PKG, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_header_compiles_as_c99_and_links_every_entry_point(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "21 entry points" in r.stdout


@pytest.mark.gpu
def test_c_program_drives_the_library(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "--run"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi smoke ok" in r.stdout

"""The C-ABI used from C: tests/c/abi_roundtrip.c is compiled with gcc
against include/rar.h, linked with librar.so and the CUDA runtime, and run
(GPU).  The compile-and-link step alone also runs without a GPU."""
import os
import subprocess
import tempfile

import pytest

from ring_all_reduce_rar_gb300 import _build
from tests.conftest import ROOT

SRC = os.path.join(ROOT, "tests", "c", "abi_roundtrip.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out):
    _build.build()
    libdir = os.path.dirname(_build.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(CUDA, "include"), SRC, "-o", out, "-L", libdir, "-lrar", "-L",
           os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True)


def test_c_program_compiles_and_links():
    with tempfile.TemporaryDirectory() as d:
        _compile(os.path.join(d, "abi_roundtrip"))


@pytest.mark.gpu
def test_c_program_runs_the_page_example():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "abi_roundtrip")
        _compile(exe)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "c-abi roundtrip ok" in r.stdout

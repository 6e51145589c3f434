"""The library used from plain C, through include/dpr.h alone: tests/c_consumer.c
is compiled with the host C compiler against the header, linked with libdpr and
the CUDA runtime, and run.  It reduces the pages' worked example (K = 4, chunks
of several tiles) through the reduce-scatter in both modes, the all-gather and
the all-reduce, checks every element against the closed form, and checks that
an invalid call is refused without effect."""
import os
import shutil
import subprocess

import pytest

import gradient_reduction_gb300 as dpr

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    pytest.fail("no CUDA toolkit to compile the C consumer against")


def test_plain_c_consumer(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "no host C compiler"
    libdir = os.path.dirname(dpr.LIB_PATH)
    dpr.lib()                                    # built (raises otherwise)
    cuda = _cuda_home()
    exe = str(tmp_path / "c_consumer")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_consumer.c"), "-o", exe,
           "-L", libdir, "-ldpr", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "C_CONSUMER_OK" in r.stdout, r.stdout + r.stderr

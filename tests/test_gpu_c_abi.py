"""The C ABI from C alone: tests/c_abi_check.c, built with gcc against
include/asr.h, libasr.so and the oracle's library, runs a two-step
multi-tensor AdamW-SR update over three tensors of different dtypes and
bases and a run of Philox words, and compares them byte for byte with the
oracle's C functions."""
import os
import shutil
import subprocess

import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_through_the_abi(tmp_path):
    torch_cuda()
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    from oracle import build as oracle_build
    from stochastic_rounding_gb300 import build as lib_build
    lib = lib_build.build()
    orc = oracle_build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "c_abi_check"
    libdirs = [os.path.dirname(lib), os.path.dirname(orc), os.path.join(cuda, "lib64")]
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           *[f"-L{d}" for d in libdirs], "-lasr", "-loracle", "-lcudart", "-lm",
           *[f"-Wl,-rpath,{d}" for d in libdirs], "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "C_ABI_OK" in r.stdout, r.stdout + r.stderr

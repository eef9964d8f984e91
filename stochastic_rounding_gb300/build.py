"""Build ``libasr.so`` (the CUDA kernels and the C ABI) in-tree for sm_103a.

Device code: every float operation in the kernels is an explicitly rounded
intrinsic; -fmad=false additionally keeps nvcc from contracting anything else.
Host code: -ffp-contract=off so the per-step scalars are formed exactly as
written in binary64 (GCC on aarch64 would otherwise fuse 1 - lr*wd).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "asr.cu")
HDR = os.path.join(ROOT, "include", "asr.h")
# textually included by asr.cu (one translation unit)
INCLUDED = [os.path.join(HERE, "csrc", f) for f in (
    "common.cuh", "pipeline.cuh", "adamw_kernels.cuh", "rounding_kernels.cuh", "static_table.cuh",
    "host_pipeline.cuh", "gemm_sr.cuh")]
LIB = os.path.join(HERE, "libasr.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17", "-fmad=false",
    "-Xcompiler", "-fPIC,-ffp-contract=off,-O2",
    "-shared",
]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if missing or older than its sources."""
    deps = [SRC, HDR, *INCLUDED, __file__]
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(d) for d in deps)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

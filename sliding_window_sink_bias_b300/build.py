"""Build the CUDA library in-tree: nvcc for sm_103a -> libsinkattn.so next to this file."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libsinkattn.so")
# the same sources with -DSINKATTN_TEST_HOOKS -DSINKATTN_CHECKS: the library the
# timeout-path and bounds-check tests load (it can stall one wait on purpose
# and checks every access in the kernels); the product never loads it
TEST_LIB = os.path.join(HERE, "libsinkattn_test.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "shared", "-Xlinker", "-rpath=/usr/local/cuda/lib64",
]


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(HERE, "csrc", "*.cuh"))) + \
        [os.path.join(ROOT, "include", "sinkattn.h")]


def _build_one(out: str, extra, force: bool, verbose: bool) -> None:
    if not force and os.path.exists(out):
        t = os.path.getmtime(out)
        if all(os.path.getmtime(d) <= t for d in deps()):
            return
    cmd = [NVCC, *NVCC_FLAGS, *extra, "-I", os.path.join(ROOT, "include")]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += ["-o", out, *sources()]
    subprocess.run(cmd, check=True)


def build(force: bool = False, verbose: bool = False, test_lib: bool = True) -> str:
    """Compile every .cu under csrc/ into the shared library (and, unless told
    not to, the test build of the same sources); each is skipped when up to
    date.  Returns the product library's path."""
    _build_one(LIB, [], force, verbose)
    if test_lib:
        _build_one(TEST_LIB, ["-DSINKATTN_TEST_HOOKS", "-DSINKATTN_CHECKS"], force, verbose)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

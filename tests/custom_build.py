"""Builds tests/custom/task_processor.cu (a task processor compiled through
include/tg_custom.cuh) against the in-tree libtg."""
import os
import subprocess

from logits_processing_token_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "custom", "task_processor.cu")


def nvcc_cmd(out, shared=True):
    inc = ["-I" + os.path.join(_build.ROOT, "include"), "-I" + _build.CSRC]
    if shared:
        return ([_build.nvcc()] + _build.ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                "-shared", SRC, "-o", out, "-L" + _build.BUILD, "-ltg", "-Xlinker", "-rpath," + _build.BUILD] + inc)
    return ([_build.nvcc()] + _build.ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
            "-c", SRC, "-o", out] + inc)


def build(tmpdir):
    lib = _build.build()
    out = os.path.join(str(tmpdir), "libtask_processor.so")
    r = subprocess.run(nvcc_cmd(out), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(r.stderr)
    return out, lib

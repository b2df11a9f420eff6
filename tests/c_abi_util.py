"""Builds tests/c_abi/layer_step.c, a C program that runs one layer step through include/mm.h and
libmm.so with no Python or PyTorch involved."""
import os
import shutil
import subprocess

from moe_ffn_expert_gb300 import _abi

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if nvcc else None


def build_layer_step(out_dir):
    """Compiles the example with the host C compiler; returns the executable's path."""
    cuda = cuda_home()
    assert cuda, "no CUDA toolkit found"
    lib_dir = os.path.dirname(_abi.LIB_PATH)
    cudart_dirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                               os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                               os.path.join(cuda, "targets", "x86_64-linux", "lib"))
                   if os.path.exists(os.path.join(d, "libcudart.so"))]
    assert cudart_dirs, "libcudart.so not found"
    exe = os.path.join(out_dir, "layer_step")
    cmd = [os.environ.get("CC", "cc"), "-std=c11", "-O2", "-Wall", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "c_abi", "layer_step.c"), "-o", exe,
           "-L", lib_dir, "-lmm", "-L", cudart_dirs[0], "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + cudart_dirs[0]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe

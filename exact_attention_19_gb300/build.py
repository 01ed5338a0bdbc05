"""Build libfa_gb300.so in-tree with nvcc (sm_103a only).

Three translation units: fa_api.cu (the C-ABI front end with every forward,
split-KV merge and backward kernel instantiation), fa_probe.cu (the
exp2-throughput probe) and fa_selftest.cu (the bounded-wait self-test),
compiled in one nvcc call.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libfa_gb300.so")
SOURCES = [os.path.join(CSRC, f) for f in ("fa_api.cu", "fa_probe.cu", "fa_selftest.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("fa_ptx.cuh", "fa_fwd_kernel.cuh", "fa_fwd_persist.cuh", "fa_bwd_kernel.cuh")] + [
    os.path.join(INCLUDE, "fa.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")
    return path


def command(out: str = LIB_PATH, verbose_ptxas: bool = False) -> list[str]:
    cmd = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-o", out, *SOURCES, "-lcudart"]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in DEPS)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if force or needs_build():
        os.makedirs(LIB_DIR, exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        res = subprocess.run(command(tmp, verbose_ptxas), capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{res.stdout}\n{res.stderr}")
        if verbose_ptxas:
            sys.stderr.write(res.stderr)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB_PATH)

"""Builds the CUDA libraries in-tree for sm_103a with nvcc.

libgqa.so           -- the product library (csrc/gqa_api.cu and the kernels
                       it includes), C ABI declared in include/gqa.h
libgqa_selftest.so  -- single-CTA checks of the TMA / tcgen05 building
                       blocks, used only by the GPU test suite
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I" + INCLUDE, "-I" + CSRC]

LIBS = {
    "libgqa.so": ["gqa_api.cu"],
    "libgqa_selftest.so": ["selftest.cu"],
}


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list:
    out = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    return out


def lib_path(name: str = "libgqa.so") -> str:
    return os.path.join(PKG, name)


def build(force: bool = False, verbose: bool = False) -> list:
    """Compile every library whose sources changed; returns the built paths."""
    nvcc = nvcc_path()
    newest = max(os.path.getmtime(p) for p in _deps())
    built = []
    for name, srcs in LIBS.items():
        out = lib_path(name)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
            continue
        tmp = out + ".tmp%d" % os.getpid()
        cmd = [nvcc] + ARCH + FLAGS + ["-o", tmp] + [os.path.join(CSRC, s) for s in srcs]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        subprocess.check_call(cmd)
        os.replace(tmp, out)
        built.append(out)
    return built


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

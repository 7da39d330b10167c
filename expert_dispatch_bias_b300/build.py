"""Builds the shared libraries in-tree with nvcc for sm_103a.

  expert_dispatch_bias_b300/libmoe.so  - the MoE-layer library (C ABI in include/moe.h)
  synth/libsynth.so                    - the device side of the seeded input generator
  synth/libsynth_host.so               - its host side in C (gcc + OpenMP)

Run as ``python expert_dispatch_bias_b300/build.py [--force]`` (by path: importing the
package first would load the library that is about to be rebuilt).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared"]

TARGETS = [
    # (output, main source, dependencies that trigger a rebuild)
    ("expert_dispatch_bias_b300/libmoe.so", "expert_dispatch_bias_b300/csrc/moe_api.cu",
     ["expert_dispatch_bias_b300/csrc", "include/moe.h"]),
    ("synth/libsynth.so", "synth/csrc/synth.cu", ["synth/csrc"]),
]

# Host-side C (gcc, OpenMP): the fast host generator.
HOST_TARGETS = [
    ("synth/libsynth_host.so", "synth/csrc/synth_host.c", ["synth/csrc"]),
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")


def _mtime(path: str) -> float:
    p = os.path.join(ROOT, path)
    if os.path.isdir(p):
        return max((os.path.getmtime(os.path.join(p, f)) for f in os.listdir(p)), default=0.0)
    return os.path.getmtime(p)


def build(force: bool = False, verbose: bool = False) -> None:
    nvcc = _nvcc()
    for out, src, deps in TARGETS:
        out_p = os.path.join(ROOT, out)
        if not force and os.path.exists(out_p) and os.path.getmtime(out_p) >= max(_mtime(d) for d in deps + [src]):
            continue
        cmd = [nvcc, *FLAGS, *ARCH, "-I", os.path.join(ROOT, "include"), "-o", out_p + ".tmp",
               os.path.join(ROOT, src)]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(out_p + ".tmp", out_p)
    for out, src, deps in HOST_TARGETS:
        out_p = os.path.join(ROOT, out)
        if not force and os.path.exists(out_p) and os.path.getmtime(out_p) >= max(_mtime(d) for d in deps + [src]):
            continue
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-o", out_p + ".tmp",
               os.path.join(ROOT, src)]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(out_p + ".tmp", out_p)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

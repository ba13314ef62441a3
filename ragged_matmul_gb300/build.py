"""Compile the CUDA library (libgmm.so) in-tree for sm_103a with nvcc.

One translation unit, one -gencode, no cmake: this runs in seconds on both
the x86_64 build container and the aarch64 GPU hosts.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
INCLUDE_DIR = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG_DIR, "csrc")
SOURCES = [os.path.join(CSRC, "gmm.cu")]
LIB_PATH = os.path.join(PKG_DIR, "libgmm.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-shared", "-Xcompiler", "-fPIC"]


def _depends():
    deps = list(SOURCES) + [os.path.join(INCLUDE_DIR, f) for f in os.listdir(INCLUDE_DIR) if f.endswith(".h")]
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return deps


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def needs_build(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in _depends())


def build(force: bool = False, extra_flags=(), out: str | None = None, sources=None) -> str:
    """Build libgmm.so (only when a source is newer, unless force) and return its path."""
    out = out or LIB_PATH
    if not force and not needs_build(out):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *NVCC_FLAGS, *extra_flags, "-I", INCLUDE_DIR, "-o", tmp, *(sources or SOURCES)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out

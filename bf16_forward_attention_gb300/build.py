"""Builds the CUDA library in-tree: ``_lib/libattn_fwd.so`` for sm_103a.

    python -m bf16_forward_attention_gb300.build [--force] [--debug]

``--debug`` builds ``_lib/libattn_fwd_debug.so`` with -DATTN_DEBUG=1 instead: the
same kernels with bounds and protocol checks that report through the device
status word (see include/attn_fwd.h).

Two translation units (the kernels with their launcher, and the host-buffer
pipeline), one -gencode; the CUDA runtime is linked statically and the driver's
tensor-map encoder is looked up at run time, so the library loads (and
reports ATTN_ERR_NO_DEVICE) on a machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libattn_fwd.so")
LIB_PATH_DEBUG = os.path.join(LIB_DIR, "libattn_fwd_debug.so")
SOURCES = [os.path.join(CSRC, "attn_fwd.cu"), os.path.join(CSRC, "attn_host.cu")]
GENCODE = "arch=compute_103a,code=sm_103a"


def _deps():
    deps = list(SOURCES)
    for d in (CSRC, INCLUDE):
        deps += [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cuh", ".h", ".cu"))]
    return deps


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found (set CUDA_HOME or put nvcc on PATH)")


def lib_path(debug: bool = False) -> str:
    return LIB_PATH_DEBUG if debug else LIB_PATH


def up_to_date(debug: bool = False) -> bool:
    path = lib_path(debug)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (release, or the debug flavour) if any source is newer
    than it. Returns its path."""
    path = lib_path(debug)
    if not force and up_to_date(debug):
        return path
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-o", tmp] + SOURCES
    if debug:
        cmd.insert(1, "-DATTN_DEBUG=1")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))

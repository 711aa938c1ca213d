"""Builds the in-tree CUDA library ``libfp8mqa.so`` for sm_103a with nvcc.

Usage: ``python -m fp8_mqa_logits_02_gb300.nvcc_build`` (also called by the package's
``build()`` helper).  The outputs (``libfp8mqa.so`` and its bounds-checking variant
``libfp8mqa_debug.so``) land next to this file and are git-ignored.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, "fp8_mqa_logits.cu")]
LIB = os.path.join(HERE, "libfp8mqa.so")
# The same library built with FP8MQA_DEBUG_BOUNDS: every global access and TMA coordinate
# of the kernel is checked first, and a violation is recorded in the status word
# (fp8_mqa_logits_check_error then returns FP8MQA_ERR_BOUNDS) instead of being made.
DEBUG_LIB = os.path.join(HERE, "libfp8mqa_debug.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfp8mqa.so")
    return cand


def deps() -> list:
    """Every file the library is compiled from: all of csrc/, the public header and this
    script (a change to any of them triggers a rebuild)."""
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    return files + [os.path.join(ROOT, "include", "fp8_mqa_logits.h"), os.path.abspath(__file__)]


def up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in deps())


def _command(out: str, debug: bool, verbose: bool) -> list:
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-I", os.path.join(ROOT, "include"), "-o", out, *SOURCES]
    if debug:
        cmd.insert(1, "-DFP8MQA_DEBUG_BOUNDS")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Build the library (debug=False), its bounds-checking variant (debug=True), or both
    at once (debug=None, the default; returns the regular library's path).  Each is rebuilt
    only when a source is newer, unless `force`."""
    targets = [False, True] if debug is None else [bool(debug)]
    jobs = []
    for dbg in targets:
        lib = DEBUG_LIB if dbg else LIB
        if not force and up_to_date(lib):
            continue
        tmp = lib + f".tmp{os.getpid()}"
        proc = subprocess.Popen(_command(tmp, dbg, verbose), stdout=subprocess.PIPE,
                                stderr=subprocess.STDOUT, text=True)
        jobs.append((lib, tmp, proc))
    failed = []
    for lib, tmp, proc in jobs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            failed.append(f"nvcc failed for {os.path.basename(lib)}:\n{out}")
            continue
        if verbose:
            sys.stderr.write(out)
        os.replace(tmp, lib)
    if failed:
        raise RuntimeError("\n".join(failed))
    return DEBUG_LIB if debug else LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

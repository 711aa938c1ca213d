"""CPU oracle for the prefill FP8 MQA indexer logits -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (``fp8_mqa_logits_02_gb300``) never imports
it, and the two share no code.

The arithmetic lives in ``fp8_mqa_logits_oracle.c`` (plain C99, fp64, one pthread per
slice of rows); this module only compiles it with gcc and marshals numpy arrays.

Source of the definition: ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA
logits", section "Motivation":
``logits[m,n] = sum_h relu(Q[m,h,:].K[n,:]) * w[m,h] * kv_scale[n]`` for n in
``[ks[m], ke[m])`` and ``-inf`` elsewhere.

Parity pins (all in ``tests/test_oracle.py``): the e4m3 table against torch's own
``float8_e4m3fn`` conversion and hand-decoded codes, hand-computed fixtures under
``tests/golden/``, an exact int64 dot, the positive-input special case reduced to one
matrix product, and the invariants of the formula (linearity in w and kv_scale,
-inf outside the window, head permutation, row/column independence).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_mqa_logits_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: fp64 in source order)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load an oracle shared library from ``path`` (the tests also bind deliberately
    broken copies of the oracle to check that the pins catch them)."""
    lib = ctypes.CDLL(path)
    lib.oracle_e4m3_table.argtypes = [ctypes.c_void_p]
    lib.oracle_e4m3_table.restype = None
    lib.oracle_fp8_mqa_logits.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32]
    lib.oracle_fp8_mqa_logits.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(_LIB)
    return _lib


def source_path() -> str:
    return _SRC


def e4m3_table(lib=None) -> np.ndarray:
    """The oracle's 256-entry OCP E4M3 -> float64 decode table."""
    t = np.empty(256, dtype=np.float64)
    (lib or _load()).oracle_e4m3_table(t.ctypes.data)
    return t


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def fp8_mqa_logits(q, k, kv_scale, w, ks, ke, clean_logits: int, out=None, rows=None,
                   nthreads: int | None = None, lib=None) -> np.ndarray:
    """fp64 logits for host arrays.

    q: uint8 [M,H,D] (E4M3 bytes), k: uint8 [N,D], kv_scale: float32 [N], w: float32 [M,H],
    ks/ke: int32 [M].  Returns float64 [M,N] (or [len(rows),N] for the listed rows).
    With ``clean_logits=0`` entries outside the window keep the value they have in
    ``out`` (NaN when ``out`` is None).
    """
    q = np.ascontiguousarray(q, dtype=np.uint8)
    k = np.ascontiguousarray(k, dtype=np.uint8)
    kv_scale = np.ascontiguousarray(kv_scale, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    ks = np.ascontiguousarray(ks, dtype=np.int32)
    ke = np.ascontiguousarray(ke, dtype=np.int32)
    if q.ndim != 3 or k.ndim != 2:
        raise ValueError("q must be [M,H,D] and k [N,D]")
    M, H, D = q.shape
    N = k.shape[0]
    if k.shape[1] != D or w.shape != (M, H) or kv_scale.shape != (N,) \
            or ks.shape != (M,) or ke.shape != (M,):
        raise ValueError("inconsistent shapes")
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows.shape[0]
    else:
        nrows = M
    if out is None:
        out = np.full((nrows, N), np.nan, dtype=np.float64)
    else:
        if out.dtype != np.float64 or out.shape != (nrows, N) or not out.flags.c_contiguous:
            raise ValueError("out must be a C-contiguous float64 [rows, N] array")
    rc = (lib or _load()).oracle_fp8_mqa_logits(
        q.ctypes.data, k.ctypes.data, kv_scale.ctypes.data, w.ctypes.data,
        ks.ctypes.data, ke.ctypes.data, out.ctypes.data,
        M, N, H, D, 1 if clean_logits else 0,
        rows.ctypes.data if rows is not None else None, nrows,
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out

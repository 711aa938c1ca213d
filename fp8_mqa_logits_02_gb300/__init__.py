"""Python binding of the GB300 prefill FP8 MQA indexer-logits library (``libfp8mqa.so``).

Argument marshalling only: every step of the computation runs in the library's sm_103a
kernel.  The binding refuses to work without the compiled library (it raises; there is
no fallback).  The C entry points are declared in ``include/fp8_mqa_logits.h``.

    out[m, n] = kv_scale[n] * sum_h relu(Q[m,h,:] . K[n,:]) * w[m,h]  for n in [ks[m], ke[m])
    (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits", "Motivation")
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HEADS = 32
DIM = 128

STATUS = {
    0: "FP8MQA_OK",
    -1: "FP8MQA_ERR_INVALID_ARG",
    -2: "FP8MQA_ERR_UNSUPPORTED_SHAPE",
    -3: "FP8MQA_ERR_MISALIGNED",
    -4: "FP8MQA_ERR_ARCH",
    -5: "FP8MQA_ERR_LAUNCH",
    -6: "FP8MQA_ERR_TIMEOUT",
    -7: "FP8MQA_ERR_CUDA",
    -8: "FP8MQA_ERR_BOUNDS",
    -9: "FP8MQA_ERR_CAPACITY",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8mqa.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libfp8mqa_debug.so")
_lock = threading.Lock()
_libs = {}
_debug = False

# Every symbol the C header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64, _I32, _U64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
SIGNATURES = {
    "fp8_mqa_logits": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32,
                                      _I32, _P]),
    "fp8_mqa_logits_is_supported": (ctypes.c_int, [_I64, _I64, _I32, _I32, _I32]),
    "fp8_mqa_logits_default_split": (ctypes.c_int, [_I64, _I64, _I32]),
    "fp8_mqa_logits_check_error": (ctypes.c_int, [_P]),
    "fp8_mqa_logits_set_wait_limit_ns": (ctypes.c_uint64, [_U64]),
    "fp8_mqa_logits_host_workspace_bytes": (ctypes.c_uint64, [_I64, _I64, _I32, _I32]),
    "fp8_mqa_logits_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32,
                                           _I32, _I32, _P, _U64, _P]),
    "fp8_mqa_logits_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "fp8_mqa_logits_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32,
                                              _I32, _I32, _I32, _P]),
    "fp8_mqa_topk": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _P]),
    "fp8_mqa_topk_windowed": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    "fp8_mqa_topk_ex": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _I32, _I32, _P, _P, _P]),
}

TOPK_MAX_K = 2048


class Fp8MqaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Compile ``libfp8mqa.so`` (and, by default, its bounds-checking variant) in-tree with
    nvcc for sm_103a."""
    from . import nvcc_build
    return nvcc_build.build(force=force, verbose=verbose, debug=debug)


def use_debug_library(on: bool) -> None:
    """Route every later call of this module through ``libfp8mqa_debug.so``, the build whose
    kernel checks each global access first and records a violation (``check_error`` then
    returns FP8MQA_ERR_BOUNDS) instead of making it; ``False`` switches back."""
    global _debug
    _debug = bool(on)


def lib(debug: bool | None = None):
    """The loaded library (the bounds-checking build when selected); raises if it has not
    been built."""
    dbg = _debug if debug is None else bool(debug)
    path = DEBUG_LIB_PATH if dbg else LIB_PATH
    with _lock:
        if path not in _libs:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -m fp8_mqa_logits_02_gb300.nvcc_build` (there is no CPU fallback)")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _libs[path] = handle
    return _libs[path]


def strerror(status: int) -> str:
    try:
        return lib().fp8_mqa_logits_strerror(int(status)).decode()
    except Exception:  # library missing: fall back to the table above
        return STATUS.get(int(status), f"unknown status {status}")


def is_supported(M: int, N: int, H: int = HEADS, D: int = DIM, device: int = -1) -> bool:
    """Whether (M, N, H, D) is inside the contract; with ``device >= 0`` also whether that
    CUDA device is a compute-capability 10.3 GPU."""
    return bool(lib().fp8_mqa_logits_is_supported(M, N, H, D, int(device)))


def set_wait_limit_ns(ns: int) -> int:
    """Limit of one on-device pipeline wait for later launches (0: the 1 s default).
    Returns the previous limit.  For diagnostics and tests of the failure path."""
    return int(lib().fp8_mqa_logits_set_wait_limit_ns(int(ns)))


def default_split(M: int, N: int, num_sms: int) -> int:
    return int(lib().fp8_mqa_logits_default_split(M, N, num_sms))


# The current stream's raw handle in one call: torch.cuda.current_stream() builds a Stream
# object each time, which costs several microseconds per launch on the small shapes.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_entries = {}


def _stream_ptr(stream, device: torch.device | None = None) -> int:
    """The cudaStream_t of ``stream``; when it is None, of the current stream of ``device``
    (default: the current device)."""
    if stream is None:
        idx = device.index if device is not None and device.index is not None \
            else torch.cuda.current_device()
        if _raw_stream is not None:
            return int(_raw_stream(idx))
        stream = torch.cuda.current_stream(idx)
    return int(stream.cuda_stream)


def _entry(name: str):
    """The library's entry point ``name``, resolved once per library build."""
    key = (_debug, name)
    fn = _entries.get(key)
    if fn is None:
        fn = getattr(lib(), name)
        _entries[key] = fn
    return fn


def _on(dev: torch.device, fn, *args):
    """``fn(*args)`` with ``dev`` the current CUDA device; the device is switched only when
    it is not current already (the switch costs more than the check)."""
    if torch.cuda.current_device() == dev.index:
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _check(t: torch.Tensor, name: str, dtypes, ndim: int, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


FP8 = (torch.float8_e4m3fn,)


def fp8_mqa_logits(q: torch.Tensor, k: torch.Tensor, kv_scale: torch.Tensor, w: torch.Tensor,
                   ks: torch.Tensor, ke: torch.Tensor, out: torch.Tensor | None = None,
                   clean_logits: bool = True, split_n: int = 0, stream=None) -> torch.Tensor:
    """Logits of every query row against its key window, on the GPU.

    q: float8_e4m3fn [M, 32, 128]; k: float8_e4m3fn [N, 128]; kv_scale: float32 [N];
    w: float32 [M, 32]; ks, ke: int32 [M] (row m attends keys ks[m] <= n < ke[m]).
    out: optional float32 [M, N] to write into (needed to keep caller-managed values
    with ``clean_logits=False``).  Returns ``out``.  Asynchronous on ``stream``
    (default: the current stream).
    """
    _check(q, "q", FP8, 3)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor (the library has no CPU path)")
    _check(k, "k", FP8, 2, dev)
    _check(kv_scale, "kv_scale", (torch.float32,), 1, dev)
    _check(w, "w", (torch.float32,), 2, dev)
    _check(ks, "ks", (torch.int32,), 1, dev)
    _check(ke, "ke", (torch.int32,), 1, dev)
    M, H, D = q.shape
    N = k.shape[0]
    if k.shape[1] != D or tuple(w.shape) != (M, H) or kv_scale.shape[0] != N \
            or ks.shape[0] != M or ke.shape[0] != M:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    else:
        _check(out, "out", (torch.float32,), 2, dev)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M}, {N}]")
    rc = _on(dev, _entry("fp8_mqa_logits"), q.data_ptr(), k.data_ptr(), kv_scale.data_ptr(),
             w.data_ptr(), ks.data_ptr(), ke.data_ptr(), out.data_ptr(), M, N, H, D,
             1 if clean_logits else 0, int(split_n), _stream_ptr(stream, dev))
    if rc != 0:
        raise Fp8MqaError(rc, "fp8_mqa_logits")
    return out


TOPK_UNSORTED = 1  # fp8_mqa_topk_ex flag


def topk(logits: torch.Tensor, k: int, with_values: bool = True, stream=None,
         ks: torch.Tensor | None = None, ke: torch.Tensor | None = None, sorted: bool = True):
    """Per-row top-k of a float32 [M, N] CUDA tensor (rows may be strided, elements not).

    Returns (indices int32 [M, k], values float32 [M, k] or None): the k largest finite
    entries of each row, by value descending and equal values by index ascending; slots past
    a row's finite entries hold -1 / -inf.  With ``ks``/``ke`` (int32 [M] on the same device,
    the windows the logits were made with) only entries in [ks[m], ke[m]) count and nothing
    outside them is read, so the logits may come from ``clean_logits=False``.  With
    ``sorted=False`` each row holds the same entries in an unspecified order (the padding still
    last), which skips the sort for consumers that take the indices as a set.  Asynchronous on
    ``stream``.
    """
    _check_strided_rows(logits, "logits")
    if not 1 <= int(k) <= TOPK_MAX_K:
        raise ValueError(f"k must be in [1, {TOPK_MAX_K}]")
    M, N = logits.shape
    dev = logits.device
    if (ks is None) != (ke is None):
        raise ValueError("ks and ke go together")
    for name, t in (("ks", ks), ("ke", ke)):
        if t is not None and (t.dtype != torch.int32 or t.shape != (M,) or t.device != dev
                              or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 [M] tensor on {dev}")
    idx = torch.empty((M, int(k)), dtype=torch.int32, device=dev)
    val = torch.empty((M, int(k)), dtype=torch.float32, device=dev) if with_values else None
    rc = _on(dev, _entry("fp8_mqa_topk_ex"),
             logits.data_ptr(), M, N, logits.stride(0),
             ks.data_ptr() if ks is not None else None, ke.data_ptr() if ke is not None else None,
             int(k), 0 if sorted else TOPK_UNSORTED, idx.data_ptr(),
             val.data_ptr() if val is not None else None, _stream_ptr(stream, dev))
    if rc != 0:
        raise Fp8MqaError(rc, "fp8_mqa_topk_ex")
    return idx, val


def _check_strided_rows(t: torch.Tensor, name: str):
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != torch.float32 or t.dim() != 2:
        raise ValueError(f"{name} must be float32 [M, N]")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")


def check_error(stream=None) -> int:
    """Synchronize ``stream`` and return (and clear) the device status: 0 or a status code."""
    return int(lib().fp8_mqa_logits_check_error(_stream_ptr(stream)))


def host_workspace_bytes(M: int, N: int, H: int = HEADS, D: int = DIM) -> int:
    return int(lib().fp8_mqa_logits_host_workspace_bytes(M, N, H, D))


def fp8_mqa_logits_host(q, k, kv_scale, w, ks, ke, out, workspace: torch.Tensor,
                        clean_logits: bool = True, split_n: int = 0, stream=None) -> None:
    """Same operation on HOST tensors (pinned for asynchronous copies).

    q/k: CPU uint8 or float8_e4m3fn; kv_scale, w: CPU float32; ks, ke: CPU int32;
    out: CPU float32 [M, N], filled when ``stream`` is synchronized.  ``workspace`` is a
    CUDA uint8 tensor of at least ``host_workspace_bytes(M, N)`` bytes.
    """
    for t, name in ((q, "q"), (k, "k"), (kv_scale, "kv_scale"), (w, "w"), (ks, "ks"),
                    (ke, "ke"), (out, "out")):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    M, H, D = q.shape
    N = k.shape[0]
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    rc = _on(workspace.device, _entry("fp8_mqa_logits_host"),
             q.data_ptr(), k.data_ptr(), kv_scale.data_ptr(), w.data_ptr(), ks.data_ptr(),
             ke.data_ptr(), out.data_ptr(), M, N, H, D, 1 if clean_logits else 0, int(split_n),
             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
             _stream_ptr(stream, workspace.device))
    if rc != 0:
        raise Fp8MqaError(rc, "fp8_mqa_logits_host")

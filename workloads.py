"""Seeded synthetic inputs for the prefill FP8 MQA indexer logits.

This module holds no arithmetic of the method: it only draws inputs.  Both the CUDA
path's tests/bench and the CPU oracle's tests take their inputs from here.

Distributions (the same for every workload): Q and K are N(0,1) draws clipped to
+-448 and rounded to OCP E4M3 by torch's ``float8_e4m3fn`` conversion; w is
N(0,1)/sqrt(H*D) in fp32; kv_scale is U[0.5, 2] in fp32.  One CPU ``torch.Generator``
seeded with the workload's seed draws Q, K, w and kv_scale in that order.

Window families.  The benchmark workloads follow the kernel-time table of
ROCm/aiter PR #7183 ("Kernel time on the GLM-5.3-Flash table shapes"): causal chunks
whose query rows are the last M positions of an N-key context, a multi-request chunk of
four requests, and the table's "16384 x 32000 (kpool 4)" row.  The other families
("cp", "misaligned", "empty", "past_end") are readings of the op-test window modes named
in the same page's "Test plan"; the page does not define them, so each is spelled out
below.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

H_DEFAULT = 32
D_DEFAULT = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    windows: str  # window family, see ``windows()``
    seed: int
    H: int = H_DEFAULT
    D: int = D_DEFAULT
    requests: int = 1  # multi_req only


# The benchmark/parity workloads (seed = position in this list).
WORKLOADS = {
    "tiny_causal_64x256": Workload("tiny_causal_64x256", 64, 256, "causal", 0),
    "causal_8192x8192": Workload("causal_8192x8192", 8192, 8192, "causal", 1),
    "chunk_causal_4096x32768": Workload("chunk_causal_4096x32768", 4096, 32768, "causal", 2),
    "long_causal_1024x131072": Workload("long_causal_1024x131072", 1024, 131072, "causal", 3),
    "multi_req_4096x32768": Workload("multi_req_4096x32768", 4096, 32768, "multi_req", 4,
                                     requests=4),
    # The same table's "16384 x 32000 (kpool 4)" row, read as one causal chunk over a single
    # contiguous K of 32000 keys (the page does not define "kpool"), and the chunk shape
    # under the context-parallel window family of the page's op test.
    "kpool_causal_16384x32000": Workload("kpool_causal_16384x32000", 16384, 32000, "causal", 5),
    "cp_4096x32768": Workload("cp_4096x32768", 4096, 32768, "cp", 6),
    # The table's remaining rows: the causal 2048 x 65536 chunk and the multi-request
    # block (4 requests each) at 2048 x 65536, 1024 x 131072 and 8192 x 8192.
    "chunk_causal_2048x65536": Workload("chunk_causal_2048x65536", 2048, 65536, "causal", 7),
    "multi_req_2048x65536": Workload("multi_req_2048x65536", 2048, 65536, "multi_req", 8,
                                     requests=4),
    "multi_req_1024x131072": Workload("multi_req_1024x131072", 1024, 131072, "multi_req", 9,
                                      requests=4),
    "multi_req_8192x8192": Workload("multi_req_8192x8192", 8192, 8192, "multi_req", 10,
                                    requests=4),
    # The small shape the page's "Known limitations" names (M <= 128 and 1024 x 1024).
    "small_causal_1024x1024": Workload("small_causal_1024x1024", 1024, 1024, "causal", 11),
    "small_causal_128x4096": Workload("small_causal_128x4096", 128, 4096, "causal", 12),
}

WINDOW_FAMILIES = ("causal", "cp", "misaligned", "empty", "past_end", "multi_req")


def windows(family: str, M: int, N: int, requests: int = 4):
    """Per-row [ks, ke) bounds (int32) for a window family.

    causal     rows are the last M positions of an N-key context: ks=0, ke=N-M+m+1.
    multi_req  ``requests`` requests, each owning a contiguous N/requests key segment
               and M/requests query rows that are the last rows of that segment:
               for request r, row i: ks = r*S, ke = r*S + (S - R) + i + 1 with
               S = N/requests, R = M/requests.
    cp         context-parallel split: the first half of the rows is causal at a
               shifted, tile-unaligned offset, the second half is the tail chunk.
    misaligned windows that start and end in the middle of key tiles.
    empty      causal, but every third row is empty (ks == ke) and every seventh has
               ks > ke.
    past_end   ke beyond N for all rows, and some rows with ks >= N.
    """
    m = np.arange(M, dtype=np.int64)
    if family == "causal":
        ks = np.zeros(M, np.int64)
        ke = (N - M) + m + 1
    elif family == "multi_req":
        if M % requests or N % requests:
            raise ValueError("multi_req needs M and N divisible by the request count")
        S, R = N // requests, M // requests
        r, i = m // R, m % R
        ks = r * S
        ke = r * S + (S - R) + i + 1
    elif family == "cp":
        half = M // 2
        off0 = max(0, (N - M) // 3 + 5)
        ks = np.zeros(M, np.int64)
        ke = np.where(m < half, off0 + m + 1, (N - (M - half)) + (m - half) + 1)
    elif family == "misaligned":
        span = max(1, N // 3)
        ks = (37 * m + 5) % span
        ke = ks + 1 + (101 * m + 11) % max(1, (2 * N) // 3)
    elif family == "empty":
        ks = np.zeros(M, np.int64)
        ke = (N - M) + m + 1
        ks = np.where(m % 3 == 1, ke, ks)
        ks = np.where(m % 7 == 5, ke + 3, ks)
    elif family == "past_end":
        ks = (m * 13) % max(1, N)
        ke = N + 17 + m
        ks = np.where(m % 5 == 2, N + m % 3, ks)
    else:
        raise ValueError(f"unknown window family {family!r}")
    return ks.astype(np.int32), ke.astype(np.int32)


def describe(wl: Workload) -> str:
    """One-line statement of a workload's windows, for reports."""
    M, N = wl.M, wl.N
    if wl.windows == "causal":
        return f"causal: ks=0, ke={N - M}+m+1"
    if wl.windows == "multi_req":
        S, R = N // wl.requests, M // wl.requests
        return (f"multi_req: {wl.requests} requests; request r=m//{R}, row i=m%{R}: "
                f"ks={S}r, ke={S}r+{S - R}+i+1")
    if wl.windows == "cp":
        half = M // 2
        off0 = max(0, (N - M) // 3 + 5)
        return (f"cp: ks=0; rows m<{half}: ke={off0}+m+1, rows m>={half}: "
                f"ke={N - (M - half)}+(m-{half})+1")
    return wl.windows


def draw(M: int, N: int, seed: int, H: int = H_DEFAULT, D: int = D_DEFAULT):
    """Seeded Q, K, w, kv_scale as numpy arrays (q/k: uint8 E4M3 bytes)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((M, H, D), generator=g).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    k = torch.randn((N, D), generator=g).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    w = torch.randn((M, H), generator=g) / math.sqrt(H * D)
    kv = torch.rand((N,), generator=g) * 1.5 + 0.5
    return (q.view(torch.uint8).numpy(), k.view(torch.uint8).numpy(),
            kv.to(torch.float32).numpy(), w.to(torch.float32).numpy())


def make(wl: Workload, family: str | None = None):
    """All host inputs for a workload: dict of numpy arrays plus sizes."""
    q, k, kv, w = draw(wl.M, wl.N, wl.seed, wl.H, wl.D)
    ks, ke = windows(family or wl.windows, wl.M, wl.N, wl.requests)
    return {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke,
            "M": wl.M, "N": wl.N, "H": wl.H, "D": wl.D}


def valid_pairs(ks: np.ndarray, ke: np.ndarray, N: int) -> int:
    """Number of in-window (m, n) pairs: sum over rows of |[ks,ke) clamped to [0,N)|."""
    lo = np.clip(ks.astype(np.int64), 0, N)
    hi = np.clip(ke.astype(np.int64), 0, N)
    return int(np.maximum(hi - lo, 0).sum())


def draw_logits(M: int, N: int, seed: int, ties: bool = True, neg_inf_frac: float = 0.25,
                empty_rows: int = 1):
    """Seeded float32 [M, N] logit-like rows for the top-k selection: N(0.5, 0.5) values, a
    share of exact ties (values rounded to 1/8 on every 5th key), -inf on a random share of
    keys, the first ``empty_rows`` rows all -inf, and a row of equal values."""
    rng = np.random.default_rng(seed)
    x = (0.5 + 0.5 * rng.standard_normal((M, N))).astype(np.float32)
    if ties:
        x[:, ::5] = np.round(x[:, ::5] * 8.0) / 8.0
    x[rng.random((M, N)) < neg_inf_frac] = -np.inf
    x[:min(M, empty_rows)] = -np.inf
    if M > empty_rows + 1:
        x[empty_rows + 1] = 0.75
    return x

"""CPU oracle for the per-row top-k selection over indexer logits -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this module; the product path never does, and the two share no code.

What it computes.  The consumer of the indexer logits keeps, for every query row, the keys
with the k largest logits: ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA
logits", section "Test plan" (the end-to-end check compares top-512 selections), and
ROCm/aiter PR #6159 "[Triton/Gluon] GFX950 sparse mla optimizations", section "Technical
Details" (sparse MLA layers with top-k 512).  The pages fix no tie rule and no padding, so
this reading is taken:

  - only finite entries are eligible; -inf (a key outside the row's window) never is;
  - the selection is ordered by value, descending; equal values by index, ascending
    (-0.0 and +0.0 are equal values);
  - when a row has fewer than k finite entries, the remaining slots hold index -1 and
    value -inf.

Under this reading the result is unique, so it is compared exactly.
"""
from __future__ import annotations

import numpy as np


def topk_rows(logits: np.ndarray, k: int):
    """Top-k of every row of ``logits`` (float32 [M, N]).

    Returns (indices int32 [M, k], values float32 [M, k]).  Plain per-row selection:
    gather the finite entries, order them by (value descending, index ascending) with a
    two-key lexicographic sort, keep the first k.
    """
    logits = np.asarray(logits, dtype=np.float32)
    if logits.ndim != 2:
        raise ValueError("logits must be 2-D")
    if k < 1:
        raise ValueError("k must be positive")
    M, _ = logits.shape
    idx = np.full((M, k), -1, dtype=np.int32)
    val = np.full((M, k), -np.inf, dtype=np.float32)
    for m in range(M):
        row = logits[m]
        cand = np.nonzero(np.isfinite(row))[0]
        v = row[cand].astype(np.float64) + 0.0  # -0.0 + 0.0 == +0.0: equal zeros compare equal
        # np.lexsort sorts by the last key first: value descending, then index ascending
        order = np.lexsort((cand, -v))
        take = cand[order[:k]]
        idx[m, :len(take)] = take
        val[m, :len(take)] = row[take]
    return idx, val

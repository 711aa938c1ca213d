"""Pins for the top-k oracle (no GPU): hand-worked cases, a special case that reduces to a
stable library sort, and the invariants that define the selection."""
import json
import math
import os

import numpy as np
import pytest

from oracle.topk import topk_rows

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "topk_cases.json")


def _f(x):
    return float(x) if not isinstance(x, str) else float(x.replace("inf", "inf"))


def test_hand_cases():
    for c in json.load(open(GOLDEN))["cases"]:
        row = np.array([[_f(x) for x in c["row"]]], dtype=np.float32)
        idx, val = topk_rows(row, c["k"])
        assert idx[0].tolist() == c["indices"], c["name"]
        want = np.array([_f(x) for x in c["values"]], dtype=np.float32)
        assert np.array_equal(val[0].view(np.uint32), want.view(np.uint32)), c["name"]


def _rows(seed, M=40, N=300):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N)).astype(np.float32)
    x[:, ::7] = np.round(x[:, ::7])             # plenty of exact ties
    mask = rng.random((M, N)) < 0.3
    x[mask] = -np.inf                          # keys outside the window
    x[3] = -np.inf                             # an empty window
    x[5, :] = 1.0                              # a row of equal values
    return x


@pytest.mark.parametrize("k", [1, 7, 64, 300, 512])
def test_selection_invariants(k):
    x = _rows(k)
    idx, val = topk_rows(x, k)
    for m in range(x.shape[0]):
        row = x[m]
        fin = np.isfinite(row)
        n_sel = min(k, int(fin.sum()))
        sel = idx[m, :n_sel]
        assert (idx[m, n_sel:] == -1).all() and np.isneginf(val[m, n_sel:]).all()
        assert len(set(sel.tolist())) == n_sel and fin[sel].all()
        assert np.array_equal(val[m, :n_sel], row[sel])
        # ordered by value descending, equal values by index ascending
        for a, b in zip(sel[:-1], sel[1:]):
            assert row[a] > row[b] or (row[a] == row[b] and a < b)
        if n_sel and n_sel < fin.sum():
            rest = np.setdiff1d(np.nonzero(fin)[0], sel)
            kth = row[sel[-1]]
            assert (row[rest] <= kth).all()
            # among entries equal to the k-th value, the selected ones have the lower indices
            ties_out = rest[row[rest] == kth]
            if len(ties_out):
                assert sel[row[sel] == kth].max() < ties_out.min()


def test_k_covering_all_entries_is_a_stable_descending_sort():
    # with k >= the number of finite entries, the selection is every finite entry in the
    # order of a stable sort on the negated values
    x = _rows(99, M=12, N=50)
    idx, _ = topk_rows(x, 64)
    for m in range(x.shape[0]):
        row = x[m]
        fin = np.nonzero(np.isfinite(row))[0]
        order = fin[np.argsort(-(row[fin].astype(np.float64) + 0.0), kind="stable")]
        assert idx[m, :len(order)].tolist() == order.tolist()
        assert (idx[m, len(order):] == -1).all()


def test_planted_mistakes_are_caught():
    # each broken variant of the rule must disagree with a hand case
    cases = json.load(open(GOLDEN))["cases"]

    def check(fn):
        for c in cases:
            row = np.array([[_f(x) for x in c["row"]]], dtype=np.float32)
            if fn(row, c["k"])[0].tolist() != [c["indices"]]:
                return False
        return True

    def ties_by_high_index(x, k):
        i, v = topk_rows(x[:, ::-1], k)
        return np.where(i >= 0, x.shape[1] - 1 - i, -1), v

    def ascending(x, k):
        return topk_rows(-x, k)

    def neg_inf_eligible(x, k):
        y = np.where(np.isneginf(x), np.float32(-3.4e38), x)
        return topk_rows(y, k)

    assert check(topk_rows)
    for bad in (ties_by_high_index, ascending, neg_inf_eligible):
        assert not check(bad), bad.__name__

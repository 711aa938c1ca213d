"""GPU parity of the per-row top-k (fp8_mqa_topk) against the CPU oracle: indices exact,
values bit-exact (the selection is unique under the library's tie rule)."""
import numpy as np
import pytest
import torch

import fp8_mqa_logits_02_gb300 as fm
import workloads
from oracle.topk import topk_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.build()
    fm.lib()


def _check(x: np.ndarray, k: int, gpu_rows=None, what=""):
    t = torch.from_numpy(x).cuda() if gpu_rows is None else gpu_rows
    idx, val = fm.topk(t, k)
    torch.cuda.synchronize()
    ri, rv = topk_rows(x, k)
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    bad = np.nonzero((gi != ri).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: {len(bad)} rows differ, first {bad[0]}: " \
                          f"gpu {gi[bad[0]][:8]} oracle {ri[bad[0]][:8]}"
    assert np.array_equal(gv.view(np.uint32), rv.view(np.uint32)), what


@pytest.mark.parametrize("M,N,k", [(1, 1, 1), (3, 5, 8), (64, 300, 1), (64, 300, 7),
                                   (40, 1000, 512), (33, 4097, 512), (16, 5000, 2048),
                                   (8, 1500, 2048), (200, 2500, 64),
                                   # many rows: several row groups per CTA, of one, two
                                   # and four warps, with rows left over for some groups
                                   (1000, 2000, 100), (1111, 4100, 256), (700, 9000, 512),
                                   (300, 20000, 1024)])
def test_random_rows(M, N, k):
    _check(workloads.draw_logits(M, N, seed=M * 7 + k), k, what=f"{M}x{N} k={k}")


def test_ties_straddle_the_cut():
    x = np.full((6, 3000), 0.5, dtype=np.float32)
    x[0, ::3] = 2.0                       # 1000 larger entries, then the cut inside the ties
    x[1, 100:120] = 3.0
    x[2, :] = np.float32(-0.0)
    x[2, 1::2] = 0.0                      # alternating signed zeros: all equal values
    x[3, 2999] = 7.0                      # the largest entry last
    x[4, ::7] = -np.inf
    x[5, :] = np.float32(1e-45)           # subnormal ties
    for k in (1, 5, 999, 1000, 1001, 2048):
        _check(x, k, what=f"ties k={k}")


def test_special_values():
    x = np.array([[3.0e38, -3.0e38, 1e-30, -1e-30, 1e-45, -1e-45, 0.0, -0.0, -np.inf, 1.0]],
                 dtype=np.float32)
    for k in (1, 3, 9, 10, 12):
        _check(x, k, what=f"special k={k}")


def test_empty_and_short_rows():
    x = workloads.draw_logits(10, 50, seed=3, neg_inf_frac=0.9, empty_rows=3)
    for k in (1, 20, 64):
        _check(x, k, what=f"short k={k}")
    idx, val = fm.topk(torch.empty((4, 0), dtype=torch.float32, device="cuda"), 3)
    assert (idx.cpu() == -1).all() and torch.isneginf(val.cpu()).all()


def test_strided_rows():
    wide = workloads.draw_logits(50, 1200, seed=5)
    t = torch.from_numpy(wide).cuda()[:, 100:1100]   # rows 1200 floats apart
    _check(wide[:, 100:1100].copy(), 300, gpu_rows=t, what="strided")


def test_long_rows():
    x = workloads.draw_logits(20, 131072, seed=9)
    for k in (512, 2048):
        _check(x, k, what=f"long k={k}")


def test_cut_resolves_ties_across_index_65536_in_long_rows():
    # Rows of 131072 keys where the k-th largest value is a tie whose first winners lie on
    # both sides of index 65536: the cut's index passes must cover the index's third byte.
    # The planted values sit outside the sampled sectors (element e is sampled when
    # e % 64 < 8), so the threshold comes from the background and the kept entries fit the
    # buffer: the sampled path's cut is the one under test.
    N = 131072
    rng = np.random.default_rng(17)
    x = (-rng.random((3, N))).astype(np.float32)          # background in (-1, 0]
    pos = np.nonzero(np.arange(N) % 64 >= 8)[0]
    for r in range(3):
        top = rng.choice(pos, 300, replace=False)
        rest = np.setdiff1d(pos, top)
        below = rest[(rest >= 60000) & (rest < 65536)]
        above = rest[rest >= 65536]
        x[r, top] = 5.0
        x[r, rng.choice(below, 100, replace=False)] = 4.0   # 1000 ties at the k-th value,
        x[r, rng.choice(above, 900, replace=False)] = 4.0   # 100 of them below 65536
    for k in (512, 1024, 2048):
        _check(x, k, what=f"ties across 65536 k={k}")


def test_indexer_pipeline_top512_matches_the_oracle_pipeline():
    # logits from the GPU kernel, then top-512 on the GPU, against top-512 of the fp64
    # oracle's logits (rounded to fp32) on sampled rows.  The logits agree only within the
    # parity tolerance, so near-ties at the cut may order differently; the selections must
    # be identical on nearly every row and overlap almost fully on the rest.
    from gpu_helpers import run_oracle, to_device
    wl = workloads.WORKLOADS["chunk_causal_4096x32768"]
    inp = workloads.make(wl)
    dev = to_device(inp)
    out = fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"])
    rows = np.sort(np.random.default_rng(1).choice(inp["M"], size=48, replace=False))
    gi, _ = fm.topk(out[torch.from_numpy(rows).cuda()].contiguous(), 512)
    ref = run_oracle(inp, clean=True, rows=rows).astype(np.float32)
    ri, _ = topk_rows(ref, 512)
    gi = gi.cpu().numpy()
    same = sum(set(a.tolist()) == set(b.tolist()) for a, b in zip(gi, ri))
    overlap = min(len(set(a.tolist()) & set(b.tolist())) for a, b in zip(gi, ri))
    assert same >= 0.9 * len(rows) and overlap >= 500, (same, overlap)


@pytest.mark.parametrize("N", [3000, 5000, 20000, 40000, 70000])
def test_crowded_threshold_bin_takes_the_multi_pass_path(N):
    # More entries than the threshold-bin buffer holds share the top 11 key bits of the k-th
    # largest, so the select resolves the remaining bits with further passes over the row.
    # The buffers hold 2048 entries for rows of up to 65536 keys at k <= 512 (two rows per
    # CTA), 4096 for rows of up to 32768 keys at k > 512, and 8192 for the others (one row per
    # CTA).  So N = 3000 reaches the multi-pass path at k <= 512 only, N = 5000 and 20000 at
    # every k, N = 40000 in the two-row kernel at k <= 512 and the one-row kernel beyond, and
    # N = 70000 in the one-row kernel at every k.
    x = np.empty((5, N), dtype=np.float32)
    x[0] = 1.0                                            # all equal: ties in index order
    x[1] = 1.0 + np.arange(N, dtype=np.float32) * 2.0 ** -23   # distinct, one top bin
    x[2] = x[1][::-1]
    x[3] = 1.0
    x[3, 7::13] = 1.0 + 2.0 ** -20                        # a few slightly larger ones first
    x[4] = 1.0 + (np.arange(N) % 97).astype(np.float32) * 2.0 ** -23   # many tie groups
    for k in (1, 5, 100, 1537, 2048):
        _check(x, k, what=f"crowded k={k}")


@pytest.mark.parametrize("k", [1, 512, 1000, 1024, 1025, 2048])
def test_full_8192_key_rows_causal_tails(k):
    # rows of exactly 8192 keys (the staged-row path's largest at k <= 1024), each with a window of
    # its own length and -inf after it, as the causal logits have
    M, N = 300, 8192
    x = workloads.draw_logits(M, N, seed=k + 11, neg_inf_frac=0.0, empty_rows=1)
    for m in range(M):
        x[m, (37 * m * m + 5) % N + 1:] = -np.inf
    _check(x, k, what=f"causal tails k={k}")


@pytest.mark.parametrize("k", [1, 300, 512, 1024, 2048])
def test_full_8192_key_rows_with_heavy_ties(k):
    N = 8192
    x = np.full((5, N), 0.25, dtype=np.float32)
    x[1, ::2] = 0.5                                       # 4096 equal winners above the cut
    x[2, 4000:] = np.float32(-0.0)
    x[2, 6000:] = 0.0
    x[3] = np.float32(1.0) + np.float32(2.0 ** -23) * (np.arange(N) % 3)   # three tie groups
    x[4, ::5] = -np.inf
    x[4, 3::7] = 3.0e38
    _check(x, k, what=f"heavy ties k={k}")


def _sampled_positions(N):
    # For rows of up to 8192 keys (k <= 1024) the kernel estimates its threshold from every
    # eighth element.
    e = np.arange(N)
    return e % 8 == 0


@pytest.mark.parametrize("k", [1, 64, 512, 1024, 2048])
def test_threshold_estimate_misses_take_the_full_row_path(k):
    N = 8192
    rng = np.random.default_rng(k)
    s = _sampled_positions(N)
    x = rng.standard_normal((8, N)).astype(np.float32)
    x[0, s] = 4.0 + rng.random(s.sum()).astype(np.float32)    # the estimate sees only the top
    x[1] = 1.5
    x[1, s] = 1.0                                              # everything unsampled is larger
    x[2, rng.random(N) < 0.3] = np.inf                         # +inf is not eligible
    x[3, s] = np.inf
    x[4, ~s] = np.inf
    x[5, rng.random(N) < 0.5] = np.nan
    x[6, s] = -np.inf                                          # the estimate sees nothing
    x[7, :] = -np.inf
    x[7, ~s & (rng.random(N) < 0.2)] = 1.0                     # ties, none of them sampled
    _check(x, k, what=f"estimate misses k={k}")


def test_unaligned_rows_of_the_staged_row_path():
    wide = workloads.draw_logits(40, 8400, seed=21)
    for off, n in ((101, 8192), (3, 8001), (2, 4097)):
        t = torch.from_numpy(wide).cuda()[:, off:off + n]       # rows start off 16 bytes
        for k in (512, 2048):
            _check(wide[:, off:off + n].copy(), k, gpu_rows=t, what=f"unaligned {off} k={k}")


@pytest.mark.parametrize("N", [8193, 32768, 32769, 65536, 65537])
@pytest.mark.parametrize("k", [512, 2048])
def test_row_lengths_at_the_dispatch_boundaries(N, k):
    # each side of every switch between kernels and sample resolutions: at k <= 512 two rows
    # per CTA up to 65536 keys (an 11-bit sample up to 32768, 12-bit beyond), then one row
    # per CTA; at k > 512 two rows per CTA up to 32768 keys (a 12-bit sample beyond 8192 keys
    # when k > 1024), then one row per CTA
    x = workloads.draw_logits(4, N, seed=N % 1000 + k, neg_inf_frac=0.1)
    _check(x, k, what=f"{N} keys k={k}")
    _check_unsorted(x, k, what=f"unsorted {N} keys k={k}")


def test_unaligned_rows_of_the_long_row_kernels():
    # rows that start off 16 bytes take the candidate pass's one-element-per-thread loop: rows
    # of 20000 keys in the two-row kernels, of 70001 keys in the one-row kernel
    wide = workloads.draw_logits(6, 70010, seed=23, neg_inf_frac=0.05)
    for off, n in ((1, 20000), (3, 70001)):
        t = torch.from_numpy(wide).cuda()[:, off:off + n]
        for k in (64, 512, 2048):
            _check(wide[:, off:off + n].copy(), k, gpu_rows=t, what=f"unaligned {off}+{n} k={k}")


def _check_unsorted(x, k, ks=None, ke=None, what=""):
    # the unsorted result: per row the oracle's entries as a set, each index with its exact
    # value, then the padding
    M, N = x.shape
    ref = x
    if ks is not None:
        ref = np.full_like(x, -np.inf)
        for m in range(M):
            lo, hi = max(int(ks[m]), 0), min(int(ke[m]), N)
            if lo < hi:
                ref[m, lo:hi] = x[m, lo:hi]
    t = torch.from_numpy(x).cuda()
    win = {} if ks is None else {"ks": torch.from_numpy(ks).cuda(), "ke": torch.from_numpy(ke).cuda()}
    idx, val = fm.topk(t, k, sorted=False, **win)
    torch.cuda.synchronize()
    ri, _ = topk_rows(ref, k)
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    for m in range(M):
        n = int((ri[m] >= 0).sum())
        assert set(gi[m, :n].tolist()) == set(ri[m, :n].tolist()), f"{what}: row {m} differs"
        assert (gi[m, n:] == -1).all() and np.isneginf(gv[m, n:]).all(), f"{what}: row {m} padding"
        assert np.array_equal(gv[m, :n].view(np.uint32), x[m, gi[m, :n]].view(np.uint32)), \
            f"{what}: row {m} values"


@pytest.mark.parametrize("M,N,k", [(300, 8192, 512), (100, 5000, 1024), (40, 300, 512),
                                   (60, 20000, 512), (40, 20000, 2048), (40, 8192, 2048),
                                   (6, 70000, 512), (6, 70000, 2048)])
def test_unsorted_topk_selects_the_same_entries(M, N, k):
    # every layout: the staged-row kernel, the two-row kernels (k <= 512 and wider), the
    # one-row kernel; rows shorter than k get padding
    x = workloads.draw_logits(M, N, seed=M + N + k, neg_inf_frac=0.2)
    _check_unsorted(x, k, what=f"unsorted {M}x{N} k={k}")
    rng = np.random.default_rng(N + k)
    ks, ke = _windows(M, N, rng)
    _check_unsorted(x, k, ks, ke, what=f"unsorted windowed {M}x{N} k={k}")


def _windows(M, N, rng):
    # random windows, with empty ones, windows off either end and whole rows
    a = rng.integers(-50, N + 50, size=M)
    b = a + rng.integers(-20, N, size=M)
    a[::7], b[::7] = 0, N
    a[3::11], b[3::11] = N // 2, N // 2
    return a.astype(np.int32), b.astype(np.int32)


def _check_windowed(x, ks, ke, k, what):
    # the oracle sees the matrix with everything outside the windows made -inf
    M, N = x.shape
    ref = np.full_like(x, -np.inf)
    for m in range(M):
        lo, hi = max(int(ks[m]), 0), min(int(ke[m]), N)
        if lo < hi:
            ref[m, lo:hi] = x[m, lo:hi]
    poisoned = x.copy()
    for m in range(M):                    # garbage outside the windows: never read
        lo, hi = max(int(ks[m]), 0), min(int(ke[m]), N)
        poisoned[m, :max(lo, 0)] = np.nan
        poisoned[m, max(hi, 0):] = 3.0e38
    t = torch.from_numpy(poisoned).cuda()
    idx, val = fm.topk(t, k, ks=torch.from_numpy(ks).cuda(), ke=torch.from_numpy(ke).cuda())
    torch.cuda.synchronize()
    ri, rv = topk_rows(ref, k)
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    bad = np.nonzero((gi != ri).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: {len(bad)} rows differ, first {bad[0]}: " \
                          f"gpu {gi[bad[0]][:8]} oracle {ri[bad[0]][:8]}"
    assert np.array_equal(gv.view(np.uint32), rv.view(np.uint32)), what


@pytest.mark.parametrize("M,N", [(300, 8192), (200, 5000), (64, 1000), (40, 20000), (8, 40000),
                                 (6, 70000)])
@pytest.mark.parametrize("k", [1, 64, 512, 1024, 2048])
def test_windowed_rows_ignore_everything_outside_the_window(M, N, k):
    rng = np.random.default_rng(M + N + k)
    x = workloads.draw_logits(M, N, seed=N + k, neg_inf_frac=0.1)
    ks, ke = _windows(M, N, rng)
    _check_windowed(x, ks, ke, k, f"windowed {M}x{N} k={k}")


def test_windowed_topk_on_unclean_logits_equals_topk_on_clean_logits():
    from gpu_helpers import to_device
    for name in ("multi_req_8192x8192", "causal_8192x8192"):
        wl = workloads.WORKLOADS[name]
        dev = to_device(workloads.make(wl))
        args = (dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"])
        clean = fm.fp8_mqa_logits(*args)
        raw = torch.full_like(clean, float("nan"))
        fm.fp8_mqa_logits(*args, out=raw, clean_logits=False)   # outside the windows: NaN
        for k in (512, 2048):
            i0, v0 = fm.topk(clean, k)
            i1, v1 = fm.topk(raw, k, ks=dev["ks"], ke=dev["ke"])
            torch.cuda.synchronize()
            assert torch.equal(i0, i1) and torch.equal(v0.view(torch.int32), v1.view(torch.int32)), \
                f"{name} k={k}"

"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle element by element."""
import numpy as np
import torch

import fp8_mqa_logits_02_gb300 as fm
import oracle

NEG_INF_BITS = np.uint32(0xFF800000)
POISON_BITS = np.uint32(0x7FC0DEAD)  # a quiet NaN with a recognisable payload
ATOL = 1e-3
RTOL = 1e-3


def to_device(inp, device="cuda"):
    t = {}
    t["q"] = torch.from_numpy(inp["q"]).to(device).view(torch.float8_e4m3fn)
    t["k"] = torch.from_numpy(inp["k"]).to(device).view(torch.float8_e4m3fn)
    t["kv_scale"] = torch.from_numpy(inp["kv_scale"]).to(device)
    t["w"] = torch.from_numpy(inp["w"]).to(device)
    t["ks"] = torch.from_numpy(inp["ks"]).to(device)
    t["ke"] = torch.from_numpy(inp["ke"]).to(device)
    return t


def poisoned(M, N, device="cuda"):
    bits = torch.full((M, N), int(POISON_BITS.view(np.int32)), dtype=torch.int32, device=device)
    return bits.view(torch.float32)


def run_gpu(inp, clean=True, split_n=0, dev=None, out=None):
    dev = dev or to_device(inp)
    M, N = inp["M"], inp["N"]
    if out is None:
        out = poisoned(M, N)
    fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                      out=out, clean_logits=clean, split_n=split_n)
    status = fm.check_error()
    assert status == 0, fm.strerror(status)
    return out.cpu().numpy()


def run_oracle(inp, clean=True, rows=None):
    return oracle.fp8_mqa_logits(inp["q"], inp["k"], inp["kv_scale"], inp["w"], inp["ks"],
                                 inp["ke"], 1 if clean else 0, rows=rows)


def window_mask(ks, ke, N, rows=None):
    ks = ks.astype(np.int64)
    ke = ke.astype(np.int64)
    if rows is not None:
        ks, ke = ks[rows], ke[rows]
    n = np.arange(N, dtype=np.int64)[None, :]
    return (n >= np.clip(ks, 0, N)[:, None]) & (n < np.clip(ke, 0, N)[:, None])


def assert_parity(gpu, ref, inside, clean, extra_tol=None, what=""):
    """gpu: float32 [R,N]; ref: float64 [R,N] from the oracle; inside: bool mask."""
    bits = gpu.view(np.uint32)
    outside = ~inside
    if clean:
        bad = outside & (bits != NEG_INF_BITS)
        assert not bad.any(), f"{what}: {bad.sum()} out-of-window entries are not -inf " \
                              f"(first at {np.argwhere(bad)[0]})"
        assert np.all(np.isneginf(ref[outside]))
    else:
        bad = outside & (bits != POISON_BITS)
        assert not bad.any(), f"{what}: {bad.sum()} out-of-window entries were written " \
                              f"(first at {np.argwhere(bad)[0]})"
    g = gpu[inside].astype(np.float64)
    r = ref[inside]
    assert np.all(np.isfinite(r))
    assert np.all(np.isfinite(g)), f"{what}: non-finite in-window values"
    tol = ATOL + RTOL * np.abs(r)
    if extra_tol is not None:
        tol = tol + extra_tol[inside]
    err = np.abs(g - r)
    worst = np.argmax(err - tol) if err.size else 0
    assert np.all(err <= tol), (f"{what}: {int((err > tol).sum())} in-window values out of "
                                f"tolerance; worst |err|={err.flat[worst]:.3e} "
                                f"tol={tol.flat[worst]:.3e} ref={r.flat[worst]:.6g}")


def assert_parity_full(outputs, inp, block_rows=256, what=""):
    """Every entry of full-size GPU outputs against the oracle.

    outputs: list of (label, float32 [M, N] host array, clean) for one workload's inputs.
    The oracle runs once, in blocks of ``block_rows`` rows (bounded host memory), and every
    output is compared element by element with each block: the mask bit-exact (-inf with
    clean_logits=1, the untouched poison with 0) and every in-window value within the
    tolerance."""
    M, N = inp["M"], inp["N"]
    for r0 in range(0, M, block_rows):
        rows = np.arange(r0, min(M, r0 + block_rows), dtype=np.int64)
        ref = run_oracle(inp, clean=True, rows=rows)
        inside = window_mask(inp["ks"], inp["ke"], N, rows)
        for label, gpu, clean in outputs:
            assert_parity(gpu[r0:r0 + len(rows)], ref, inside, clean,
                          what=f"{what} {label} rows {r0}..{r0 + len(rows) - 1}")

"""The bounds-checking build (libfp8mqa_debug.so, compiled with FP8MQA_DEBUG_BOUNDS).

Its kernel checks every global store and load, every TMA coordinate and every TMEM column
before using it, and records the first violation in the status word instead of making the
access (fp8_mqa_logits_check_error then returns FP8MQA_ERR_BOUNDS).  That build stands in
for a memory checker, which cannot be run here.  The small cases of the parity suite run
through it once: every call must record nothing and match the oracle.
"""
import numpy as np
import pytest
import torch

import fp8_mqa_logits_02_gb300 as fm
import workloads
from gpu_helpers import assert_parity, poisoned, run_gpu, run_oracle, to_device, window_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _debug_lib():
    fm.build()
    fm.use_debug_library(True)
    fm.lib()
    yield
    fm.use_debug_library(False)


def _inputs(M, N, family, seed):
    q, k, kv, w = workloads.draw(M, N, seed)
    ks, ke = workloads.windows(family, M, N)
    return {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke, "M": M, "N": N,
            "H": 32, "D": 128}


@pytest.mark.parametrize("family", workloads.WINDOW_FAMILIES)
def test_window_families_record_no_violation(family):
    inp = _inputs(96, 1040, family, seed=41)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    for clean in (True, False):
        for split_n in (0, 1, 3, 20):
            gpu = run_gpu(inp, clean=clean, split_n=split_n)  # asserts check_error() == 0
            assert_parity(gpu, ref, inside, clean, what=f"debug {family} {clean} {split_n}")


@pytest.mark.parametrize("M,N", [(1, 1), (3, 127), (9, 129), (127, 1000), (129, 128), (64, 256)])
def test_ragged_shapes_record_no_violation(M, N):
    for family in ("causal", "misaligned", "past_end"):
        inp = _inputs(M, N, family, seed=M * 7 + N)
        gpu = run_gpu(inp, clean=True)
        assert_parity(gpu, run_oracle(inp, clean=True), window_mask(inp["ks"], inp["ke"], N),
                      True, what=f"debug M={M} N={N} {family}")


def test_noalloc_and_host_entries_record_no_violation():
    inp = _inputs(200, 3000, "multi_req", seed=43)
    dev = to_device(inp)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], 3000)
    out = poisoned(200, 3000)
    stream = torch.cuda.current_stream().cuda_stream
    rc = fm.lib().fp8_mqa_logits_noalloc(dev["q"].data_ptr(), dev["k"].data_ptr(),
                                         dev["kv_scale"].data_ptr(), dev["w"].data_ptr(),
                                         dev["ks"].data_ptr(), dev["ke"].data_ptr(),
                                         out.data_ptr(), 200, 3000, 32, 128, 1, 0, stream)
    assert rc == 0
    assert fm.check_error() == 0
    assert_parity(out.cpu().numpy(), ref, inside, True, what="debug noalloc")
    cpu = {k: torch.from_numpy(inp[k]).pin_memory() for k in ("q", "k", "kv_scale", "w", "ks", "ke")}
    hout = torch.empty((200, 3000), dtype=torch.float32).pin_memory()
    ws = torch.empty(fm.host_workspace_bytes(200, 3000), dtype=torch.uint8, device="cuda")
    fm.fp8_mqa_logits_host(cpu["q"], cpu["k"], cpu["kv_scale"], cpu["w"], cpu["ks"], cpu["ke"],
                           hout, ws)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    assert_parity(hout.numpy(), ref, inside, True, what="debug host entry")


def test_full_size_causal_records_no_violation():
    inp = workloads.make(workloads.WORKLOADS["causal_8192x8192"])
    dev = to_device(inp)
    out = poisoned(8192, 8192)
    fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                      out=out)
    assert fm.check_error() == 0
    rows = np.array([0, 1, 127, 128, 4095, 8191])
    assert_parity(out.cpu().numpy()[rows], run_oracle(inp, clean=True, rows=rows),
                  window_mask(inp["ks"], inp["ke"], 8192, rows), True, what="debug causal")

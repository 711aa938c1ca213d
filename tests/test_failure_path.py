"""The kernel's failure path, made to run without planting anything.

Every pipeline wait inside the kernel is bounded; when one runs out the CTA raises an abort
flag and a status bit, waits for its own copies and tensor-core work in flight (under a
separate bound), frees its tensor memory and exits, and the last CTA resets the launch's
scheduler slot.  A short wait limit (fp8_mqa_logits_set_wait_limit_ns) makes the waits of a
normal call run out.  The tests check that the call returns, that check_error reports
FP8MQA_ERR_TIMEOUT, and that later calls on the same device -- through every scheduler slot,
including the one the failed call used -- are correct again.  (Failure detection in its
safe form: a bounded wait that gives up, never a GPU fault.)
"""
import numpy as np
import pytest
import torch

import fp8_mqa_logits_02_gb300 as fm
import workloads
from gpu_helpers import assert_parity, poisoned, run_oracle, to_device, window_mask

pytestmark = pytest.mark.gpu

TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.build()
    fm.lib()
    yield
    fm.set_wait_limit_ns(0)


def _inputs(M, N, family, seed):
    q, k, kv, w = workloads.draw(M, N, seed)
    ks, ke = workloads.windows(family, M, N)
    return {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke, "M": M, "N": N,
            "H": 32, "D": 128}


def test_short_wait_limit_times_out_then_every_slot_recovers():
    big = _inputs(2048, 8192, "causal", seed=31)
    dbig = to_device(big)
    out_big = poisoned(2048, 8192)
    small = _inputs(96, 1040, "misaligned", seed=32)
    dsmall = to_device(small)
    ref = run_oracle(small, clean=True)
    inside = window_mask(small["ks"], small["ke"], small["N"])
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    prev = fm.set_wait_limit_ns(200)  # far below a pipeline stage's latency
    try:
        for split_n in (0, 5):
            fm.fp8_mqa_logits(dbig["q"], dbig["k"], dbig["kv_scale"], dbig["w"], dbig["ks"],
                              dbig["ke"], out=out_big, split_n=split_n)
            assert fm.check_error() == TIMEOUT
    finally:
        fm.set_wait_limit_ns(prev)
    # status cleared by the read
    assert fm.check_error() == 0
    # 260 calls walk the whole ring of 256 direct-launch slots, so the two that failed are
    # reused; each call's output must match the oracle
    outs = [poisoned(96, 1040) for _ in range(4)]
    for i in range(260):
        o = outs[i % 4]
        fm.fp8_mqa_logits(dsmall["q"], dsmall["k"], dsmall["kv_scale"], dsmall["w"],
                          dsmall["ks"], dsmall["ke"], out=o, split_n=i % 3)
        if i % 4 == 3 or i == 259:
            torch.cuda.synchronize()
            for oo in outs:
                assert_parity(oo.cpu().numpy(), ref, inside, True, what=f"after timeout, call {i}")
                oo.copy_(poisoned(96, 1040))
    assert fm.check_error() == 0
    # the full-size call is correct again too
    out_big.copy_(poisoned(2048, 8192))
    fm.fp8_mqa_logits(dbig["q"], dbig["k"], dbig["kv_scale"], dbig["w"], dbig["ks"], dbig["ke"],
                      out=out_big)
    assert fm.check_error() == 0
    rows = np.array([0, 1, 7, 8, 1023, 1024, 2040, 2047])
    assert_parity(out_big.cpu().numpy()[rows], run_oracle(big, clean=True, rows=rows),
                  window_mask(big["ks"], big["ke"], big["N"], rows), True, what="big after")


def test_noalloc_entry_reports_its_timeout_through_check_error():
    inp = _inputs(1024, 8192, "causal", seed=33)
    dev = to_device(inp)
    lib = fm.lib()
    stream = torch.cuda.current_stream().cuda_stream

    def call(out):
        rc = lib.fp8_mqa_logits_noalloc(dev["q"].data_ptr(), dev["k"].data_ptr(),
                                        dev["kv_scale"].data_ptr(), dev["w"].data_ptr(),
                                        dev["ks"].data_ptr(), dev["ke"].data_ptr(),
                                        out.data_ptr(), 1024, 8192, 32, 128, 1, 0, stream)
        assert rc == 0, fm.strerror(rc)

    out = poisoned(1024, 8192)
    call(out)
    assert fm.check_error() == 0  # the array's status word reads zero after a normal call
    prev = fm.set_wait_limit_ns(200)
    try:
        call(out)
        assert fm.check_error() == TIMEOUT
    finally:
        fm.set_wait_limit_ns(prev)
    assert fm.check_error() == 0
    out.copy_(poisoned(1024, 8192))
    call(out)
    assert fm.check_error() == 0
    rows = np.array([0, 5, 511, 512, 1016, 1023])
    assert_parity(out.cpu().numpy()[rows], run_oracle(inp, clean=True, rows=rows),
                  window_mask(inp["ks"], inp["ke"], 8192, rows), True, what="noalloc after")

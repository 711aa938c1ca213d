"""The allocation-free entry point, fp8_mqa_logits_noalloc, against fp8_mqa_logits.

Some callers cannot allocate device memory: serving engines that reserve nearly all
HBM for their own pools, plug-in interfaces that bar a plug-in from allocating, and
latency-critical loops that cannot afford an allocation that may synchronize the
device.  For them the library keeps this entry point's scratch in a fixed device array
compiled into the library.  This test calls it through the C ABI twice in a row and
checks that each output equals the regular entry point's output bit for bit (the two run
the same kernel on the same inputs; with clean_logits = 0 the untouched poison must
survive too), that check_error reads a clear status word after each call, and that the
second call leaves the free device memory unchanged.  It only needs a GPU, so it passes
alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import fp8_mqa_logits_02_gb300 as fm
import workloads
from gpu_helpers import poisoned, to_device

pytestmark = pytest.mark.gpu


def _call(fn, dev, out, M, N, clean, split_n):
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["kv_scale"].data_ptr(),
            dev["w"].data_ptr(), dev["ks"].data_ptr(), dev["ke"].data_ptr(), out.data_ptr(),
            M, N, 32, 128, clean, split_n, stream)
    assert rc == 0, fm.strerror(rc)


@pytest.mark.parametrize("clean", [1, 0])
def test_noalloc_matches_regular_entry_on_two_calls(clean):
    fm.build()
    fm.use_debug_library(False)
    lib = fm.lib()
    M, N = 300, 3000
    q, k, kv, w = workloads.draw(M, N, seed=21)
    ks, ke = workloads.windows("misaligned", M, N)
    inp = {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke, "M": M, "N": N}
    dev = to_device(inp)

    ref = poisoned(M, N)
    _call(lib.fp8_mqa_logits, dev, ref, M, N, clean, 0)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    ref_bits = ref.cpu().numpy().view(np.uint32)

    for call in range(2):
        out = poisoned(M, N)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _call(lib.fp8_mqa_logits_noalloc, dev, out, M, N, clean, 0)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free_after == free_before, "the allocation-free entry point allocated"
        assert fm.check_error() == 0, "the allocation-free call recorded a failure"
        bits = out.cpu().numpy().view(np.uint32)
        diff = bits != ref_bits
        assert not diff.any(), (f"noalloc call {call} clean={clean}: {int(diff.sum())} entries "
                                f"differ from fp8_mqa_logits (first at {np.argwhere(diff)[0]})")

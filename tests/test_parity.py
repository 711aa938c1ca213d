"""GPU parity: the sm_103a CUDA path, called through the C ABI, against the fp64 CPU oracle.

Bar: the -inf mask bit-exact (IEEE 0xff800000 outside [ks, ke) with clean_logits=1,
untouched poison with clean_logits=0) and every in-window value within
1e-3 + 1e-3*|oracle| of the fp64 oracle, on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import fp8_mqa_logits_02_gb300 as fm
import workloads
from gpu_helpers import (assert_parity, assert_parity_full, poisoned, run_gpu, run_oracle,
                         to_device, window_mask)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fm.build()
    fm.lib()


def _inputs(M, N, family, seed, requests=4):
    q, k, kv, w = workloads.draw(M, N, seed)
    ks, ke = workloads.windows(family, M, N, requests)
    return {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke, "M": M, "N": N,
            "H": 32, "D": 128}


# ------------------------------------------------------------------ the tiny workload, full
@pytest.mark.parametrize("clean", [True, False])
@pytest.mark.parametrize("split_n", [0, 1, 2])
def test_tiny_causal_full(clean, split_n):
    inp = workloads.make(workloads.WORKLOADS["tiny_causal_64x256"])
    gpu = run_gpu(inp, clean=clean, split_n=split_n)
    ref = run_oracle(inp, clean=clean)
    assert_parity(gpu, ref, window_mask(inp["ks"], inp["ke"], inp["N"]), clean,
                  what=f"tiny clean={clean} split={split_n}")


# ------------------------------------------------------------------ window families
@pytest.mark.parametrize("family", workloads.WINDOW_FAMILIES)
@pytest.mark.parametrize("clean", [True, False])
def test_window_families(family, clean):
    M, N = 96, 1040  # several row blocks and key tiles, ragged last tile
    inp = _inputs(M, N, family, seed=17)
    ref = run_oracle(inp, clean=clean)
    inside = window_mask(inp["ks"], inp["ke"], N)
    for split_n in (0, 1, 3, 20):
        gpu = run_gpu(inp, clean=clean, split_n=split_n)
        assert_parity(gpu, ref, inside, clean, what=f"{family} clean={clean} split={split_n}")


# ------------------------------------------------------------------ ragged shapes
@pytest.mark.parametrize("M", [1, 3, 8, 9, 127, 129])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 1000])
def test_ragged_shapes(M, N):
    for family in ("causal", "misaligned"):
        inp = _inputs(M, N, family, seed=M * 1000 + N)
        ref = run_oracle(inp, clean=True)
        gpu = run_gpu(inp, clean=True)
        assert_parity(gpu, ref, window_mask(inp["ks"], inp["ke"], N), True,
                      what=f"M={M} N={N} {family}")


def test_all_rows_empty_and_out_of_range():
    M, N = 40, 700
    inp = _inputs(M, N, "causal", seed=5)
    inp["ks"] = np.array([(7 * m) % N + 3 for m in range(M)], np.int32)
    inp["ke"] = inp["ks"] - (np.arange(M, dtype=np.int32) % 3)       # ks >= ke: empty
    inp["ks"][::5] = N + 10                                            # starts past the end
    inp["ke"][::5] = N + 50
    inp["ks"][1::7] = -100                                             # negative, still empty
    inp["ke"][1::7] = -3
    gpu = run_gpu(inp, clean=True)
    assert np.all(gpu.view(np.uint32) == 0xFF800000)
    out0 = run_gpu(inp, clean=False)
    assert np.all(out0.view(np.uint32) == 0x7FC0DEAD)


# ------------------------------------------------------------------ invariants on the GPU
def test_split_n_bit_identical_and_clean_consistent():
    inp = _inputs(200, 3000, "misaligned", seed=9)
    dev = to_device(inp)
    base = run_gpu(inp, clean=True, split_n=1, dev=dev)
    for split_n in (0, 2, 3, 7, 20, 24, 1000):
        other = run_gpu(inp, clean=True, split_n=split_n, dev=dev)
        assert np.array_equal(base.view(np.uint32), other.view(np.uint32)), split_n
    unclean = run_gpu(inp, clean=False, split_n=5, dev=dev)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    assert np.array_equal(base.view(np.uint32)[inside], unclean.view(np.uint32)[inside])


def test_wide_dynamic_range_codes():
    # Q, K drawn uniformly over every finite E4M3 code (subnormals to +-448).  The dots
    # then reach ~1e7 and fp32 accumulation on the tensor cores is the precision the
    # page specifies, so the bound adds 2^-19 x sum_h relu(S)|w| kv (oracle with |w|).
    rng = np.random.default_rng(3)
    M, N = 64, 512
    inp = _inputs(M, N, "misaligned", seed=3)
    for name, shape in (("q", (M, 32, 128)), ("k", (N, 128))):
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        inp[name] = np.where((c & 0x7F) == 0x7F, c & 0xF8, c).astype(np.uint8)
    ref = run_oracle(inp, clean=True)
    absw = dict(inp, w=np.abs(inp["w"]))
    mag = np.abs(run_oracle(absw, clean=True))
    mag[~np.isfinite(mag)] = 0
    gpu = run_gpu(inp, clean=True)
    assert_parity(gpu, ref, window_mask(inp["ks"], inp["ke"], N), True,
                  extra_tol=mag * 2.0 ** -19, what="wide range")


def test_many_calls_reuse_scheduler_slots():
    # more calls than the library's ring of 256 scheduler slots, back to back on one stream
    inp = _inputs(24, 600, "misaligned", seed=11)
    dev = to_device(inp)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    outs = [poisoned(24, 600) for _ in range(270)]
    for i, o in enumerate(outs):
        fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                          out=o, clean_logits=True, split_n=i % 4)
    assert fm.check_error() == 0
    for o in outs:
        assert_parity(o.cpu().numpy(), ref, inside, True, what="repeat")


def test_two_streams_concurrently():
    inp = _inputs(300, 2500, "causal", seed=12)
    dev = to_device(inp)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, o2 = poisoned(300, 2500), poisoned(300, 2500)
    torch.cuda.synchronize()
    fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                      out=o1, stream=s1)
    fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                      out=o2, stream=s2, split_n=3)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    assert_parity(o1.cpu().numpy(), ref, inside, True, what="stream 1")
    assert_parity(o2.cpu().numpy(), ref, inside, True, what="stream 2")


def test_host_buffer_entry_point():
    inp = _inputs(50, 900, "multi_req", seed=13, requests=2)
    ref = run_oracle(inp, clean=True)
    cpu = {k: torch.from_numpy(inp[k]).pin_memory()
           for k in ("q", "k", "kv_scale", "w", "ks", "ke")}
    out = torch.empty((50, 900), dtype=torch.float32).pin_memory()
    ws = torch.empty(fm.host_workspace_bytes(50, 900), dtype=torch.uint8, device="cuda")
    fm.fp8_mqa_logits_host(cpu["q"], cpu["k"], cpu["kv_scale"], cpu["w"], cpu["ks"], cpu["ke"],
                           out, ws)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    assert_parity(out.numpy(), ref, window_mask(inp["ks"], inp["ke"], 900), True, what="host")


@pytest.mark.parametrize("clean", [True, False])
def test_host_buffer_entry_point_in_chunks(clean):
    # 4096 x 8192 logits are 134 MB: the host entry splits them into four row chunks whose
    # input copies, kernels and read-backs overlap.  Parity on sampled rows of every chunk;
    # with clean_logits = 0 the poisoned host buffer must come back untouched outside the
    # windows.  The result also equals the device-buffer entry's, bit for bit (the kernel
    # output does not depend on how rows or keys are split).
    M, N = 4096, 8192
    inp = _inputs(M, N, "causal", seed=17)
    cpu = {k: torch.from_numpy(inp[k]).pin_memory()
           for k in ("q", "k", "kv_scale", "w", "ks", "ke")}
    out = poisoned(M, N, device="cpu").pin_memory()
    ws = torch.empty(fm.host_workspace_bytes(M, N), dtype=torch.uint8, device="cuda")
    fm.fp8_mqa_logits_host(cpu["q"], cpu["k"], cpu["kv_scale"], cpu["w"], cpu["ks"], cpu["ke"],
                           out, ws, clean_logits=clean)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    host = out.numpy()
    rows = np.array(sorted({0, 1, 1023, 1024, 1025, 2047, 2048, 3071, 3072, 4094, 4095}
                           | set(np.random.default_rng(3).choice(M, 21, replace=False).tolist())))
    ref = run_oracle(inp, clean=clean, rows=rows)
    assert_parity(host[rows], ref, window_mask(inp["ks"], inp["ke"], N, rows), clean,
                  what=f"host chunks clean={clean}")
    dev = run_gpu(inp, clean=clean)
    assert np.array_equal(host.view(np.uint32), dev.view(np.uint32))


# ------------------------------------------------------------------ full-size workloads
# Every workload at full size, every output entry against the oracle (computed in row
# blocks), for each (clean_logits, split_n) the bench and the page's table use.
FULL_SIZE = {
    "causal_8192x8192": [(1, 0), (0, 0)],
    "chunk_causal_4096x32768": [(1, 0), (0, 0)],
    "long_causal_1024x131072": [(1, 0)],
    "multi_req_4096x32768": [(1, 0), (1, 20), (0, 0)],
    "kpool_causal_16384x32000": [(1, 0)],
    "cp_4096x32768": [(1, 0), (0, 3)],
    "chunk_causal_2048x65536": [(1, 0)],
    "multi_req_2048x65536": [(1, 0)],
    "multi_req_1024x131072": [(1, 0), (1, 20)],
    "multi_req_8192x8192": [(1, 0)],
    "small_causal_1024x1024": [(1, 0), (0, 0), (1, 3)],
    "small_causal_128x4096": [(1, 0), (0, 0)],
}


@pytest.mark.parametrize("name", list(FULL_SIZE))
def test_full_workloads(name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make(wl)
    M, N = inp["M"], inp["N"]
    dev = to_device(inp)
    outputs = []
    for clean, split_n in FULL_SIZE[name]:
        out = poisoned(M, N)
        fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                          out=out, clean_logits=bool(clean), split_n=split_n)
        assert fm.check_error() == 0
        outputs.append((f"clean={clean} split={split_n}", out.cpu().numpy(), bool(clean)))
        del out
    # the output does not depend on the split: the in-window bits of every variant agree
    base = outputs[0][1].view(np.uint32)
    for label, gpu, _ in outputs[1:]:
        bits = gpu.view(np.uint32)
        for r0 in range(0, M, 512):
            inside = window_mask(inp["ks"], inp["ke"], N, np.arange(r0, min(M, r0 + 512)))
            assert np.array_equal(base[r0:r0 + 512][inside], bits[r0:r0 + 512][inside]), label
    assert_parity_full(outputs, inp, block_rows=max(8, (1 << 25) // N), what=name)


def test_call_captured_in_a_cuda_graph():
    # After the first call on the device (which sets up the library's scratch), a call can be
    # captured on a stream and replayed; every replay recomputes the whole output.
    inp = _inputs(200, 3000, "misaligned", seed=13)
    dev = to_device(inp)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    out = poisoned(200, 3000)
    fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                      out=out)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fm.fp8_mqa_logits(dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"],
                          out=out, stream=s)
    for _ in range(3):
        out.copy_(poisoned(200, 3000))
        graph.replay()
        torch.cuda.synchronize()
        assert fm.check_error() == 0
        assert_parity(out.cpu().numpy(), ref, inside, True, what="graph replay")


def test_graph_replay_while_direct_calls_run_on_another_stream():
    # A captured launch keeps its scheduler slot for every replay.  Replays on one stream
    # while 300 direct calls (more than the ring of 256 direct slots) go out on another must
    # not share a slot with any of them.
    inp = _inputs(160, 2600, "misaligned", seed=23)
    dev = to_device(inp)
    ref = run_oracle(inp, clean=True)
    inside = window_mask(inp["ks"], inp["ke"], inp["N"])
    args = (dev["q"], dev["k"], dev["kv_scale"], dev["w"], dev["ks"], dev["ke"])
    out_g = poisoned(160, 2600)
    fm.fp8_mqa_logits(*args, out=out_g)  # set-up before capture
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=sa):
        fm.fp8_mqa_logits(*args, out=out_g, stream=sa)
    outs = [poisoned(160, 2600) for _ in range(8)]
    torch.cuda.synchronize()
    replays = []
    for i in range(300):
        if i % 25 == 0:
            with torch.cuda.stream(sa):
                out_g.copy_(poisoned(160, 2600))
                graph.replay()
                replays.append(out_g.clone())
        fm.fp8_mqa_logits(*args, out=outs[i % 8], stream=sb, split_n=i % 3)
    torch.cuda.synchronize()
    assert fm.check_error() == 0
    for o in outs + replays:
        assert_parity(o.cpu().numpy(), ref, inside, True, what="graph and direct calls")


def test_host_entry_captured_in_a_cuda_graph():
    # The host-buffer entry forks its two library streams from the caller's stream and joins
    # them again, so a call (here in two row chunks: 67 MB of logits) can be captured and
    # replayed; each replay copies in, computes and copies back the whole output.
    M, N = 2048, 8192
    inp = _inputs(M, N, "causal", seed=19)
    cpu = {k: torch.from_numpy(inp[k]).pin_memory()
           for k in ("q", "k", "kv_scale", "w", "ks", "ke")}
    out = poisoned(M, N, device="cpu").pin_memory()
    ws = torch.empty(fm.host_workspace_bytes(M, N), dtype=torch.uint8, device="cuda")
    args = (cpu["q"], cpu["k"], cpu["kv_scale"], cpu["w"], cpu["ks"], cpu["ke"], out, ws)
    fm.fp8_mqa_logits_host(*args)  # the first call on the device sets the library up
    torch.cuda.synchronize()
    rows = np.array(sorted({0, 7, 1023, 1024, 1031, 2047}
                           | set(np.random.default_rng(5).choice(M, 10, replace=False).tolist())))
    ref = run_oracle(inp, clean=True, rows=rows)
    inside = window_mask(inp["ks"], inp["ke"], N, rows)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fm.fp8_mqa_logits_host(*args, stream=s)
    for _ in range(2):
        out.copy_(poisoned(M, N, device="cpu"))
        graph.replay()
        torch.cuda.synchronize()
        assert fm.check_error() == 0
        assert_parity(out.numpy()[rows], ref, inside, True, what="host entry graph replay")


# ------------------------------------------------------------------ randomized configurations
def _random_config(rng):
    M = int(rng.integers(1, 100))
    N = int(rng.integers(1, 2000))
    q, k, kv, w = workloads.draw(M, N, int(rng.integers(0, 1 << 30)))
    # arbitrary per-row windows: negative starts, ends past N, empty and reversed rows
    ks = rng.integers(-50, N + 50, size=M)
    ke = ks + rng.integers(-20, N + 100, size=M)
    return {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks.astype(np.int32),
            "ke": ke.astype(np.int32), "M": M, "N": N, "H": 32, "D": 128}


@pytest.mark.parametrize("case", range(40))
def test_randomized_configs(case):
    rng = np.random.default_rng(1000 + case)
    inp = _random_config(rng)
    clean = bool(rng.integers(0, 2))
    split = int(rng.choice([0, 1, 2, 3, 7, 50]))
    gpu = run_gpu(inp, clean=clean, split_n=split)
    ref = run_oracle(inp, clean=clean)
    assert_parity(gpu, ref, window_mask(inp["ks"], inp["ke"], inp["N"]), clean,
                  what=f"random case {case}: M={inp['M']} N={inp['N']} clean={clean} "
                       f"split={split}")

"""Benchmark of the prefill FP8 MQA indexer logits on one GB300 (or N replicas).

A step is one call of the whole path (``fp8_mqa_logits``) on one batch of the
causal 8192 x 8192 workload (H=32, D=128; the kernel-time table's first shape in
ROCm/aiter PR #7183).  Inputs are resident in HBM before the timed region; L2 is
flushed (a 256 MiB write) before every timed call, and each call is timed on the
launching stream with CUDA events.  The metric is valid-window FP8 TFLOP/s:
2*H*D*sum_m |window_m| per call over the call's device time.

The same JSON line carries a "workloads" block: every other configuration of the page's
kernel-time table (and the clean_logits = 0 and explicit-split variants) timed the same
way, so that each figure quoted for them comes from this run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference] [--no-cpu-baseline] [--no-workloads]

``--gpus N`` with N > 1 outside torchrun starts N replica ranks itself (one per GPU,
through torch.distributed.run); under torchrun each rank runs the same full call and the
job time is the slowest rank's.  ``--impl reference`` times the CPU oracle (test
infrastructure) on the host cores on a bounded sample of the same workload and prints the
same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import socket
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "valid-window FP8 TFLOP/s and µs/call at 1 GB300; % of dense FP8 tensor peak"
DEFAULT_WORKLOAD = "causal_8192x8192"
FLUSH_BYTES = 256 << 20


def host_lead(stream):
    """Keep the GPU busy for about 2 ms (a fixed-length spin on `stream`) before a device-timed
    loop: the host then enqueues the first steps ahead of the GPU, so no host-side launch
    latency (argument checks, allocations, the clock sampler starting) falls between a step's
    start event and its launch.  Later steps stay queued: each takes the GPU longer than the
    host needs to issue it."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(4_000_000)


# the recipe's fallback peaks, used only when the measured file is absent
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0  # nominal dense ratio 4.5 / 2.25 PFLOP/s
REFERENCE_BUDGET_S = 90.0  # CPU seconds for a whole --impl reference run

# The per-workload block: (workload, clean_logits, split_n); split_n 0 is the default.
WORKLOAD_TABLE = [
    ("tiny_causal_64x256", 1, 0),
    ("small_causal_128x4096", 1, 0),
    ("small_causal_1024x1024", 1, 0),
    ("causal_8192x8192", 0, 0),
    ("chunk_causal_4096x32768", 1, 0),
    ("chunk_causal_4096x32768", 0, 0),
    ("chunk_causal_2048x65536", 1, 0),
    ("long_causal_1024x131072", 1, 0),
    ("kpool_causal_16384x32000", 1, 0),
    ("cp_4096x32768", 1, 0),
    ("multi_req_4096x32768", 1, 0),
    ("multi_req_4096x32768", 1, 20),
    ("multi_req_4096x32768", 0, 0),
    ("multi_req_2048x65536", 1, 0),
    ("multi_req_1024x131072", 1, 0),
    ("multi_req_1024x131072", 1, 20),
    ("multi_req_8192x8192", 1, 0),
]


def valid_flops(inp) -> float:
    return 2.0 * inp["H"] * inp["D"] * workloads.valid_pairs(inp["ks"], inp["ke"], inp["N"])


def algorithmic_bytes(inp, clean: int) -> float:
    """HBM bytes one call must move: the logits it writes (every entry with clean_logits=1,
    the in-window ones with 0), Q and w once, K and kv_scale once, ks and ke."""
    M, N, H, D = inp["M"], inp["N"], inp["H"], inp["D"]
    pairs = workloads.valid_pairs(inp["ks"], inp["ke"], N)
    out = 4.0 * (M * N if clean else pairs)
    return out + M * H * D + M * H * 4 + N * (D + 4) + 8.0 * M


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                    "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                         d["bf16_tflops"])),
                    "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                             "hw": f[5], "hw_thermal": f[6], "sw_thermal": f[7],
                             "sw_power": f[8]})
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"),
                              ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(busy)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the rank-aggregation the timing contract asks for)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = "cuda" if backend == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def replica_command(gpus: int, argv, port: int | None = None):
    """The torch.distributed.run command that starts `gpus` replica ranks of this script
    with the same arguments (one process per GPU, rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={gpus}", "--master-addr=127.0.0.1",
            f"--master-port={port or _free_port()}", os.path.abspath(__file__), *argv]


def cpu_oracle_sample(inp, budget_rows: int, threads: int):
    """Time the oracle on an evenly spaced sample of query rows; returns TFLOP/s etc."""
    import oracle
    M = inp["M"]
    stride = max(1, M // budget_rows)
    rows = np.arange(0, M, stride, dtype=np.int64)[:budget_rows]
    pairs = workloads.valid_pairs(inp["ks"][rows], inp["ke"][rows], inp["N"])
    flops = 2.0 * inp["H"] * inp["D"] * pairs
    t0 = time.perf_counter()
    oracle.fp8_mqa_logits(inp["q"], inp["k"], inp["kv_scale"], inp["w"], inp["ks"], inp["ke"],
                          1, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"tflops": flops / dt / 1e12, "seconds": dt, "rows": int(len(rows)),
            "stride": int(stride), "flops": flops}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make(wl)
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    # size each step so the whole run (warm-up + steps) takes about REFERENCE_BUDGET_S
    probe = cpu_oracle_sample(inp, 64, threads)
    per_row = probe["seconds"] / probe["rows"]
    rows_per_step = int(REFERENCE_BUDGET_S / per_row / (args.steps + 0.25 * args.warmup))
    rows_per_step = max(8, min(inp["M"], rows_per_step))
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, max(8, rows_per_step // 4), threads)
    samples = [cpu_oracle_sample(inp, rows_per_step, threads) for _ in range(args.steps)]
    flops = sum(s["flops"] for s in samples)
    secs = sum(s["seconds"] for s in samples)
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "H": wl.H, "D": wl.D,
                   "windows": workloads.describe(wl), "clean_logits": int(args.clean),
                   "split_n": args.split_n, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{samples[0]['rows']} query rows per step (every "
                                   f"{samples[0]['stride']}th row) of {wl.name}, fp64 C "
                                   f"oracle on {threads} host threads"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _device_inputs(inp, dev):
    import torch
    return (torch.from_numpy(inp["q"]).to(dev).view(torch.float8_e4m3fn),
            torch.from_numpy(inp["k"]).to(dev).view(torch.float8_e4m3fn),
            torch.from_numpy(inp["kv_scale"]).to(dev), torch.from_numpy(inp["w"]).to(dev),
            torch.from_numpy(inp["ks"]).to(dev), torch.from_numpy(inp["ke"]).to(dev))


def time_calls(fm, args_dev, out, clean, split_n, steps, warmup, flush, stream, dev):
    """Mean device time (ms) of `steps` calls, each after an L2 flush, CUDA events on the
    launching stream; plus the clocks sampled meanwhile."""
    import torch

    def call():
        fm.fp8_mqa_logits(*args_dev, out=out, clean_logits=bool(clean), split_n=split_n,
                          stream=stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    if fm.check_error(stream) != 0:
        raise RuntimeError("device status after warm-up is not OK")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks:
        host_lead(stream)
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    status = fm.check_error(stream)
    if status != 0:
        raise RuntimeError(f"device status {fm.strerror(status)}")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], clocks.summary()


def back_to_back_us(fm, args_dev, out, clean, split_n, calls, stream, dev):
    """Mean µs per call over `calls` calls issued back to back between two events."""
    import torch
    for _ in range(10):
        fm.fp8_mqa_logits(*args_dev, out=out, clean_logits=bool(clean), split_n=split_n,
                          stream=stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(calls):
        fm.fp8_mqa_logits(*args_dev, out=out, clean_logits=bool(clean), split_n=split_n,
                          stream=stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    if fm.check_error(stream) != 0:
        raise RuntimeError("device status after back-to-back calls is not OK")
    return 1e3 * a.elapsed_time(b) / calls


def workload_block(fm, dev, stream, flush, steps, warmup, fp8_peak, hbm_peak, sm_count):
    """Every configuration of WORKLOAD_TABLE timed like the headline call."""
    import torch
    rows = []
    cache = {}
    for name, clean, split_n in WORKLOAD_TABLE:
        wl = workloads.WORKLOADS[name]
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            inp = workloads.make(wl)
            cache[name] = (inp, _device_inputs(inp, dev))
        inp, args_dev = cache[name]
        out = torch.empty((inp["M"], inp["N"]), dtype=torch.float32, device=dev)
        ms, clocks = time_calls(fm, args_dev, out, clean, split_n, steps, warmup, flush,
                                stream, dev)
        back_to_back = None
        if inp["M"] * inp["N"] <= (1 << 22):
            # small problems: also the mean over calls issued back to back (no flush between
            # them), where a call's launch overlaps the previous call's execution
            back_to_back = back_to_back_us(fm, args_dev, out, clean, split_n, 200, stream, dev)
        del out
        mean_s = statistics.mean(ms) * 1e-3
        flops = valid_flops(inp)
        nbytes = algorithmic_bytes(inp, clean)
        split_used = split_n or fm.default_split(inp["M"], inp["N"], sm_count)
        rows.append({
            "workload": name, "windows": workloads.describe(wl), "clean_logits": clean,
            "split_n": split_n, "split_used": split_used, "steps": steps,
            "us_per_call": mean_s * 1e6, "us_min": min(ms) * 1e3,
            "tflops": flops / mean_s / 1e12, "frac_of_fp8_peak": flops / mean_s / 1e12 / fp8_peak,
            "hbm_gbs": nbytes / mean_s / 1e9, "frac_of_hbm": nbytes / mean_s / 1e9 / hbm_peak,
            "us_per_call_back_to_back": back_to_back, "clocks": clocks})
    return rows


def run_gpu(args):
    import torch

    import fp8_mqa_logits_02_gb300 as fm

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fm.lib()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make(wl)
    M, N, H, D = inp["M"], inp["N"], inp["H"], inp["D"]
    flops = valid_flops(inp)
    args_dev = _device_inputs(inp, dev)
    out = torch.empty((M, N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if ws > 1:
        torch.distributed.barrier()
    ms, clocks = time_calls(fm, args_dev, out, args.clean, args.split_n, args.steps,
                            args.warmup, flush, stream, dev)
    if ws > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(ms), ws)
    value = flops * args.steps * ws / (total_ms * 1e-3) / 1e12
    per_launch_s = statistics.mean(ms) * 1e-3

    # end to end through the host-buffer C entry point: pinned inputs copied in, the
    # kernel, and the whole logits matrix copied back, every step
    hq = torch.from_numpy(inp["q"]).pin_memory()
    hk = torch.from_numpy(inp["k"]).pin_memory()
    hkv = torch.from_numpy(inp["kv_scale"]).pin_memory()
    hw = torch.from_numpy(inp["w"]).pin_memory()
    hks = torch.from_numpy(inp["ks"]).pin_memory()
    hke = torch.from_numpy(inp["ke"]).pin_memory()
    hout = torch.empty((M, N), dtype=torch.float32).pin_memory()
    wsp = torch.empty(fm.host_workspace_bytes(M, N), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hkv, hw, hks, hke))
    if not args.clean:
        h2d += hout.numel() * 4  # with clean_logits = 0 the logits buffer goes in as well
    d2h = hout.numel() * 4

    def e2e_step():
        fm.fp8_mqa_logits_host(hq, hk, hkv, hw, hks, hke, hout, wsp,
                               clean_logits=bool(args.clean), split_n=args.split_n,
                               stream=stream)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    e2e_value = flops * e2e_steps * ws / (e2e_ms * 1e-3) / 1e12
    if fm.check_error(stream) != 0:
        raise RuntimeError("device status after e2e is not OK")
    del wsp, hout

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    achieved = flops / per_launch_s / 1e12
    traffic = committed_traffic("fp8_mqa_logits_kernel", wl.name, KERNEL_REV)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "us_per_call": 1e3 * total_ms / args.steps,
        "frac_of_fp8_peak": value / ws / fp8_peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3*fp8e4m3->f32", "data": "synthetic",
        "config": {"workload": wl.name, "M": M, "N": N, "H": H, "D": D,
                   "windows": workloads.describe(wl), "clean_logits": int(args.clean),
                   "split_n": args.split_n,
                   "split_used": args.split_n or fm.default_split(M, N, sm_count),
                   "valid_flops_per_call": flops,
                   "l2": f"flushed before every timed call ({FLUSH_BYTES >> 20} MiB write)",
                   "timing": "CUDA events per call on the launching stream"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": achieved / fp8_peak, "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16:g} "
                                    "(nominal fp8/bf16 ratio)",
                     "kernel": "fp8_mqa_logits_kernel", "kernel_rev": KERNEL_REV},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "entry": "fp8_mqa_logits_host (pinned host buffers)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if ws == 1 and not args.no_workloads and args.clean:
        # the headline's logits (the last timed call's, -inf outside the windows) feed the top-k
        line["topk"] = topk_block(fm, dev, stream, flush, out, inp, wl.name, min(args.steps, 20),
                                  args.warmup, peaks["hbm_gbs"])
    if ws == 1 and not args.no_workloads:
        line["workloads"] = workload_block(fm, dev, stream, flush, min(args.steps, 20),
                                           args.warmup, fp8_peak, peaks["hbm_gbs"], sm_count)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.default_threads()
        cb = cpu_oracle_sample(inp, args.reference_rows, threads)
        line["cpu_baseline"] = {
            "value": cb["tflops"], "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{cb['rows']} query rows (every {cb['stride']}th) of {wl.name}, "
                      f"fp64 C oracle, {cb['seconds']:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def time_topk(fm, logits, k, steps, warmup, flush, stream, dev, win):
    """Mean device time (ms) of `steps` fm.topk calls on `logits`, each after an L2 flush, CUDA
    events on the launching stream; plus the clocks sampled meanwhile."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fm.topk(logits, k, stream=stream, **win)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(dev.index) as clocks:
        host_lead(stream)
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            fm.topk(logits, k, stream=stream, **win)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    return statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)), clocks.summary()


def topk_block(fm, dev, stream, flush, logits, inp, wl_name, steps, warmup, hbm_peak):
    """The per-row top-k over the headline call's logits, at k = 512 and 2048, timed like
    the headline: the indexer's consumer, so that its numbers are in the default line."""
    M, N = inp["M"], inp["N"]
    block = []
    for k in TOPK_DEFAULT_KS:
        ms, clocks = time_topk(fm, logits, k, steps, warmup, flush, stream, dev, {})
        ms_unsorted, _ = time_topk(fm, logits, k, steps, warmup, flush, stream, dev,
                                   {"sorted": False})
        gbs = (M * N * 4 + M * k * 8) / (ms * 1e-3) / 1e9
        kernel = topk_kernel_name(N, k)
        block.append({"workload": wl_name, "k": k, "us_per_call": ms * 1e3, "gbs": gbs,
                      "frac_of_hbm": gbs / hbm_peak, "kernel": kernel, "kernel_rev": TOPK_REV,
                      "traffic": committed_traffic(kernel, wl_name, TOPK_REV, k),
                      "unsorted_us_per_call": ms_unsorted * 1e3,
                      "steps": steps, "clocks": clocks})
    return block


def run_topk(args):
    """Time fp8_mqa_topk on the logits of a workload: one step is the top-k of every row."""
    import torch

    import fp8_mqa_logits_02_gb300 as fm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make(wl)
    M, N = inp["M"], inp["N"]
    t = {key: torch.from_numpy(inp[key]).to(dev) for key in ("q", "k", "kv_scale", "w", "ks", "ke")}
    largs = (t["q"].view(torch.float8_e4m3fn), t["k"].view(torch.float8_e4m3fn), t["kv_scale"],
             t["w"], t["ks"], t["ke"])
    # --windowed: the logits without the -inf fill, and the top-k restricted to the windows
    logits = fm.fp8_mqa_logits(*largs, clean_logits=not args.windowed)
    win = {"ks": t["ks"], "ke": t["ke"]} if args.windowed else {}
    if args.unsorted:
        win["sorted"] = False
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ms, clock_summary = time_topk(fm, logits, args.topk, args.steps, args.warmup, flush, stream,
                                  dev, win)
    # bytes the call must move: the whole matrix, or only the windows when the top-k is windowed
    read_elems = workloads.valid_pairs(inp["ks"], inp["ke"], N) if args.windowed else M * N
    algo_bytes = read_elems * 4 + M * args.topk * 8
    peaks = load_peaks()
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    kernel = topk_kernel_name(N, args.topk)

    # the indexer step as a whole, cold: logits then top-k, in both forms
    def pipeline(clean):
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
        kw = {} if clean else {"ks": t["ks"], "ke": t["ke"]}
        def step():
            fm.fp8_mqa_logits(*largs, out=out, clean_logits=clean, stream=stream)
            fm.topk(out, args.topk, stream=stream, sorted=not args.unsorted, **kw)
        for _ in range(args.warmup):
            flush.zero_()
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        host_lead(stream)
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev)

    pipe = {"clean_logits_then_topk_us": pipeline(True),
            "unclean_logits_then_windowed_topk_us": pipeline(False)}
    print(json.dumps({
        "metric": "per-row top-k over the logits, GB/s of algorithmic traffic",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "us_per_call": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "M": M, "N": N, "k": args.topk,
                   "windowed": bool(args.windowed), "sorted": not args.unsorted,
                   "read_bytes": "windows only (clean_logits=0 logits)" if args.windowed
                   else "the whole matrix (clean_logits=1 logits)",
                   "l2": f"flushed before every timed call ({FLUSH_BYTES >> 20} MiB write)"},
        "pipeline": pipe,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None if args.windowed
                     else committed_traffic(kernel, wl.name, TOPK_REV, args.topk),
                     "peak_source": f"{peaks['source']} copy bandwidth",
                     "kernel": kernel, "kernel_rev": TOPK_REV},
        "gpu_launches": args.steps, "clocks": clock_summary,
    }), flush=True)
    return 0


def run_split_sweep(args):
    """Time the workload at each explicit split_n of --sweep-split and at the default
    (split_n = 0): one JSON line with the table and the default's distance from the best."""
    import torch

    import fp8_mqa_logits_02_gb300 as fm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fm.lib()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make(wl)
    args_dev = _device_inputs(inp, dev)
    out = torch.empty((inp["M"], inp["N"]), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = valid_flops(inp)
    default = fm.default_split(inp["M"], inp["N"], sm_count)
    table = []
    for split_n in [0] + [int(x) for x in args.sweep_split.split(",")]:
        ms, clocks = time_calls(fm, args_dev, out, args.clean, split_n, args.steps,
                                args.warmup, flush, stream, dev)
        us = statistics.mean(ms) * 1e3
        table.append({"split_n": split_n, "split_used": split_n or default, "us_per_call": us,
                      "tflops": flops / us / 1e6,
                      "sm_mhz": clocks["sm_mhz"] if clocks else None})
    best = min(table[1:], key=lambda r: r["us_per_call"])
    print(json.dumps({
        "metric": "split_n sweep, µs per call", "workload": wl.name,
        "windows": workloads.describe(wl), "clean_logits": args.clean, "steps": args.steps,
        "default_split": default, "default_us": table[0]["us_per_call"],
        "best_explicit": best["split_n"], "best_us": best["us_per_call"],
        "default_over_best": table[0]["us_per_call"] / best["us_per_call"],
        "table": table}), flush=True)
    return 0


def run_family_sweep(args):
    """Time every window family at the workload's shape (the page's op-test families), with
    the computed key tiles and valid pairs of each, so that the cost of rows that share a
    block with longer rows (time follows the block's window union) shows."""
    import torch

    import fp8_mqa_logits_02_gb300 as fm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fm.lib()
    wl = workloads.WORKLOADS[args.workload]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    q, k, kv, w = workloads.draw(wl.M, wl.N, wl.seed)
    out = torch.empty((wl.M, wl.N), dtype=torch.float32, device=dev)
    rows = []
    for fam in workloads.WINDOW_FAMILIES:
        ks, ke = workloads.windows(fam, wl.M, wl.N, wl.requests if wl.requests > 1 else 4)
        inp = {"q": q, "k": k, "kv_scale": kv, "w": w, "ks": ks, "ke": ke, "M": wl.M,
               "N": wl.N, "H": wl.H, "D": wl.D}
        args_dev = _device_inputs(inp, dev)
        ms, clocks = time_calls(fm, args_dev, out, args.clean, args.split_n, args.steps,
                                args.warmup, flush, stream, dev)
        pairs = workloads.valid_pairs(ks, ke, wl.N)
        # key tiles the kernel computes: per 8-row block, the tiles meeting its window union
        lo = np.clip(ks.astype(np.int64), 0, wl.N)
        hi = np.clip(ke.astype(np.int64), 0, wl.N)
        tiles = 0
        for b in range(0, wl.M, 8):
            l, h = lo[b:b + 8], hi[b:b + 8]
            live = h > l
            if live.any():
                tiles += int(-(-h[live].max() // 128) - l[live].min() // 128)
        us = statistics.mean(ms) * 1e3
        rows.append({"family": fam, "us_per_call": us, "valid_pairs": pairs,
                     "computed_pairs": tiles * 128 * 8,
                     "valid_fraction_of_computed": pairs / max(1, tiles * 128 * 8),
                     "ns_per_valid_kpair": us * 1e6 / max(1, pairs),
                     "ns_per_computed_kpair": us * 1e6 / max(1, tiles * 128 * 8),
                     "sm_mhz": clocks["sm_mhz"] if clocks else None})
    print(json.dumps({"metric": "window families at one shape, µs per call",
                      "shape": f"{wl.M}x{wl.N}", "clean_logits": args.clean,
                      "steps": args.steps, "table": rows}), flush=True)
    return 0


# Revision tags of the kernels the committed ncu traffic figures were taken on.
KERNEL_REV = "v7"
TOPK_REV = "t13"
TOPK_DEFAULT_KS = (512, 2048)  # the top-k sizes the default line times


def committed_traffic(kernel, workload, rev, k=None):
    """dram read + write bytes per launch from profiles/traffic.json for this kernel, workload,
    revision (and k), else None: a figure taken on another revision is not reported."""
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        entries = json.load(open(tpath))
    except (OSError, ValueError):
        return None
    for e in entries if isinstance(entries, list) else [entries]:
        if (e.get("kernel", "fp8_mqa_logits_kernel") == kernel and e.get("workload") == workload
                and e.get("kernel_rev") == rev and e.get("k") == k):
            return e.get("bytes_per_launch")
    return None


def topk_kernel_name(N, k):
    """The kernel fp8_mqa_topk launches for rows of N keys and this k."""
    if N <= 8192 and k <= 1024:
        return "topk_reg_kernel"
    if N <= 65536 and k <= 512:
        return "topk_kernel<TopkSmemPair>"
    if N <= 32768:
        return "topk_kernel<TopkSmemPairWide>"
    return "topk_kernel<TopkSmemOne>"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--clean", type=int, default=1, choices=(0, 1))
    ap.add_argument("--split-n", type=int, default=0)
    ap.add_argument("--impl", default="native", choices=("native", "reference"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload block (the headline call only)")
    ap.add_argument("--topk", type=int, default=0,
                    help="time the per-row top-k (this k) over the workload's logits instead")
    ap.add_argument("--windowed", action="store_true",
                    help="with --topk: the windowed top-k over clean_logits=0 logits")
    ap.add_argument("--unsorted", action="store_true",
                    help="with --topk: each row's entries in selection order (no sort)")
    ap.add_argument("--family-sweep", action="store_true",
                    help="time every window family at the workload's shape instead")
    ap.add_argument("--sweep-split", default="",
                    help="comma-separated split_n values: time each (and the default) instead")
    ap.add_argument("--reference-rows", type=int, default=4096,
                    help="query rows of the workload the CPU-baseline sample computes")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    args = parse_args(argv)
    if args.gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    ws, _, _ = dist_env()
    if "WORLD_SIZE" in os.environ:
        if ws != args.gpus:
            raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={ws}: launch one rank per GPU")
    elif args.gpus > 1:
        # replicas: one rank per GPU, each running the same full call
        return subprocess.call(replica_command(args.gpus, argv))
    if args.impl == "reference":
        return run_reference(args)
    if args.topk:
        return run_topk(args)
    if args.sweep_split:
        return run_split_sweep(args)
    if args.family_sweep:
        return run_family_sweep(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: exact attention forward on the GPT-2-medium-shaped prefill, plus split-KV decode.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = the whole forward path over one batch: fa_fwd non-causal and fa_fwd causal on
B=64, H=16, N=Nk=1024, d=dv=64 (bf16 inputs iid N(0,1), seed 0; bf16 O and fp32 LSE).
FLOPs follow the pages' count, 4*N*Nk*d per head (2*N*Nk*d for Q K^T plus 2*N*Nk*dv for
P V), halved for causal.  Inputs (403 MB) are larger than the 129 MB L2, so no flush is
needed between iterations.  The split-KV decode (B=16, H=32, d=128, lengths uniform in
[1024, 32768], 4.4 GB of K/V read per call) is timed in the same run and reported under
"decode" in GB/s of algorithmic K/V bytes.

Timing: W untimed warm-up steps, then exactly K steps launched back to back between two
CUDA events on the launching stream, with a barrier and a device synchronisation on both
sides, max over ranks (`value`, `ms_per_step`).  A second pass of K steps records an event
between the two calls of every step for the per-kernel times (`kernels`, `roofline`); the
events serialise the kernels, so that pass's steps are slightly longer.  SM clocks and
throttle reasons are sampled with nvidia-smi during both passes.  Under torchrun every rank runs the same per-GPU work on its own
GPU (replicas: the path has no data exchange), so scaling is weak.

--impl reference times the CPU FP64 oracle on the host cores instead (each step a bounded
sample of two (b, h) slices in each causal mode of the same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fa_inputs import attention_inputs, decode_inputs, gqa_decode_inputs, grad_output, sample_slices  # noqa: E402

METRIC = "attention fwd TFLOP/s (% of BF16 peak); decode KV GB/s (% of HBM peak)"
UNIT = "TFLOP/s"
FWD = dict(B=64, H=16, N=1024, Nk=1024, d=64)
DEC = dict(B=16, H=32, Nk_max=32768, d=128, lo=1024, hi=32768)
WORKLOAD = "GPT-2-medium-shaped prefill B=64 H=16 N=Nk=1024 d=dv=64, fa_fwd non-causal + causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of the dominant kernel from one ncu capture, keyed by
# the SHA-256 of the kernel code it was taken on (comments excluded); reported only while the
# code is unchanged.
KERNEL_TRAFFIC = {
    # profiles/fa_fwd_kernel_d64_gpt2medium_prefill.md: non-causal launch, 402.83 MB read + 110.14 MB written
    "4688c1bddd942f36e123d6b798eb987b8ded2daa60f131211566712ca0c85b13": 512.97e6,
}


def fwd_flops(B, H, N, Nk, d, causal):
    f = 4.0 * N * Nk * d * B * H
    return f / 2 if causal else f


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash():
    """SHA-256 of the forward kernel's code with comments and blank lines removed, so that an
    edit to comments alone keeps a traffic capture valid while any change to code drops it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("fa_fwd_kernel.cuh", "fa_kernel_common.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "exact_tiled_attention_fa_gb300", "csrc", name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------------------------
def oracle_sample(slices_per_mode, seed=0):
    """Time the FP64 oracle on (b, h) slices of the forward workload, both causal modes.

    Returns (seconds, flops, threads, description)."""
    import oracle
    oracle.build()
    B, H, N, Nk, d = FWD["B"], FWD["H"], FWD["N"], FWD["Nk"], FWD["d"]
    g = torch.Generator().manual_seed(seed)
    picks = sample_slices(B * H, slices_per_mode, seed=1)
    # only the picked heads are generated (same per-head distribution as the full batch)
    q = torch.randn((len(picks), N, d), generator=g).to(torch.bfloat16)
    k = torch.randn((len(picks), Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((len(picks), Nk, d), generator=g).to(torch.bfloat16)
    threads = oracle.cores()
    t0 = time.perf_counter()
    for causal in (False, True):
        oracle.attention(q, k, v, causal=causal, scale=1 / math.sqrt(d), threads=threads)
    dt = time.perf_counter() - t0
    flops = len(picks) * (fwd_flops(1, 1, N, Nk, d, False) + fwd_flops(1, 1, N, Nk, d, True))
    desc = (f"{len(picks)} (b,h) slices of N=Nk=1024 d=64, non-causal + causal each, "
            f"FP64 C oracle on {threads} threads")
    return dt, flops, threads, desc


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    per_step = 2
    for _ in range(args.warmup):
        oracle_sample(per_step)
    total_t, total_f, threads, desc = 0.0, 0.0, 1, ""
    for _ in range(args.steps):
        dt, fl, threads, desc = oracle_sample(per_step)
        total_t += dt
        total_f += fl
    value = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + " (bounded sample per step)", "sample_per_step": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import exact_tiled_attention_fa_gb300 as fa
    fa.library()  # fails loudly if the CUDA library is not built
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    if args.decode_only:
        decode = run_decode(fa, dev, stream, args, world, rank)
        gqa = [run_decode_gqa(fa, dev, stream, args, world, Hkv=h) for h in (8, 4)]
        pre = run_splitkv_prefill(fa, dev, stream, args, world)
        if rank == 0:
            print(json.dumps({"decode": decode, "decode_gqa": gqa, "splitkv_prefill": pre}), flush=True)
        return 0
    if args.splitkv_only:
        pre = run_splitkv_prefill(fa, dev, stream, args, world)
        if rank == 0:
            print(json.dumps({"splitkv_prefill": pre}), flush=True)
        return 0
    if args.bwd_only:
        backward = run_bwd(fa, dev, stream, args, world)
        if rank == 0:
            print(json.dumps({"backward": backward}), flush=True)
        return 0
    B, H, N, Nk, d = FWD["B"], FWD["H"], FWD["N"], FWD["Nk"], FWD["d"]
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=rank, device=dev)
    o_nc = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    o_c = torch.empty_like(o_nc)
    l_nc = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    l_c = torch.empty_like(l_nc)
    scale = 1.0 / math.sqrt(d)
    f_nc, f_c = fwd_flops(B, H, N, Nk, d, False), fwd_flops(B, H, N, Nk, d, True)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fwd(q, k, v, causal=False, scale=scale, out=o_nc, lse=l_nc)
        if ev is not None:
            ev[1].record(stream)
            ev[2].record(stream)
        fa.fwd(q, k, v, causal=True, scale=scale, out=o_c, lse=l_c)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert fa.get_device_error(dev) == fa.FA_OK
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    # Kernel breakdown: the same K steps again with an event recorded between the two calls.  An
    # event between two kernels serialises them (the second no longer starts its setup during the
    # first one's tail), so these steps take a little longer than the back-to-back ones above.
    b_start, b_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    b_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    breakdown_ms = b_start.elapsed_time(b_end)
    nc_all = [e[0].elapsed_time(e[1]) for e in evs]
    c_all = [e[2].elapsed_time(e[3]) for e in evs]
    nc_ms, c_ms = statistics.mean(nc_all), statistics.mean(c_all)
    assert fa.get_device_error(dev) == fa.FA_OK
    value = world * args.steps * (f_nc + f_c) / (total_ms / 1e3) / 1e12

    # ---- end to end through the public API: pinned host inputs in, O and LSE back to the host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(fa, dev, stream, args, world, (q, k, v), (o_nc, o_c, l_nc, l_c), scale, f_nc + f_c)

    # ---- split-KV decode in the same run
    decode = None
    hbm = measure_hbm_peaks(dev, stream)
    if not args.no_decode:
        decode = run_decode(fa, dev, stream, args, world, rank, hbm)

    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])
    achieved = f_nc / (nc_ms / 1e3) / 1e12
    src_hash = kernel_source_hash()
    traffic = KERNEL_TRAFFIC.get(src_hash)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "Nk": Nk, "d": d, "dv": d, "o_dtype": "bf16",
                   "flops_per_step": f_nc + f_c, "l2": "inputs 403 MB > 129 MB L2 (no flush needed)",
                   "parallelism": f"replicas x{world}"},
        "kernels": {
            "pass": f"{args.steps} more steps with an event between the two calls, "
                    f"{breakdown_ms / args.steps:.4f} ms per step (events serialise the launches)",
            "fa_fwd non-causal": {"ms": nc_ms, "tflops": achieved, "frac_of_peak": achieved / peak,
                                  "timing": {"ms_median": statistics.median(nc_all), "ms_min": min(nc_all),
                                             "ms_max": max(nc_all), "calls": len(nc_all)}},
            "fa_fwd causal": {"ms": c_ms, "tflops": f_c / (c_ms / 1e3) / 1e12,
                              "frac_of_peak": f_c / (c_ms / 1e3) / 1e12 / peak,
                              "timing": {"ms_median": statistics.median(c_all), "ms_min": min(c_all),
                                         "ms_max": max(c_all), "calls": len(c_all)}},
        },
        "roofline": {"kernel": "fa_fwd_kernel<64, non-causal, bf16>", "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{pk_src} bf16_tflops (burst; kernel timed in short launches)",
                     "algorithmic_flops_per_launch": f_nc},
        "e2e": e2e,
        "hbm_peaks_live": hbm,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if decode is not None:
        line["decode"] = decode
        line["decode_gqa"] = [run_decode_gqa(fa, dev, stream, args, world, Hkv=h) for h in (8, 4)]
        line["splitkv_prefill"] = run_splitkv_prefill(fa, dev, stream, args, world)
    if not args.no_extra:
        line["other_fwd_configs"] = run_other_fwd(fa, dev, stream, args, world, rank)
    if not args.no_bwd:
        line["backward"] = run_bwd(fa, dev, stream, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, threads, desc = oracle_sample(args.cpu_slices)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_e2e(fa, dev, stream, args, world, inputs, outputs, scale, flops_per_step, chunks=8):
    """The headline step end to end: every step copies its Q, K, V from pinned host memory,
    runs both forward calls and copies O and LSE back.  The batch is cut into `chunks` pieces
    and three streams (copy in, compute, copy out) joined by events overlap the copies of one
    piece with the kernels of another (host->device and device->host use separate copy
    engines).  Device buffers are reused across steps: a piece's inputs are overwritten only
    after the previous step's kernels read them, its outputs only after they were copied out."""
    q, k, v = inputs
    o_nc, o_c, l_nc, l_c = outputs
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho_nc, ho_c = (torch.empty(o_nc.shape, dtype=o_nc.dtype).pin_memory() for _ in range(2))
    hl_nc, hl_c = (torch.empty(l_nc.shape, dtype=l_nc.dtype).pin_memory() for _ in range(2))
    dq, dk, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B = q.shape[0]
    bounds = [B * c // chunks for c in range(chunks + 1)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream
    ev = lambda: torch.cuda.Event()  # noqa: E731
    copied_in = [ev() for _ in range(chunks)]
    computed = [ev() for _ in range(chunks)]
    copied_out = [ev() for _ in range(chunks)]
    started = [False] * chunks

    def e2e_step():
        for c in range(chunks):
            a_, b_ = bounds[c], bounds[c + 1]
            with torch.cuda.stream(s_in):
                if started[c]:
                    s_in.wait_event(computed[c])  # the previous step's kernels have read this piece
                dq[a_:b_].copy_(hq[a_:b_], non_blocking=True)
                dk[a_:b_].copy_(hk[a_:b_], non_blocking=True)
                dv_[a_:b_].copy_(hv[a_:b_], non_blocking=True)
                copied_in[c].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(copied_in[c])
                if started[c]:
                    s_cmp.wait_event(copied_out[c])  # the previous step's outputs have left
                fa.fwd(dq[a_:b_], dk[a_:b_], dv_[a_:b_], causal=False, scale=scale, out=o_nc[a_:b_], lse=l_nc[a_:b_])
                fa.fwd(dq[a_:b_], dk[a_:b_], dv_[a_:b_], causal=True, scale=scale, out=o_c[a_:b_], lse=l_c[a_:b_])
                computed[c].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[c])
                ho_nc[a_:b_].copy_(o_nc[a_:b_], non_blocking=True)
                hl_nc[a_:b_].copy_(l_nc[a_:b_], non_blocking=True)
                ho_c[a_:b_].copy_(o_c[a_:b_], non_blocking=True)
                hl_c[a_:b_].copy_(l_c[a_:b_], non_blocking=True)
                copied_out[c].record(s_out)
            started[c] = True

    for _ in range(args.warmup):
        e2e_step()
    n_e2e = args.steps
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    torch.cuda.synchronize(dev)  # every copy out of the last step has landed in host memory
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world)
    barrier(world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(t.numel() * t.element_size() for t in (ho_nc, ho_c, hl_nc, hl_c))
    e2e_value = world * n_e2e * flops_per_step / (e2e_ms / 1e3) / 1e12
    ok = torch.equal(ho_c.to(dev), o_c) and torch.equal(hl_nc.to(dev), l_nc)  # results made it back
    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": e2e_ms / n_e2e, "pipeline": f"{chunks} batch pieces, copy-in / compute / copy-out streams",
            "timer": "host wall clock around the steps, synchronised on both sides", "results_returned": ok}


# The other forward configurations of the parity suite, timed the same way (not the headline):
# (name, B, H, N, Nk, d, input multiplier, causal, oracle sample: heads, query rows or None for all)
OTHER_FWD = (
    ("single head 256x256 d=64", 1, 1, 256, 256, 64, 1.0, False, 1, None),
    ("single head 256x256 d=64 causal", 1, 1, 256, 256, 64, 1.0, True, 1, None),
    ("ragged 4097 d=128 x2", 4, 16, 4097, 4097, 128, 2.0, False, 4, None),
    ("ragged 4097 d=128 x2 causal", 4, 16, 4097, 4097, 128, 2.0, True, 4, None),
    ("ragged 77x513 d=32 x2", 8, 8, 77, 513, 32, 2.0, False, 64, None),
    ("ragged 77x513 d=32 x2 causal", 8, 8, 77, 513, 32, 2.0, True, 64, None),
    ("long causal 16384 d=128", 2, 32, 16384, 16384, 128, 1.0, True, 4, (0, 2048)),
)


def visible_pairs(N, Nk, causal, r0=0, r1=None):
    """(query, key) pairs that attend: all of them without a mask; with one, query i (position
    Nk - N + i) sees keys 0 .. Nk - N + i."""
    r1 = N if r1 is None else r1
    if not causal:
        return (r1 - r0) * Nk
    off = Nk - N
    return sum(min(Nk, max(0, off + i + 1)) for i in range(r0, r1))


# --quick (for profiler launch lists): short timing blocks.  Set by main().
QUICK = {"on": False}


def time_stats(call, dev, stream, world, warmup=3, min_calls=100, min_s=0.5, blocks=5, max_block=10000):
    """Milliseconds per call from `blocks` blocks of back-to-back calls, each block timed with
    CUDA events on `stream`; blocks are sized so that together they make at least `min_calls`
    calls and last at least `min_s` seconds.  Returns the median, min and max block (max over
    ranks) and the number of timed calls."""
    if QUICK["on"]:
        warmup, min_calls, min_s, blocks = 1, 2, 0.0, 2
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(3):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est = max(e0.elapsed_time(e1) / 3, 1e-4)
    per_block = max(math.ceil(min_calls / blocks), math.ceil(min_s * 1e3 / blocks / est))
    per_block = min(per_block, max_block)
    times = []
    for _ in range(blocks):
        e0.record(stream)
        for _ in range(per_block):
            call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(max_over_ranks(e0.elapsed_time(e1) / per_block, world))
    return {"ms": statistics.median(times), "ms_min": min(times), "ms_max": max(times), "calls": per_block * blocks}


def oracle_fwd_sample(B, H, N, Nk, d, mult, causal, heads, rows, seed=0):
    """Time the FP64 C oracle on `heads` of the B*H heads (inputs drawn on the host from the
    workload's distribution) over query rows `rows` (all when None).  Returns a cpu_baseline dict
    with the sample's time and TFLOP/s and the time of the full configuration extrapolated by
    FLOPs (labelled as such)."""
    import oracle
    oracle.build()
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(shape, generator=g).to(torch.bfloat16) * mult
               for shape in ((heads, N, d), (heads, Nk, d), (heads, Nk, d)))
    threads = oracle.cores()
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=causal, scale=1 / math.sqrt(d), rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    r0, r1 = rows if rows is not None else (0, N)
    fl = 4.0 * d * heads * visible_pairs(N, Nk, causal, r0, r1)
    full = 4.0 * d * B * H * visible_pairs(N, Nk, causal)
    desc = f"{heads} of {B * H} heads" + (f", query rows {r0}..{r1 - 1}" if rows is not None else ", all rows")
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle", "seconds": dt,
            "sample": desc + f", FP64 C oracle on {threads} threads (visible-pair FLOPs)",
            "full_config_seconds_extrapolated": dt * full / fl}


def run_other_fwd(fa, dev, stream, args, world, rank):
    pk, _ = peaks()
    peak = float(pk["bf16_tflops"])
    out = {}
    for name, B, H, N, Nk, d, mult, causal, o_heads, o_rows in OTHER_FWD:
        q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, mult=mult, device=dev)
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        call = lambda: fa.fwd(q, k, v, causal=causal, out=o, lse=lse)  # noqa: E731
        st = time_stats(call, dev, stream, world, warmup=max(args.warmup, 3))
        fl = fwd_flops(B, H, N, Nk, d, causal)
        fl_exact = 4.0 * d * B * H * visible_pairs(N, Nk, causal)
        ms = st["ms"]
        rec = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12, "frac_of_peak": fl / (ms / 1e3) / 1e12 / peak,
               "flops": fl, "flops_exact_visible_pairs": fl_exact,
               "tflops_exact": fl_exact / (ms / 1e3) / 1e12, "timing": st}
        if ms < 0.05:  # launch-bound: also the per-call time with no host launch cost (CUDA graph of 20 calls)
            rec["graph_us_per_call"] = graph_us(call, dev, stream, world)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            rec["cpu_baseline"] = oracle_fwd_sample(B, H, N, Nk, d, mult, causal, o_heads, o_rows)
        out[name] = rec
        del q, k, v, o, lse
    assert fa.get_device_error(dev) == fa.FA_OK
    return out


def measure_hbm_peaks(dev, stream):
    """Live HBM denominators on this GPU: a device-to-device copy of 2 GiB (read + write bytes)
    and two read-dominated streams over a 4 GiB bf16 matrix (cuBLAS GEMV, which reads the matrix
    once, and a sum reduction); best of 10 each, CUDA events."""
    n = 1 << 30
    a = torch.empty(n, dtype=torch.bfloat16, device=dev).uniform_()
    b = torch.empty_like(a)
    A = torch.empty((1 << 16, 1 << 15), dtype=torch.bfloat16, device=dev).uniform_()
    x = torch.empty(1 << 15, dtype=torch.bfloat16, device=dev).uniform_()

    def best(fn, nbytes):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ms = []
        for _ in range(10):
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        return nbytes / (min(ms) / 1e3) / 1e9

    copy = best(lambda: b.copy_(a), 2 * a.numel() * 2)
    gemv = best(lambda: torch.mv(A, x), A.numel() * 2)
    red = best(lambda: A.view(torch.int64).max(), A.numel() * 2)
    del a, b, A, x
    torch.cuda.empty_cache()
    return {"copy_gbs": copy, "read_gemv_gbs": gemv, "read_max_gbs": red,
            "method": "best of 10 CUDA-event-timed launches: b.copy_(a) over 1 Gi bf16 (read + write bytes); "
                      "torch.mv of a [65536, 32768] bf16 matrix (cuBLAS GEMV) and the int64 max reduction of "
                      "the same 4 GiB (read only)"}


# DRAM peak that ncu's gpu__dram_throughput is a percentage of, on this GB300 pool: the decode
# capture in profiles/fa_decode_split_kernel_d128.md reads 6.76 TB/s at 85.4 % of it.
NCU_DRAM_PEAK_GBS = 6760.0 / 0.854


def bwd_flops(B, H, N, Nk, d, causal):
    """Five products of 2*N*Nk*d each per head (S, dP, dV, dK, dQ), halved for causal."""
    f = 10.0 * B * H * N * Nk * d
    return f / 2 if causal else f


def run_bwd(fa, dev, stream, args, world):
    """fa_bwd on the GPT-2-medium shape (dO given, O and LSE from fa_fwd), bf16 gradients."""
    B, H, N, Nk, d = FWD["B"], FWD["H"], FWD["N"], FWD["Nk"], FWD["d"]
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, device=dev)
    do = grad_output(B, H, N, d, seed=0, device=dev)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    grads = tuple(torch.empty((B, H, n, d), dtype=torch.bfloat16, device=dev) for n in (N, Nk, Nk))
    pk, src = peaks()
    peak = float(pk["bf16_tflops"])
    out = {"workload": f"backward B={B} H={H} N=Nk={N} d=dv={d}, bf16 dQ/dK/dV, 3 launches per call",
           "peak_source": f"{src} bf16_tflops"}
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal)
        barrier(world)
        st = time_stats(lambda: fa.bwd(q, k, v, o, lse, do, causal=causal, grads=grads, workspace=ws),
                        dev, stream, world, warmup=max(args.warmup, 3))
        ms = st["ms"]
        fl = bwd_flops(B, H, N, Nk, d, causal)
        tf = world * fl / (ms / 1e3) / 1e12
        out["causal" if causal else "non-causal"] = {"ms": ms, "tflops": tf, "frac_of_peak": tf / peak / world,
                                                     "flops": fl, "timing": st}
    assert fa.get_device_error(dev) == fa.FA_OK
    return out


def oracle_decode_all(q, k, v, lens):
    """Time the FP64 C oracle on every (sequence, head) of a decode batch: each sequence's valid
    cache prefix is copied to the host first (outside the timed region)."""
    import oracle
    oracle.build()
    threads = oracle.cores()
    dt, kv_bytes = 0.0, 0
    for b, n in enumerate(lens.tolist()):
        qb = q[b:b + 1].cpu()
        kb = k[b:b + 1, :, :n].contiguous().cpu()
        vb = v[b:b + 1, :, :n].contiguous().cpu()
        t0 = time.perf_counter()
        oracle.decode(qb, kb, vb, [n], threads=threads)
        dt += time.perf_counter() - t0
        kv_bytes += 2 * kb.numel() * 2
    return {"value": kv_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle", "seconds": dt,
            "sample": f"all {q.shape[0] * q.shape[1]} (sequence, head) pairs, FP64 C oracle on {threads} threads "
                      "(bf16 K/V bytes of the cached prefixes / time)"}


def run_decode(fa, dev, stream, args, world, rank=0, hbm=None):
    B, H, Nk_max, d = DEC["B"], DEC["H"], DEC["Nk_max"], DEC["d"]
    q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=0, lo=DEC["lo"], hi=DEC["hi"], device=dev)
    lens_d = lens.to(dev)
    n = fa.decode_default_splits(B, H, Nk_max, fa.num_sms(dev))
    ws = torch.empty(fa.decode_workspace_size(B, H, d, n), dtype=torch.uint8, device=dev)
    o = torch.empty((B, H, 1, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    barrier(world)
    st = time_stats(lambda: fa.decode_splitkv(q, k, v, lens_d, n_splits=n, out=o, lse=lse, workspace=ws),
                    dev, stream, world, warmup=max(args.warmup, 3))
    barrier(world)
    ms = st["ms"]
    assert fa.get_device_error(dev) == fa.FA_OK
    kv_bytes = sum(2 * H * int(n_b) * d * 2 for n_b in lens.tolist())
    other = B * H * (d * 2 + d * 2 + 4)
    pk, src = peaks()
    gbs = world * (kv_bytes + other) / (ms / 1e3) / 1e9
    # the same decode with the combine fused into the split kernel (one launch per call)
    wsf = fa.decode_fused_workspace(B, H, Nk_max, d, n_splits=n, device=dev)
    fused = lambda: fa.decode_splitkv_fused(q, k, v, lens_d, wsf, n_splits=n, out=o, lse=lse)  # noqa: E731
    st_f = time_stats(fused, dev, stream, world, warmup=max(args.warmup, 3))
    ms_f = st_f["ms"]
    # a short-context decode, where the second launch is a visible share of the call
    qs, ks, vs, ls = decode_inputs(1, 32, 2048, d, d, seed=1, lo=2048, hi=2048, device=dev)
    ls_d = ls.to(dev)
    os_ = torch.empty((1, 32, 1, d), dtype=torch.bfloat16, device=dev)
    ns = fa.decode_default_splits(1, 32, 2048, fa.num_sms(dev))
    ws2 = torch.empty(fa.decode_workspace_size(1, 32, d, ns), dtype=torch.uint8, device=dev)
    wsf2 = fa.decode_fused_workspace(1, 32, 2048, d, n_splits=ns, device=dev)
    two = lambda: fa.decode_splitkv(qs, ks, vs, ls_d, n_splits=ns, out=os_, workspace=ws2, return_lse=False)  # noqa: E731
    one = lambda: fa.decode_splitkv_fused(qs, ks, vs, ls_d, wsf2, n_splits=ns, out=os_, return_lse=False)  # noqa: E731
    short = {"workload": f"B=1 H=32 Nk=2048 d={d}", "n_splits": ns,
             "two_launches_us": 1e3 * time_stats(two, dev, stream, world)["ms"],
             "fused_us": 1e3 * time_stats(one, dev, stream, world)["ms"],
             # the same calls replayed from a CUDA graph of 20 calls: no per-call launch cost
             "graph_two_launches_us": graph_us(two, dev, stream, world),
             "graph_fused_us": graph_us(one, dev, stream, world)}
    assert fa.get_device_error(dev) == fa.FA_OK
    out = {"workload": "split-KV decode B=16 H=32 d=128, lengths U[1024,32768] (seed 0), bf16 O",
           "n_splits": n, "ms": ms, "timing": st, "gbs": gbs, "kv_bytes": kv_bytes,
           "frac_of_hbm": gbs / float(pk["hbm_gbs"]), "frac_of_8tbs": gbs / 8000.0, "peak_source": src,
           "launches_per_call": 2,
           "fused_combine": {"ms": ms_f, "timing": st_f, "gbs": world * (kv_bytes + other) / (ms_f / 1e3) / 1e9,
                             "launches_per_call": 1},
           "short_context": short}
    if hbm is not None:
        # against the larger of the live copy and read-stream bandwidths of this GPU
        read_peak = max(hbm["copy_gbs"], hbm["read_gemv_gbs"], hbm["read_max_gbs"])
        out["frac_of_live_read_peak"] = gbs / world / read_peak
        out["live_read_peak_gbs"] = read_peak
    # every library stream measured reads slower than this kernel, so the bound that holds is the
    # DRAM peak ncu reports throughput against
    out["frac_of_ncu_dram_peak"] = gbs / world / NCU_DRAM_PEAK_GBS
    if out["frac_of_ncu_dram_peak"] > 1.0:
        print(f"warning: decode at {out['frac_of_ncu_dram_peak']:.3f} of the DRAM peak: timing suspect", file=sys.stderr)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = oracle_decode_all(q, k, v, lens)
    return out


def graph_us(call, dev, stream, world, reps=20):
    """Microseconds per call with `reps` calls captured into one CUDA graph and the graph replayed
    (after one eager call on a side stream for the first-use set-up)."""
    if QUICK["on"]:
        return None
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            call()
    return 1e3 * time_calls(g.replay, dev, stream, 3, 10, world) / reps


def time_calls(call, dev, stream, warmup, steps, world):
    """Average milliseconds per call over `steps` calls, CUDA events on `stream`, max over ranks."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return max_over_ranks(e0.elapsed_time(e1), world) / steps


GQA = dict(B=16, Hq=32, Hkv=8, Nk_max=32768, d=128, lo=1024, hi=32768)


def run_decode_gqa(fa, dev, stream, args, world, Hkv=None):
    """Split-KV decode with grouped key/value heads (32 query heads over 8: Llama-style; over 4)."""
    B, Hq, Nk_max, d = GQA["B"], GQA["Hq"], GQA["Nk_max"], GQA["d"]
    Hkv = GQA["Hkv"] if Hkv is None else Hkv
    q, k, v, lens = gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, d, seed=0, lo=GQA["lo"], hi=GQA["hi"], device=dev)
    lens_d = lens.to(dev)
    n = 0  # the library's automatic split count
    n_auto = fa.decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, fa.num_sms(dev))
    ws = torch.empty(fa.decode_workspace_size(B, Hq, d, n_auto), dtype=torch.uint8, device=dev)
    o = torch.empty((B, Hq, 1, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=dev)
    barrier(world)
    st = time_stats(lambda: fa.decode_splitkv_gqa(q, k, v, lens_d, n_splits=n, out=o, lse=lse, workspace=ws),
                    dev, stream, world, warmup=max(args.warmup, 3))
    barrier(world)
    ms = st["ms"]
    assert fa.get_device_error(dev) == fa.FA_OK
    kv_bytes = sum(2 * Hkv * int(n_b) * d * 2 for n_b in lens.tolist())
    other = B * Hq * (d * 2 + d * 2 + 4)
    pk, src = peaks()
    gbs = world * (kv_bytes + other) / (ms / 1e3) / 1e9
    return {"workload": f"GQA split-KV decode B={B} Hq={Hq} Hkv={Hkv} d={d}, lengths U[1024,32768] (seed 0), bf16 O",
            "group": Hq // Hkv, "n_splits": n_auto, "timing": st, "unit": "CUDA cores" if Hq // Hkv in (1, 2) or (Hq // Hkv == 4 and d != 128) else "tensor core", "ms": ms, "gbs": gbs, "kv_bytes": kv_bytes, "frac_of_hbm": gbs / float(pk["hbm_gbs"]),
            "frac_of_8tbs": gbs / 8000.0, "peak_source": src, "launches_per_call": 2}


SPLIT_PREFILL = dict(B=1, H=8, N=512, Nk=32768, d=128)


def run_splitkv_prefill(fa, dev, stream, args, world):
    """Few query tiles over a long context (B=1 H=8 N=512 Nk=32K d=128, causal): fa_fwd keeps
    B*H*N/128 = 32 query tiles (16 CTAs); fa_fwd_splitkv splits the keys and merges."""
    B, H, N, Nk, d = (SPLIT_PREFILL[x] for x in ("B", "H", "N", "Nk", "d"))
    q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, device=dev)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    n = fa.fwd_splitkv_default_splits(B, H, N, Nk, fa.num_sms(dev))
    ws = torch.empty(fa.fwd_splitkv_workspace_size(B, H, N, d, n), dtype=torch.uint8, device=dev)
    # visible pairs: query i (position Nk - N + i) sees Nk - N + i + 1 keys
    fl = 4.0 * B * H * d * sum(Nk - N + i + 1 for i in range(N))
    out = {"workload": f"causal prefill B={B} H={H} N={N} Nk={Nk} d={d}, bf16 O", "flops_exact": fl, "n_splits": n}
    for name, call in (("fa_fwd", lambda: fa.fwd(q, k, v, causal=True, out=o, lse=lse)),
                       ("fa_fwd_splitkv", lambda: fa.fwd_splitkv(q, k, v, causal=True, n_splits=n, out=o, lse=lse,
                                                                 workspace=ws))):
        st = time_stats(call, dev, stream, world, warmup=max(args.warmup, 3))
        ms = st["ms"]
        out[name] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12, "timing": st}
    assert fa.get_device_error(dev) == fa.FA_OK
    return out


def _case_call(fa, dev, name):
    """(callable, description) for one named workload of the suite, inputs built on `dev`."""
    fwd_cases = {name: i for i, name in enumerate(("fwd-c1", "fwd-c1-causal", "fwd-c3a", "fwd-c3a-causal", "fwd-c3b",
                                                   "fwd-c3b-causal", "fwd-c4"))}
    if name in fwd_cases or name in ("fwd-c2", "fwd-c2-causal"):
        if name in fwd_cases:
            desc, B, H, N, Nk, d, mult, causal = OTHER_FWD[fwd_cases[name]][:8]
        else:
            B, H, N, Nk, d, mult, causal = FWD["B"], FWD["H"], FWD["N"], FWD["Nk"], FWD["d"], 1.0, name.endswith("causal")
            desc = WORKLOAD + (" causal" if causal else " non-causal")
        q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, mult=mult, device=dev)
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        return (lambda: fa.fwd(q, k, v, causal=causal, out=o, lse=lse)), desc
    if name in ("gqa4", "gqa8", "gqa16", "gqa32"):
        B, Hq, Nk_max, d = GQA["B"], GQA["Hq"], GQA["Nk_max"], GQA["d"]
        Hkv = Hq // int(name[3:])
        q, k, v, lens = gqa_decode_inputs(B, Hq, Hkv, Nk_max, d, d, seed=0, lo=GQA["lo"], hi=GQA["hi"], device=dev)
        lens_d = lens.to(dev)
        n = fa.decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, fa.num_sms(dev))
        ws = torch.empty(fa.decode_workspace_size(B, Hq, d, n), dtype=torch.uint8, device=dev)
        o = torch.empty((B, Hq, 1, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=dev)
        return (lambda: fa.decode_splitkv_gqa(q, k, v, lens_d, n_splits=n, out=o, lse=lse, workspace=ws),
                f"GQA decode B={B} Hq={Hq} Hkv={Hkv} d={d}")
    if name == "splitkv-prefill":
        B, H, N, Nk, d = (SPLIT_PREFILL[x] for x in ("B", "H", "N", "Nk", "d"))
        q, k, v = attention_inputs(B, H, N, Nk, d, d, seed=0, device=dev)
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        n = fa.fwd_splitkv_default_splits(B, H, N, Nk, fa.num_sms(dev))
        ws = torch.empty(fa.fwd_splitkv_workspace_size(B, H, N, d, n), dtype=torch.uint8, device=dev)
        return (lambda: fa.fwd_splitkv(q, k, v, causal=True, n_splits=n, out=o, lse=lse, workspace=ws),
                f"causal split-KV prefill B={B} H={H} N={N} Nk={Nk} d={d}")
    if name == "decode":
        B, H, Nk_max, d = DEC["B"], DEC["H"], DEC["Nk_max"], DEC["d"]
        q, k, v, lens = decode_inputs(B, H, Nk_max, d, d, seed=0, lo=DEC["lo"], hi=DEC["hi"], device=dev)
        lens_d = lens.to(dev)
        n = fa.decode_default_splits(B, H, Nk_max, fa.num_sms(dev))
        ws = torch.empty(fa.decode_workspace_size(B, H, d, n), dtype=torch.uint8, device=dev)
        o = torch.empty((B, H, 1, d), dtype=torch.bfloat16, device=dev)
        return (lambda: fa.decode_splitkv(q, k, v, lens_d, n_splits=n, out=o, workspace=ws, return_lse=False),
                f"split-KV decode B={B} H={H} d={d}")
    raise SystemExit(f"unknown --case {name}")


def run_case(args, local):
    """One workload alone, `warmup` untimed and `steps` timed calls (for profiling captures)."""
    import exact_tiled_attention_fa_gb300 as fa
    fa.library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    call, desc = _case_call(fa, dev, args.case)
    ms = time_calls(call, dev, stream, args.warmup, args.steps, 1)
    assert fa.get_device_error(dev) == fa.FA_OK
    print(json.dumps({"case": args.case, "workload": desc, "calls": args.steps, "ms_per_call": ms}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None,
                    help="run one workload alone (fwd-c1, fwd-c1-causal, fwd-c2, fwd-c2-causal, fwd-c3a, "
                         "fwd-c3a-causal, fwd-c3b, fwd-c3b-causal, fwd-c4, decode, gqa4, gqa8, gqa16, gqa32, splitkv-prefill) for profiling")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-decode", action="store_true", help="skip the split-KV decode measurement")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other forward configurations")
    ap.add_argument("--decode-only", action="store_true", help="only the split-KV decode (profiling)")
    ap.add_argument("--decode-batch", type=int, default=DEC["B"], help="decode batch (smaller cache for profiling)")
    ap.add_argument("--cpu-slices", type=int, default=1024)
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward measurement")
    ap.add_argument("--bwd-only", action="store_true", help="only the backward (profiling)")
    ap.add_argument("--splitkv-only", action="store_true", help="only the split-KV prefill workload (profiling)")
    ap.add_argument("--quick", action="store_true",
                    help="short timing blocks and no CPU baselines (for profiler launch lists; not a measurement)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup()
    DEC["B"] = args.decode_batch
    if args.quick:
        QUICK["on"] = True
        args.no_cpu_baseline = True
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.case:
        return run_case(args, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: affine group-64 quantized matmul y = x . W^T on GB300.

Default workload: the 4-bit decode GEMV (N=4096, K=4096, one bf16 activation
row).  One step is one call of the library (one pass of the hot path over one
activation batch).  The timed region holds exactly `--steps` calls, captured
in CUDA graphs and cycling through enough copies of the weights that their
total exceeds twice the L2 size (every call reads its weights from HBM).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|small|split3:I|layer:I|prefill:I|quantize:I|
                                layerstep:I|widths:I|attention:I] [--all]

widths:I times aq_matmul_ex on other code widths and group sizes;
attention:I times aq_attention_decode (decode attention over a quantised KV
cache).  layerstep:I times one decoder-layer step (seven projections; I = 0/1
fused or not at M = 1, 2/3 at M = 8).  quantize:I times the float -> affine
quantiser (aq_quantize) on the weight shapes of
workloads.QUANTIZE_WORKLOADS instead of the matmul.

The matmul workloads also carry `gpu_comparisons` (context, not targets):
torch.matmul (cuBLAS) on the weights dequantised once, and a torch-op
dequantise of the packed words followed by torch.matmul on every call
(--no-compare skips them).

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica on its own GPU ("replicas only": the method needs no
exchange between GPUs); the time is the maximum over ranks.

--impl reference times the fp64 C oracle on the host cores instead (the
reference arm of this method has no GPU implementation to run): each step is
a bounded sample of output columns of the same workload, scaled to the
metric's unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = ("µs/call and effective HBM GB/s (fraction of roofline), 3/4-bit group-64 "
          "y=x·Wᵀ, M=1..512")
DEFAULT_WORKLOAD = "decode"
GRAPH_CHUNK = 1024


def reduce_max(value: float, device: str = "cpu") -> float:
    """Maximum of `value` over all ranks (identity without a process group).
    Replicas share nothing but this: the job's time is its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(us_per_call_slowest_rank: float, world: int) -> float:
    """Time per call for the whole job: every rank ran the same number of
    calls concurrently, so the job completes world x calls in the slowest
    rank's time."""
    return us_per_call_slowest_rank / max(1, world)


def parse_workload(spec: str):
    name, _, idx = spec.partition(":")
    return name, int(idx or 0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def traffic_record(fname="traffic.txt"):
    """dram bytes per launch from a committed ncu summary, if the kernel
    source it was taken on is unchanged (source hash recorded beside it)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", fname)
    try:
        rec = {}
        for line in open(path):
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                rec[k.strip()] = v.strip()
    except OSError:
        return {}
    src = os.path.join(ROOT, "quantized_matmul_affine_gb300", "csrc")
    h = hashlib.sha256()
    # the files that define the kernel (all kernel sources if not listed)
    names = [n.strip() for n in rec.get("sources", "").split(",") if n.strip()]
    if not names:
        names = [fn for fn in sorted(os.listdir(src)) if fn.endswith((".cu", ".cuh", ".h"))]
    for fn in names:
        try:
            h.update(open(os.path.join(src, fn), "rb").read())
        except OSError:
            return {}
    if rec.get("csrc_sha256") != h.hexdigest():
        return {}
    return rec


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0, t1 = (self.marks + [0, 0])[:2] if len(self.marks) >= 2 else (0, time.time())
        inside, near = [], []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            near.append(parts)
            if t0 <= ts <= t1 + 0.2:
                inside.append(parts)
        use = inside or near[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(p[1]) for p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(
                    (float(p[3]) for p in use if p[3].replace(".", "").isdigit()), default=None)}


def device_problem(p, copies, torch, aq):
    """Pack the weights on the device and replicate them `copies` times."""
    codes = torch.from_numpy(p.codes).cuda()
    Wq = aq.aq_pack(codes, p.bits)
    del codes
    s = torch.from_numpy(p.scales).cuda()
    b = torch.from_numpy(p.biases).cuda()
    xt = torch.from_numpy(p.x_bits.view(np.int16)).cuda()
    x = xt.view(torch.bfloat16 if p.x_dtype == "bf16" else torch.float16)
    ws = [(Wq, s, b)] + [(Wq.clone(), s.clone(), b.clone()) for _ in range(copies - 1)]
    return x, ws


def gpu_comparisons(p, ws, x, torch, l2, stream):
    """Context, not targets: (1) torch.matmul (cuBLAS) on the weights
    dequantised once to x's dtype; (2) "expand": dequantise the packed words
    with torch ops on every call, then torch.matmul (4-bit only).  Both
    cold-L2 over rotating copies, CUDA events around CUDA-graph replays."""
    dt = x.dtype
    G = p.K // 64
    s0 = ws[0][1].float().view(p.N, G, 1)
    b0 = ws[0][2].float().view(p.N, G, 1)
    codes = torch.from_numpy(p.codes).cuda().float().view(p.N, G, 64)
    w0 = (codes * s0 + b0).view(p.N, p.K).to(dt)
    del codes
    dbytes = p.N * p.K * 2
    dcopies = max(2, -(-2 * l2 // dbytes) + 1)
    dense = [w0] + [w0.clone() for _ in range(dcopies - 1)]
    shifts = torch.arange(0, 32, 4, device="cuda", dtype=torch.int32)

    def expand(c):
        Wq, sc, bi = ws[c % len(ws)]
        q = (Wq.view(torch.int32).view(p.N, p.K // 8, 1) >> shifts) & 15
        w = q.view(p.N, G, 64).to(dt) * sc.view(p.N, G, 1).to(dt) + bi.view(p.N, G, 1).to(dt)
        return torch.matmul(x, w.view(p.N, p.K).t())

    def timed(body, calls=128):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            body(0)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(calls):
                    body(i)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(4):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (4 * calls)

    out = {"dense_matmul_us": round(timed(lambda i: torch.matmul(x, dense[i % dcopies].t())), 3),
           "expand_then_matmul_us": round(timed(expand), 3) if p.bits == 4 else None,
           "note": "context only: torch.matmul (cuBLAS) on weights dequantised once to "
                   f"{'bf16' if dt == torch.bfloat16 else 'fp16'} ({dcopies} copies, cold L2); "
                   "expand = torch-op dequantise of the packed words every call, then "
                   "torch.matmul"}
    del dense, w0
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import quantized_matmul_affine_gb300 as aq

    torch.cuda.set_device(local_rank)
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    name, idx = parse_workload(args.workload)
    p = workloads.workload(name, idx)
    bytes_call = workloads.algorithmic_bytes(p.M, p.N, p.K, p.bits)
    flops_call = workloads.flops(p.M, p.N, p.K)
    wbytes = p.N * p.K * p.bits // 8 + 4 * p.N * p.G
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    copies = max(2, -(-2 * l2 // wbytes) + 1)
    x, ws = device_problem(p, copies, torch, aq)
    fn = aq.aq_matmul_bf16 if p.x_dtype == "bf16" else aq.aq_matmul
    ys = [torch.empty((p.M, p.N), dtype=x.dtype, device="cuda") for _ in range(copies)]
    variant = aq.aq_select(p.M, p.N, p.K, p.bits, aq.AQ_BF16 if p.x_dtype == "bf16" else aq.AQ_F16)
    stream = torch.cuda.Stream()

    def capture(ncalls, start):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(ncalls):
                    c = (start + i) % copies
                    Wq, s, b = ws[c]
                    fn(x, Wq, s, b, p.bits, out=ys[c], stream=stream)
        return g

    # eager sanity call, then graphs: full chunks plus a remainder
    with torch.cuda.stream(stream):
        fn(x, *ws[0], p.bits, out=ys[0], stream=stream)
    torch.cuda.synchronize()
    chunk = min(GRAPH_CHUNK, max(1, args.steps))
    g_chunk = capture(chunk, 0)
    rem = args.steps % chunk
    g_rem = capture(rem, 0) if rem else None
    warm_chunk = min(chunk, max(1, args.warmup))
    g_warm = capture(warm_chunk, 0)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        done = 0
        while done < args.warmup:
            g_warm.replay()
            done += warm_chunk
    torch.cuda.synchronize()

    sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else str(dev))
    if not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + str(sampler.gpu_id)
    sampler.start()
    time.sleep(0.5)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps // chunk):
            g_chunk.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    barrier()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)

    ms = reduce_max(ms, "cuda")
    us_call = ms * 1e3 / args.steps  # per call on one GPU (slowest rank)
    value = whole_job_us_per_call(us_call, world)

    # hot-L2 context: the same call on one weight copy, back to back
    us_hot, e2e_us = None, None
    if args.quick:
        return finish(args, p, name, idx, world, aq, variant, copies, wbytes, l2, chunk, us_call,
                      value, us_hot, e2e_us, clocks, bytes_call, flops_call)
    g_hot = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_hot, stream=stream):
            for _ in range(256):
                fn(x, *ws[0], p.bits, out=ys[0], stream=stream)
        g_hot.replay()
        torch.cuda.synchronize()
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(8):
            g_hot.replay()
        h1.record(stream)
    torch.cuda.synchronize()
    us_hot = h0.elapsed_time(h1) * 1e3 / (8 * 256)

    # end to end through the host entry point: pinned x in, pinned y out
    e2e_steps = max(1, min(args.steps, 2000))
    x_host = x.cpu().pin_memory()
    y_host = torch.empty((p.M, p.N), dtype=x.dtype).pin_memory()
    x_dev = torch.empty_like(x)
    y_dev = torch.empty((p.M, p.N), dtype=x.dtype, device="cuda")
    for _ in range(min(20, e2e_steps)):
        aq.aq_matmul_host(x_host, *ws[0], p.bits, y_host, x_dev, y_dev, stream=stream)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        aq.aq_matmul_host(x_host, *ws[i % copies], p.bits, y_host, x_dev, y_dev, stream=stream)
    torch.cuda.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / e2e_steps, "cuda")
    comp = None
    if not args.no_compare:
        comp = gpu_comparisons(p, ws, x, torch, l2, stream)
    line, p = finish(args, p, name, idx, world, aq, variant, copies, wbytes, l2, chunk, us_call,
                     value, us_hot, e2e_us, clocks, bytes_call, flops_call)
    line["gpu_comparisons"] = comp
    return line, p


def finish(args, p, name, idx, world, aq, variant, copies, wbytes, l2, chunk, us_call, value,
           us_hot, e2e_us, clocks, bytes_call, flops_call):
    err = aq.aq_device_error()
    hbm, tc, src = peaks()
    t_s = us_call * 1e-6
    bound = "hbm" if bytes_call / (hbm * 1e9) >= flops_call / (tc * 1e12) else "tensor"
    if bound == "hbm":
        achieved, peak, unit = bytes_call / t_s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = flops_call / t_s / 1e12, tc, "TFLOP/s"
    rec = traffic_record()
    traffic = None
    if rec.get("workload") == args.workload and "dram_bytes_per_launch" in rec:
        traffic = float(rec["dram_bytes_per_launch"])
    t_roof = max(bytes_call / (hbm * 1e9), flops_call / (tc * 1e12))
    line = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": us_call / 1e3,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": p.x_dtype,
        "data": "synthetic",
        "config": {
            "workload": f"{name}[{idx}]: {p.bits}-bit affine group-64, N={p.N}, K={p.K}, "
                        f"M={p.M}, x {p.x_dtype}",
            "M": p.M, "N": p.N, "K": p.K, "bits": p.bits, "x_dtype": p.x_dtype,
            "variant": aq.aq_variant_name(variant),
            "l2": f"cold: {copies} rotating weight copies, {copies * wbytes / 1e6:.0f} MB "
                  f"> 2x L2 ({l2 / 1e6:.0f} MB)",
            "timing": f"CUDA events on the launching stream around {args.steps} calls "
                      f"replayed from CUDA graphs of {chunk}",
            "parallelism": f"replicas x{world}",
        },
        "effective_gbs": round(bytes_call / t_s / 1e9, 1),
        "tflops": round(flops_call / t_s / 1e12, 3),
        "roofline_time_us": round(t_roof * 1e6, 3),
        "roofline_frac_nominal_8tbs": round(bytes_call / t_s / 8e12, 4) if bound == "hbm" else None,
        "hot_l2_us_per_call": round(us_hot, 4) if us_hot is not None else None,
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{src} (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": bytes_call,
                     "flops_per_launch": flops_call},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3)
                if e2e_us is not None else None,
                "unit": "us/call",
                "h2d_bytes_per_step": p.M * p.K * 2, "d2h_bytes_per_step": p.M * p.N * 2,
                "path": "aq_matmul_host (pinned x -> device, matmul, device -> pinned y, sync)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "device_error": err,
    }
    return line, p


QUANTIZE_METRIC = "µs/call and effective HBM GB/s (fraction of roofline), float -> affine group-64 quantiser"


def run_quantize(args, rank, world, local_rank):
    """The quantiser (aq_quantize / aq_quantize_bf16) on one of its workloads:
    device-timed calls over rotating weight copies (> 2x L2), the same through
    host buffers, and the oracle's quantiser on a row sample of the host."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    torch.cuda.set_device(local_rank)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    name, idx = parse_workload(args.workload)
    bits, N, K, dt, seed = workloads.QUANTIZE_WORKLOADS[name][idx]
    b16, vals = workloads.make_weights(N, K, dt, seed)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    w0 = torch.from_numpy(b16.view(np.int16)).cuda().view(tdt)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    copies = max(2, -(-2 * l2 // (2 * N * K)) + 1)
    ws = [w0.clone() for _ in range(copies)]
    q = aq.aq_quantize_bf16 if dt == "bf16" else aq.aq_quantize
    outs = [q(w, bits) for w in ws]
    stream = torch.cuda.Stream()

    def capture(ncalls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(ncalls):
                    c = i % copies
                    f = aq.load().aq_quantize_bf16 if dt == "bf16" else aq.load().aq_quantize
                    Wq, sc, bi = outs[c]
                    f(ws[c].data_ptr(), N, K, bits, Wq.data_ptr(), sc.data_ptr(), bi.data_ptr(),
                      stream.cuda_stream)
        return g

    steps = max(1, min(args.steps, 2000))
    chunk = min(256, steps)
    g = capture(chunk)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // chunk)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else "0")
    if not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + str(sampler.gpu_id)
    sampler.start()
    time.sleep(0.5)
    torch.cuda.synchronize()
    reps = max(1, steps // chunk)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    us_call = reduce_max(ev0.elapsed_time(ev1) * 1e3 / (reps * chunk), "cuda")

    # end to end: pinned weights in, packed codes, scales and biases out
    w_host = w0.cpu().pin_memory()
    Wq_h = torch.empty_like(outs[0][0], device="cpu").pin_memory()
    s_h = torch.empty_like(outs[0][1], device="cpu").pin_memory()
    b_h = torch.empty_like(outs[0][2], device="cpu").pin_memory()
    n_e2e = 50
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            ws[0].copy_(w_host, non_blocking=True)
            Wq, sc, bi = q(ws[0], bits, stream=stream)
            Wq_h.copy_(Wq, non_blocking=True)
            s_h.copy_(sc, non_blocking=True)
            b_h.copy_(bi, non_blocking=True)
            stream.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / n_e2e, "cuda")

    hbm, _, src = peaks()
    by = workloads.quantize_bytes(N, K, bits)
    achieved = by / (us_call * 1e-6) / 1e9
    line = {
        "metric": QUANTIZE_METRIC,
        "value": round(whole_job_us_per_call(us_call, world), 4),
        "unit": "us/call",
        "n_gpus": world, "steps": reps * chunk, "warmup": args.warmup,
        "ms_per_step": us_call / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: quantise {N}x{K} {dt} weights to {bits}-bit "
                               f"affine group-64",
                   "N": N, "K": K, "bits": bits, "w_dtype": dt,
                   "l2": f"cold: {copies} rotating weight copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {reps} replays of a "
                             f"CUDA graph of {chunk} calls",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": by},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * N * K,
                "d2h_bytes_per_step": N * K * bits // 8 + 4 * N * (K // 64),
                "path": "pinned weights -> device, aq_quantize, codes/scales/biases -> pinned "
                        "host, sync"},
        "gpu_launches": reps * chunk,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        import oracle
        oracle.build()
        rows = min(N, 512)
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < min(args.cpu_budget, 10.0) or n == 0:
            oracle.quantize(vals[:rows], bits)
            n += 1
        us = (time.perf_counter() - t0) / n * (N / rows) * 1e6
        line["cpu_baseline"] = {"value": round(us, 1), "unit": "us/call", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{n} runs of the oracle quantiser on {rows} of {N} "
                                          f"rows, scaled by N/{rows}; 1 thread"}
    return line


LAYER_METRIC = ("µs per decoder-layer step and effective HBM GB/s (fraction of roofline), "
                "7 affine group-64 projections at M rows")
# name -> list of (M, fused)
LAYER_STEPS = {"layerstep": [(1, True), (1, False), (8, True), (8, False)]}


def run_layer_step(args, rank, world, local_rank):
    """One decoder-layer step of the 5120-hidden layer workload (q, k, v, o,
    gate, up, down at 4 bits, bf16): fused = q/k/v in one aq_matmul_multi
    call, gate/up + SiLU in one aq_matmul_gate_up call, then o and down;
    unfused = the seven projections as seven calls (no SiLU)."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    torch.cuda.set_device(local_rank)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    name, idx = parse_workload(args.workload)
    M, fused = LAYER_STEPS[name][idx]
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    layer_bytes = sum(workloads.algorithmic_bytes(M, N, K, 4)
                      for _, N, K in workloads.LAYER_PROJECTIONS)
    wbytes = sum(N * K // 2 + 4 * N * (K // 64) for _, N, K in workloads.LAYER_PROJECTIONS)
    copies = max(2, -(-2 * l2 // wbytes) + 1)
    base = {}
    for j, (n, N, K) in enumerate(workloads.LAYER_PROJECTIONS):
        p = workloads.make_problem(n, 4, N, K, M, "bf16", seed=30 + j)
        base[n] = (aq.aq_pack(torch.from_numpy(p.codes).cuda(), 4),
                   torch.from_numpy(p.scales).cuda(), torch.from_numpy(p.biases).cuda())
    W = [base] + [{n: tuple(t.clone() for t in w) for n, w in base.items()}
                  for _ in range(copies - 1)]
    xb = workloads.make_x(M, 5120, "bf16", seed=7)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    xo = x.clone()
    h = torch.empty((M, 13824), dtype=torch.bfloat16, device="cuda")
    outs = {n: torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            for n, N, _ in workloads.LAYER_PROJECTIONS}
    stream = torch.cuda.Stream()

    def step(d, xin):
        if fused:
            aq.aq_matmul_multi(xin, [d["q"], d["k"], d["v"]], 4,
                               outs=[outs["q"], outs["k"], outs["v"]], stream=stream)
            aq.aq_matmul_bf16(xo, *d["o"], 4, out=outs["o"], stream=stream)
            aq.aq_matmul_gate_up(xin, d["gate"], d["up"], 4, out=h, stream=stream)
            aq.aq_matmul_bf16(h, *d["down"], 4, out=outs["down"], stream=stream)
            return 4
        for n in ("q", "k", "v"):
            aq.aq_matmul_bf16(xin, *d[n], 4, out=outs[n], stream=stream)
        aq.aq_matmul_bf16(xo, *d["o"], 4, out=outs["o"], stream=stream)
        aq.aq_matmul_bf16(xin, *d["gate"], 4, out=outs["gate"], stream=stream)
        aq.aq_matmul_bf16(xin, *d["up"], 4, out=outs["up"], stream=stream)
        aq.aq_matmul_bf16(h, *d["down"], 4, out=outs["down"], stream=stream)
        return 7

    steps = max(1, min(args.steps, 4096))
    chunk = min(64, steps)
    with torch.cuda.stream(stream):
        step(W[0], x)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launches = sum(step(W[i % copies], x) for i in range(chunk))
        for _ in range(max(1, args.warmup // chunk)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else "0")
    if not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + str(sampler.gpu_id)
    sampler.start()
    time.sleep(0.5)
    reps = max(1, steps // chunk)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    us = reduce_max(ev0.elapsed_time(ev1) * 1e3 / (reps * chunk), "cuda")

    # end to end: pinned x in, the layer's last output (down) back to the host
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((M, 5120), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    n_e2e = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            step(W[i % copies], x_dev)
            y_host.copy_(outs["down"], non_blocking=True)
            stream.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / n_e2e, "cuda")

    hbm, _, src = peaks()
    achieved = layer_bytes / (us * 1e-6) / 1e9
    return {
        "metric": LAYER_METRIC,
        "value": round(whole_job_us_per_call(us, world), 3),
        "unit": "us/step",
        "n_gpus": world, "steps": reps * chunk, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: one 5120-hidden decoder layer (q,k,v,o,gate,up,"
                               f"down), 4-bit, M={M}, "
                               + ("fused: q/k/v multi, gate/up+SiLU" if fused
                                  else "seven separate calls"),
                   "M": M, "fused": fused,
                   "l2": f"cold: {copies} rotating copies of the layer's weights "
                         f"({copies * wbytes / 1e6:.0f} MB > 2x L2)",
                   "timing": f"CUDA events on the launching stream around {reps} replays of a "
                             f"CUDA graph of {chunk} steps",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": layer_bytes},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/step",
                "h2d_bytes_per_step": M * 5120 * 2, "d2h_bytes_per_step": M * 5120 * 2,
                "path": "pinned x -> device, the layer's calls, down output -> pinned host, sync"},
        "gpu_launches": reps * launches,
        "clocks": clocks,
    }


WIDTHS_METRIC = ("µs/call and effective HBM GB/s (fraction of roofline), other code widths and "
                 "group sizes, y=x·Wᵀ")
# name -> list of (bits, group, N, K, M, x dtype)
WIDTH_WORKLOADS = {"widths": [(8, 64, 4096, 4096, 1, "bf16"), (2, 32, 4096, 4096, 1, "bf16"),
                              (6, 128, 4096, 4096, 1, "bf16"), (4, 128, 4096, 4096, 1, "bf16"),
                              (8, 32, 4096, 4096, 16, "fp16")]}


def run_widths(args, rank, world, local_rank):
    """aq_matmul_ex on a width / group size other than the 3/4-bit group-64
    format: device-timed calls over rotating weight copies (> 2x L2) and the
    same through host buffers."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    torch.cuda.set_device(local_rank)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    name, idx = parse_workload(args.workload)
    bits, group, N, K, M, dt = WIDTH_WORKLOADS[name][idx]
    rng = np.random.default_rng(60 + idx)
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    s = (np.abs(rng.standard_normal((N, G))) * (0.16 / (1 << bits)) + 1e-3).astype(np.float16)
    b = (-(1 << (bits - 1)) * s.astype(np.float64)).astype(np.float16)
    xb = workloads.make_x(M, K, dt, seed=61)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(tdt)
    Wq0 = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    s0, b0 = torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda()
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    wbytes = N * K * bits // 8 + 4 * N * G
    copies = max(2, -(-2 * l2 // wbytes) + 1)
    ws = [(Wq0.clone(), s0.clone(), b0.clone()) for _ in range(copies)]
    ys = [torch.empty((M, N), dtype=tdt, device="cuda") for _ in range(copies)]
    stream = torch.cuda.Stream()
    steps = max(1, min(args.steps, 4096))
    chunk = min(256, steps)
    with torch.cuda.stream(stream):
        aq.aq_matmul_ex(x, *ws[0], bits, group, out=ys[0], stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(chunk):
                c = i % copies
                aq.aq_matmul_ex(x, *ws[c], bits, group, out=ys[c], stream=stream)
        for _ in range(max(1, args.warmup // chunk)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else "0")
    if not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + str(sampler.gpu_id)
    sampler.start()
    time.sleep(0.5)
    reps = max(1, steps // chunk)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    us = reduce_max(ev0.elapsed_time(ev1) * 1e3 / (reps * chunk), "cuda")
    x_host = torch.from_numpy(xb.view(np.int16)).view(tdt).pin_memory()
    y_host = torch.empty((M, N), dtype=tdt).pin_memory()
    x_dev = torch.empty_like(x)
    n_e2e = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            aq.aq_matmul_ex(x_dev, *ws[i % copies], bits, group, out=ys[0], stream=stream)
            y_host.copy_(ys[0], non_blocking=True)
            stream.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / n_e2e, "cuda")
    hbm, _, src = peaks()
    by = wbytes + 2 * M * K + 2 * M * N
    achieved = by / (us * 1e-6) / 1e9
    return {
        "metric": WIDTHS_METRIC,
        "value": round(whole_job_us_per_call(us, world), 3),
        "unit": "us/call",
        "n_gpus": world, "steps": reps * chunk, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: {bits}-bit affine group-{group}, N={N}, K={K}, "
                               f"M={M}, x {dt}",
                   "bits": bits, "group": group, "M": M, "N": N, "K": K,
                   "variant": aq.aq_variant_name(aq.AQ_VARIANT_GENERIC),
                   "l2": f"cold: {copies} rotating weight copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {reps} replays of a "
                             f"CUDA graph of {chunk} calls",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": by},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * M * K, "d2h_bytes_per_step": 2 * M * N,
                "path": "pinned x -> device, aq_matmul_ex, y -> pinned host, sync"},
        "gpu_launches": reps * chunk,
        "clocks": clocks,
    }


ATTN_METRIC = ("µs/call and effective HBM GB/s (fraction of roofline), decode attention over "
               "an affine-quantised KV cache")
# name -> list of (H, KV, N, D, bits, group, q dtype)
ATTN_WORKLOADS = {"attention": [(16, 8, 8192, 256, 4, 64, "bf16"), (16, 8, 2048, 256, 4, 64, "bf16"),
                                (16, 8, 32768, 256, 4, 64, "bf16"), (16, 8, 8192, 256, 8, 64, "bf16"),
                                (32, 8, 8192, 128, 4, 64, "bf16"), (16, 8, 8192, 512, 4, 64, "bf16")]}


def run_attention(args, rank, world, local_rank):
    """aq_attention_decode on one decode step of a quantised KV cache:
    device-timed calls over rotating cache copies (> 2x L2) and the same
    through host buffers (q in, o out)."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    torch.cuda.set_device(local_rank)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    name, idx = parse_workload(args.workload)
    H, KV, N, D, bits, group, dt = ATTN_WORKLOADS[name][idx]
    rng = np.random.default_rng(70 + idx)
    R = KV * N
    G = D // group

    def cache():
        codes = rng.integers(0, 1 << bits, size=(R, D), dtype=np.uint8)
        s = (np.abs(rng.standard_normal((R, G))) * (0.16 / (1 << bits)) + 1e-3).astype(np.float16)
        b = (-(1 << (bits - 1)) * s.astype(np.float64)).astype(np.float16)
        return (aq.aq_pack(torch.from_numpy(codes).cuda(), bits).view(KV, N, D * bits // 32),
                torch.from_numpy(s).cuda().view(KV, N, G), torch.from_numpy(b).cuda().view(KV, N, G))

    k0, v0 = cache(), cache()
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    qb = workloads.make_x(H, D, dt, seed=71)
    q = torch.from_numpy(qb.view(np.int16)).cuda().view(tdt)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    cbytes = 2 * (R * D * bits // 8 + 4 * R * G)
    copies = max(2, -(-2 * l2 // cbytes) + 1)
    caches = [(tuple(t.clone() for t in k0), tuple(t.clone() for t in v0)) for _ in range(copies)]
    outs = [torch.empty((H, D), dtype=tdt, device="cuda") for _ in range(copies)]
    stream = torch.cuda.Stream()
    steps = max(1, min(args.steps, 4096))
    chunk = min(256, steps)
    with torch.cuda.stream(stream):
        aq.aq_attention_decode(q, *caches[0], bits, group, out=outs[0], stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(chunk):
                c = i % copies
                aq.aq_attention_decode(q, *caches[c], bits, group, out=outs[c], stream=stream)
        for _ in range(max(1, args.warmup // chunk)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else "0")
    if not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + str(sampler.gpu_id)
    sampler.start()
    time.sleep(0.5)
    reps = max(1, steps // chunk)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    us = reduce_max(ev0.elapsed_time(ev1) * 1e3 / (reps * chunk), "cuda")
    q_host = torch.from_numpy(qb.view(np.int16)).view(tdt).pin_memory()
    o_host = torch.empty((H, D), dtype=tdt).pin_memory()
    q_dev = torch.empty_like(q)
    n_e2e = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            q_dev.copy_(q_host, non_blocking=True)
            aq.aq_attention_decode(q_dev, *caches[i % copies], bits, group, out=outs[0],
                                   stream=stream)
            o_host.copy_(outs[0], non_blocking=True)
            stream.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / n_e2e, "cuda")
    hbm, _, src = peaks()
    by = cbytes + 2 * 2 * H * D
    rec = traffic_record("traffic_attention.txt")
    attn_traffic = None
    if rec.get("workload") == args.workload and "dram_bytes_per_launch" in rec:
        attn_traffic = float(rec["dram_bytes_per_launch"])
    achieved = by / (us * 1e-6) / 1e9
    return {
        "metric": ATTN_METRIC,
        "value": round(whole_job_us_per_call(us, world), 3),
        "unit": "us/call",
        "n_gpus": world, "steps": reps * chunk, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: {H} query heads over {KV} KV heads of {D}, "
                               f"{N} cached rows, {bits}-bit group-{group} K and V, q {dt}",
                   "H": H, "KV": KV, "N": N, "D": D, "bits": bits, "group": group,
                   "l2": f"cold: {copies} rotating cache copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {reps} replays of a "
                             f"CUDA graph of {chunk} calls",
                   "launch": aq.aq_attention_describe(H, KV, N, D, bits, group),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": attn_traffic,
                     "peak_source": f"{src} (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": by},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * H * D, "d2h_bytes_per_step": 2 * H * D,
                "path": "pinned q -> device, aq_attention_decode, o -> pinned host, sync"},
        "gpu_launches": reps * chunk,
        "clocks": clocks,
    }


def cpu_sample_time(p, budget_s, threads):
    """Time the oracle on a column sample of p; returns (us per full call, desc)."""
    import oracle
    words = oracle.pack(p.codes, p.bits)
    x = p.x_f64()
    cols = np.arange(min(p.N, 64))
    t0 = time.perf_counter()
    oracle.matmul_cols(x, words, p.scales, p.biases, p.bits, cols)
    t_col = (time.perf_counter() - t0) / len(cols)
    full = t_col * p.N / max(1, threads)
    reps = max(1, int(budget_s / max(full, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.matmul(x, words, p.scales, p.biases, p.bits, threads=threads)
    dt = (time.perf_counter() - t0) / reps
    return dt * 1e6, f"{reps} full calls of the workload ({p.M}x{p.N}x{p.K}) on {threads} threads"


def run_reference(args, rank, world):
    """The oracle on the host cores, as the reference arm."""
    import oracle
    oracle.build()
    name, idx = parse_workload(args.workload)
    p = workloads.workload(name, idx)
    words = oracle.pack(p.codes, p.bits)
    x = p.x_f64()
    threads = os.cpu_count() or 1
    # calibrate: seconds per output column on all threads
    cols = np.arange(min(p.N, 256))
    t0 = time.perf_counter()
    oracle.matmul_cols(x, words, p.scales, p.biases, p.bits, cols)
    t_col = (time.perf_counter() - t0) / len(cols) / threads
    total = args.steps + args.warmup
    per_step_budget = 90.0 / max(1, total)
    ncols = int(min(p.N, max(threads, per_step_budget / max(t_col, 1e-9))))
    rng = np.random.default_rng(0)
    step_times = []
    for i in range(total):
        start = int(rng.integers(0, p.N - ncols + 1))
        c = slice(start, start + ncols)  # a random window of output columns
        sub_words = np.ascontiguousarray(words[c])
        t0 = time.perf_counter()
        oracle.matmul(x, sub_words, p.scales[c], p.biases[c], p.bits, threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            step_times.append(dt * p.N / ncols)
    us = statistics.mean(step_times) * 1e6
    sample = (f"each step: {ncols} of {p.N} output columns (all {p.M} rows), scaled by "
              f"N/{ncols}; {threads} threads")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(us, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": us / 1e3,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: {p.bits}-bit affine group-64, N={p.N}, K={p.K}, "
                               f"M={p.M}, x {p.x_dtype}",
                   "M": p.M, "N": p.N, "K": p.K, "bits": p.bits, "x_dtype": p.x_dtype,
                   "implementation": "fp64 C oracle (oracle/aq_oracle.c) on host cores"},
        "cpu_baseline": {"value": round(us, 3), "unit": "us/call", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 3), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=2048)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of host time for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all", action="store_true", help="one line per workload (not the default)")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only: skip the hot-L2, end-to-end and CPU legs")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the torch.matmul comparison leg of the default workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    specs = [args.workload]
    if args.all:
        specs = [f"{n}:{i}" for n, c in workloads.WORKLOADS.items() for i in range(len(c))]
    for spec in specs:
        args.workload = spec
        if parse_workload(spec)[0] in ATTN_WORKLOADS:
            line = run_attention(args, rank, world, local_rank)
            if rank == 0:
                print(json.dumps(line), flush=True)
            continue
        if parse_workload(spec)[0] in WIDTH_WORKLOADS:
            line = run_widths(args, rank, world, local_rank)
            if rank == 0:
                print(json.dumps(line), flush=True)
            continue
        if parse_workload(spec)[0] in LAYER_STEPS:
            line = run_layer_step(args, rank, world, local_rank)
            if rank == 0:
                print(json.dumps(line), flush=True)
            continue
        if parse_workload(spec)[0] in workloads.QUANTIZE_WORKLOADS:
            line = run_quantize(args, rank, world, local_rank)
            if rank == 0:
                print(json.dumps(line), flush=True)
            continue
        line, p = run_ours(args, rank, world, local_rank)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline and not args.all and not args.quick:
                import oracle
                oracle.build()
                threads = os.cpu_count() or 1
                us, desc = cpu_sample_time(p, args.cpu_budget, threads)
                line["cpu_baseline"] = {"value": round(us, 1), "unit": "us/call",
                                        "cores": threads, "kind": "oracle", "sample": desc}
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: affine group-64 quantized matmul y = x . W^T on GB300.

Default: one JSON line for the largest single-GPU configuration of the
metric (4-bit 28672 x 8192 prefill at M = 512, bf16 activations; the metric
spans M = 1..512), carrying a `per_config` map with the time of every other
configuration measured in the same invocation:

    small     4-bit 1024 x 512, M = 1, fp16
    decode    4-bit 4096 x 4096, M = 1, bf16
    split3    3-bit 10240 x 5120, M in {1, 9, 16, 32, 64}, fp16
    layer     the seven 4-bit projections of a 5120-hidden decoder layer,
              M = 1, bf16, and the whole layer step (fused calls)
    prefill   4-bit 28672 x 8192, M in {128, 512}, bf16 (and M = 256 beside
              them: the middle of the tensor-core range)

One step is one library call (one pass of the hot path over one batch of
activations).  The headline's timed region holds exactly `--steps` calls,
replayed from CUDA graphs that were themselves replayed during the warm-up,
cycling through enough copies of the weights that their total exceeds twice
the L2 size (every call reads its weights from HBM).  A short device-side
sleep is queued before the start event, so the events bracket the device's
execution of exactly those calls and not the host's graph submission.
Each `per_config` entry is the median over five such regions of
max(--steps, 200) calls.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload small|decode|split3:I|layer:I|prefill:I|quantize:I|
                                layerstep:I|widths:I|attention:I|attnws:I] [--all]

--workload times one workload alone (no per_config).  widths:I times
aq_matmul_ex on other code widths and group sizes; attention:I times
aq_attention_decode (decode attention over a quantised KV cache), attnws:I
the same shapes through aq_attention_decode_ws (a workspace: several
clusters a KV head);
layerstep:I times one decoder-layer step (seven projections; I = 0/1 fused or
not at M = 1, 2/3 at M = 8); quantize:I times the float -> affine quantiser.

Matmul lines also carry `gpu_comparisons` (context, not targets):
torch.matmul (cuBLAS) on the weights dequantised once, and (4-bit) a torch-op
dequantise of the packed words followed by torch.matmul on every call
(--no-compare skips them).  `cpu_baseline` is the fp64 oracle timed on the
host cores, once on all cores and once on one core, each on a bounded sample
of output columns scaled to a full call.

Prints one JSON line per workload (rank 0).  Under torchrun (N > 1) every
rank runs an independent replica on its own GPU ("replicas only": the method
needs no exchange between GPUs); the time is the maximum over ranks.

--impl reference times the fp64 C oracle on the host cores instead (the
method has no other implementation to run here): each step is a bounded
sample of output columns of the same workload, scaled to the metric's unit.
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
DEFAULT_WORKLOAD = "prefill:1"
GRAPH_CHUNK = 1024
SLEEP_CYCLES = 400_000        # ~0.2 ms of device sleep before a start event
PER_CONFIG_MIN_CALLS = 200
PER_CONFIG_REGIONS = 5
SUSTAIN_S = 0.6               # replays after a headline region, for the clock record
PER_CONFIG_SPECS = (["small:0", "decode:0"] + [f"split3:{i}" for i in range(5)]
                    + [f"layer:{i}" for i in range(7)] + ["layerstep:0", "prefill:0",
                                                          "prefill:2", "prefill:1"])


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


def peak_source(src):
    return f"{src} (MEASURED_PEAKS.json)" if src == "measured" else "fallback"


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
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons,
    for the whole run; window(t0, t1) summarises the samples inside one
    stretch of time."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id if str(gpu_id).startswith("GPU-") else "GPU-" + str(gpu_id)
        self.proc = None
        self.lines = []

    @classmethod
    def for_device(cls, torch, dev):
        props = torch.cuda.get_device_properties(dev)
        return cls(str(props.uuid) if hasattr(props, "uuid") else str(dev))

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.proc = None

    def window(self, t0, t1):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside, near = [], []
        for ts, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if t0 <= ts <= t1 + 0.06:
                inside.append(parts)
            elif t0 - 1.0 <= ts <= t1 + 1.0:
                near.append(parts)
        use = inside or near[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [v for v in (num(p[1]) for p in use) if v is not None]
        mx = [v for v in (num(p[2]) for p in use) if v is not None]
        pw = [v for v in (num(p[3]) for p in use) if v is not None]
        reasons = sorted({self.REASONS[i] for p in use for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(pw) if pw else None}


class GraphTimer:
    """`ncalls` calls of `call(i)` captured into CUDA graphs (full chunks plus
    a remainder) and timed with CUDA events on `stream`.

    Calls i cycle over `copies` weight copies (call(i) picks copy i % copies);
    when a chunk holds at least `copies` calls it holds a whole number of
    rotations, so successive replays continue the rotation and no copy comes
    back before the others have been read."""

    def __init__(self, torch, stream, call, ncalls, copies=1, chunk_max=GRAPH_CHUNK):
        self.torch, self.stream, self.ncalls = torch, stream, ncalls
        chunk = min(chunk_max, ncalls)
        if chunk >= copies:
            chunk -= chunk % copies
        self.chunk = chunk
        self.full = ncalls // chunk
        rem = ncalls - self.full * chunk
        self.g_chunk = self._capture(call, chunk, 0)
        self.g_rem = self._capture(call, rem, self.full * chunk) if rem else None

    def _capture(self, call, n, start):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    call(start + i)
        return g

    def _replay_all(self):
        for _ in range(self.full):
            self.g_chunk.replay()
        if self.g_rem is not None:
            self.g_rem.replay()

    def warm(self, warmup_calls):
        """Replay every graph that the timed region replays (at least once
        each), then the chunk graph until `warmup_calls` calls have run."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.g_chunk.replay()
            done = self.chunk
            if self.g_rem is not None:
                self.g_rem.replay()
            while done < warmup_calls:
                self.g_chunk.replay()
                done += self.chunk
        torch.cuda.synchronize()

    def time_ms(self):
        """Device time of exactly `ncalls` calls."""
        torch = self.torch
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record(self.stream)
            self._replay_all()
            e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    def sustain(self, seconds):
        """Replay the timed graphs back to back for about `seconds` (clock
        record under load); returns the median µs per call of those regions."""
        per = []
        t_end = time.time() + seconds
        while time.time() < t_end:
            per.append(self.time_ms() * 1e3 / self.ncalls)
        return statistics.median(per) if per else None


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# The matmul configurations
# ---------------------------------------------------------------------------

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


class MatmulSetup:
    """One matmul workload resident on the device: x, `copies` weight copies
    (> 2x L2 in total) and one output per copy."""

    def __init__(self, p, torch, aq, l2):
        self.p, self.torch, self.aq = p, torch, aq
        self.wbytes = p.N * p.K * p.bits // 8 + 4 * p.N * p.G
        self.copies = max(2, -(-2 * l2 // self.wbytes) + 1)
        self.x, self.ws = device_problem(p, self.copies, torch, aq)
        self.ys = [torch.empty((p.M, p.N), dtype=self.x.dtype, device="cuda")
                   for _ in range(self.copies)]
        self.fn = aq.aq_matmul_bf16 if p.x_dtype == "bf16" else aq.aq_matmul
        self.dtype_code = aq.AQ_BF16 if p.x_dtype == "bf16" else aq.AQ_F16
        self.variant = aq.aq_select(p.M, p.N, p.K, p.bits, self.dtype_code)
        self.stream = torch.cuda.Stream()
        self.bytes_call = workloads.algorithmic_bytes(p.M, p.N, p.K, p.bits)
        self.flops_call = workloads.flops(p.M, p.N, p.K)
        with torch.cuda.stream(self.stream):
            self.call(0)
        torch.cuda.synchronize()

    def call(self, i):
        c = i % self.copies
        Wq, s, b = self.ws[c]
        self.fn(self.x, Wq, s, b, self.p.bits, out=self.ys[c], stream=self.stream)

    def timer(self, ncalls):
        return GraphTimer(self.torch, self.stream, self.call, ncalls, self.copies)

    def l2_note(self, l2):
        return (f"cold: {self.copies} rotating weight copies, "
                f"{self.copies * self.wbytes / 1e6:.0f} MB > 2x L2 ({l2 / 1e6:.0f} MB)")

    def free(self):
        del self.x, self.ws, self.ys
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def roofline_of(bytes_call, flops_call, us):
    """(bound, achieved, peak, unit, frac, source) for one call of `us` µs."""
    hbm, tc, src = peaks()
    t = us * 1e-6
    bound = "hbm" if bytes_call / (hbm * 1e9) >= flops_call / (tc * 1e12) else "tensor"
    if bound == "hbm":
        achieved, peak, unit = bytes_call / t / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = flops_call / t / 1e12, tc, "TFLOP/s"
    return bound, achieved, peak, unit, achieved / peak, src


def config_entry(label, us_list, bytes_call, flops_call, clocks, extra):
    us = statistics.median(us_list)
    bound, achieved, peak, unit, frac, src = roofline_of(bytes_call, flops_call, us)
    e = {"workload": label, "us_per_call": round(us, 4),
         "us_min": round(min(us_list), 4), "us_max": round(max(us_list), 4),
         "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(frac, 4), "effective_gbs": round(bytes_call / (us * 1e-6) / 1e9, 1),
         "tflops": round(flops_call / (us * 1e-6) / 1e12, 3),
         "algorithmic_bytes_per_call": bytes_call, "flops_per_call": flops_call,
         "clocks": clocks}
    e.update(extra)
    return e


def time_config_regions(timer, sampler, world):
    us_list = []
    t0 = time.time()
    for _ in range(PER_CONFIG_REGIONS):
        _barrier(world)
        us_list.append(reduce_max(timer.time_ms() * 1e3 / timer.ncalls, "cuda"))
    t1 = time.time()
    return us_list, sampler.window(t0, t1)


def per_config_matmul(spec, args, torch, aq, l2, sampler, world, setup=None):
    name, idx = parse_workload(spec)
    own = setup is None
    if own:
        setup = MatmulSetup(workloads.workload(name, idx), torch, aq, l2)
    p = setup.p
    n = max(args.steps, PER_CONFIG_MIN_CALLS)
    timer = setup.timer(n)
    timer.warm(max(args.warmup, n))
    us_list, clocks = time_config_regions(timer, sampler, world)
    e = config_entry(f"{name}[{idx}]: {p.bits}-bit affine group-64, N={p.N}, K={p.K}, M={p.M}, "
                     f"x {p.x_dtype}", us_list, setup.bytes_call, setup.flops_call, clocks,
                     {"variant": aq.aq_variant_name(setup.variant),
                      "calls_per_region": n, "regions": PER_CONFIG_REGIONS,
                      "launches_per_call": 1})
    del timer
    if own:
        setup.free()
    return e


def gpu_comparisons(s, torch, l2):
    """Context, not targets: (1) torch.matmul (cuBLAS) on the weights
    dequantised once to x's dtype; (2) "expand": dequantise the packed words
    with torch ops on every call, then torch.matmul (4-bit only).  Both
    cold-L2 over rotating copies, CUDA events around CUDA-graph replays."""
    p, x, ws, stream = s.p, s.x, s.ws, s.stream
    dt = x.dtype
    G = p.K // 64
    s0 = ws[0][1].float().view(p.N, G, 1)
    b0 = ws[0][2].float().view(p.N, G, 1)
    codes = torch.from_numpy(p.codes).cuda().view(p.N, G, 64)
    w0 = (codes.float() * s0 + b0).view(p.N, p.K).to(dt)
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

    big = p.N * p.K > (1 << 26)

    def timed(body, calls):
        with torch.cuda.stream(stream):
            body(0)
        torch.cuda.synchronize()
        t = GraphTimer(torch, stream, body, calls, copies=1)
        t.warm(calls)
        return min(t.time_ms() for _ in range(3)) * 1e3 / calls

    out = {"dense_matmul_us": round(timed(lambda i: torch.matmul(x, dense[i % dcopies].t()),
                                          16 if big else 128), 3)}
    del dense, w0
    torch.cuda.empty_cache()
    out["expand_then_matmul_us"] = (round(timed(expand, 4 if big else 128), 3)
                                    if p.bits == 4 else None)
    out["note"] = ("context only: torch.matmul (cuBLAS) on weights dequantised once to "
                   f"{'bf16' if dt == torch.bfloat16 else 'fp16'} ({dcopies} copies, cold L2); "
                   "expand = torch-op dequantise of the packed words every call, then "
                   "torch.matmul")
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank, sampler, per_config):
    """The headline line for one matmul workload (exactly --steps timed calls),
    with per_config entries for every configuration when `per_config`."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    name, idx = parse_workload(args.workload)
    s = MatmulSetup(workloads.workload(name, idx), torch, aq, l2)
    p = s.p
    timer = s.timer(args.steps)
    timer.warm(args.warmup)

    _barrier(world)
    t0 = time.time()
    ms = timer.time_ms()
    t1 = time.time()
    sustained = timer.sustain(SUSTAIN_S) if not args.quick else None
    t2 = time.time()
    _barrier(world)
    clocks = sampler.window(t0, t2)
    clocks["window"] = ("timed region plus %.1f s of the same replays" % (t2 - t1)
                        if sustained is not None else "timed region")
    us_call = reduce_max(ms * 1e3 / args.steps, "cuda")
    value = whole_job_us_per_call(us_call, world)
    del timer

    us_hot = e2e_us = comp = None
    if not args.quick:
        # hot-L2 context: the same call on one weight copy, back to back
        def hot(i):
            s.fn(s.x, *s.ws[0], p.bits, out=s.ys[0], stream=s.stream)
        n_hot = 256 if p.M * p.N * p.K < (1 << 34) else 16
        th = GraphTimer(torch, s.stream, hot, n_hot)
        th.warm(n_hot)
        us_hot = th.time_ms() * 1e3 / n_hot
        del th
        # end to end through the host entry point: pinned x in, pinned y out
        e2e_steps = max(1, min(args.steps, 2000))
        x_host = s.x.cpu().pin_memory()
        y_host = torch.empty((p.M, p.N), dtype=s.x.dtype).pin_memory()
        x_dev = torch.empty_like(s.x)
        y_dev = torch.empty((p.M, p.N), dtype=s.x.dtype, device="cuda")
        for _ in range(min(5, e2e_steps)):
            aq.aq_matmul_host(x_host, *s.ws[0], p.bits, y_host, x_dev, y_dev, stream=s.stream)
        _barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            aq.aq_matmul_host(x_host, *s.ws[i % s.copies], p.bits, y_host, x_dev, y_dev,
                              stream=s.stream)
        torch.cuda.synchronize()
        e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / e2e_steps, "cuda")
        del x_dev, y_dev
        if not args.no_compare:
            comp = gpu_comparisons(s, torch, l2)

    line = matmul_line(args, p, name, idx, world, aq, s, l2, us_call, value, us_hot, e2e_us,
                       clocks, sustained)
    line["gpu_comparisons"] = comp

    if per_config:
        entries = {}
        for spec in PER_CONFIG_SPECS:
            if spec == args.workload:
                entries[spec] = per_config_matmul(spec, args, torch, aq, l2, sampler, world,
                                                  setup=s)
            elif parse_workload(spec)[0] in LAYER_STEPS:
                entries[spec] = per_config_layer_step(spec, args, torch, aq, l2, sampler, world)
            else:
                entries[spec] = per_config_matmul(spec, args, torch, aq, l2, sampler, world)
        line["per_config"] = entries
        line["per_config_note"] = (
            f"each entry: median (min, max) of {PER_CONFIG_REGIONS} regions of "
            f"max(--steps, {PER_CONFIG_MIN_CALLS}) calls, cold L2, same process; frac against "
            "the measured peak of the entry's bound (HBM copy GB/s, or bf16 burst TFLOP/s)")
    s.free()
    return line, p


def matmul_line(args, p, name, idx, world, aq, s, l2, us_call, value, us_hot, e2e_us, clocks,
                sustained):
    err = aq.aq_device_error()
    hbm, tc, src = peaks()
    bound, achieved, peak, unit, frac, src = roofline_of(s.bytes_call, s.flops_call, us_call)
    t_s = us_call * 1e-6
    rec = traffic_record()
    traffic = None
    if rec.get("workload") == args.workload and "dram_bytes_per_launch" in rec:
        traffic = float(rec["dram_bytes_per_launch"])
    t_roof = max(s.bytes_call / (hbm * 1e9), s.flops_call / (tc * 1e12))
    return {
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
            "variant": aq.aq_variant_name(s.variant),
            "l2": s.l2_note(l2),
            "timing": f"CUDA events on the launching stream around exactly {args.steps} calls "
                      "replayed from CUDA graphs (the same graphs replayed in the warm-up; a "
                      "device sleep before the start event hides the host's submission)",
            "parallelism": f"replicas x{world}",
        },
        "effective_gbs": round(s.bytes_call / t_s / 1e9, 1),
        "tflops": round(s.flops_call / t_s / 1e12, 3),
        "roofline_time_us": round(t_roof * 1e6, 3),
        "roofline_frac_nominal_8tbs": (round(s.bytes_call / t_s / 8e12, 4)
                                       if bound == "hbm" else None),
        "hot_l2_us_per_call": round(us_hot, 4) if us_hot is not None else None,
        "sustained_us_per_call": round(sustained, 4) if sustained is not None else None,
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(frac, 4), "traffic": traffic,
                     "peak_source": peak_source(src),
                     "algorithmic_bytes_per_launch": s.bytes_call,
                     "flops_per_launch": s.flops_call},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3)
                if e2e_us is not None else None,
                "unit": "us/call",
                "h2d_bytes_per_step": p.M * p.K * 2, "d2h_bytes_per_step": p.M * p.N * 2,
                "path": "aq_matmul_host (pinned x -> device, matmul, device -> pinned y, sync)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "device_error": err,
    }


# ---------------------------------------------------------------------------
# The quantiser
# ---------------------------------------------------------------------------

QUANTIZE_METRIC = "µs/call and effective HBM GB/s (fraction of roofline), float -> affine group-64 quantiser"


def run_quantize(args, rank, world, local_rank, sampler):
    """The quantiser (aq_quantize / aq_quantize_bf16) on one of its workloads:
    device-timed calls over rotating weight copies (> 2x L2), the same through
    host buffers, and the oracle's quantiser on a row sample of the host."""
    import torch
    import quantized_matmul_affine_gb300 as aq

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
    f = aq.load().aq_quantize_bf16 if dt == "bf16" else aq.load().aq_quantize

    def call(i):
        c = i % copies
        Wq, sc, bi = outs[c]
        f(ws[c].data_ptr(), N, K, bits, Wq.data_ptr(), sc.data_ptr(), bi.data_ptr(),
          stream.cuda_stream)

    steps = max(1, min(args.steps, 2000))
    timer = GraphTimer(torch, stream, call, steps, copies, chunk_max=256)
    timer.warm(args.warmup)
    _barrier(world)
    t0 = time.time()
    ms = timer.time_ms()
    clocks = sampler.window(t0, time.time())
    us_call = reduce_max(ms * 1e3 / steps, "cuda")

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
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": us_call / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: quantise {N}x{K} {dt} weights to {bits}-bit "
                               f"affine group-64",
                   "N": N, "K": K, "bits": bits, "w_dtype": dt,
                   "l2": f"cold: {copies} rotating weight copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {steps} calls "
                             f"replayed from CUDA graphs of {timer.chunk}",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": peak_source(src),
                     "algorithmic_bytes_per_launch": by},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * N * K,
                "d2h_bytes_per_step": N * K * bits // 8 + 4 * N * (K // 64),
                "path": "pinned weights -> device, aq_quantize, codes/scales/biases -> pinned "
                        "host, sync"},
        "gpu_launches": steps,
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


# ---------------------------------------------------------------------------
# One decoder-layer step
# ---------------------------------------------------------------------------

LAYER_METRIC = ("µs per decoder-layer step and effective HBM GB/s (fraction of roofline), "
                "7 affine group-64 projections at M rows")
# name -> list of (M, fused)
LAYER_STEPS = {"layerstep": [(1, True), (1, False), (8, True), (8, False)]}


class LayerSetup:
    """The 5120-hidden decoder layer's seven 4-bit projections on the device
    (copies > 2x L2), and one step of the layer: fused = q/k/v in one
    aq_matmul_multi call, gate/up + SiLU in one aq_matmul_gate_up call, then
    o and down; unfused = the seven projections as seven calls (no SiLU)."""

    def __init__(self, M, fused, torch, aq, l2):
        self.M, self.fused, self.torch, self.aq = M, fused, torch, aq
        self.layer_bytes = sum(workloads.algorithmic_bytes(M, N, K, 4)
                               for _, N, K in workloads.LAYER_PROJECTIONS)
        self.wbytes = sum(N * K // 2 + 4 * N * (K // 64) for _, N, K in workloads.LAYER_PROJECTIONS)
        self.copies = max(2, -(-2 * l2 // self.wbytes) + 1)
        base = {}
        for j, (n, N, K) in enumerate(workloads.LAYER_PROJECTIONS):
            p = workloads.make_problem(n, 4, N, K, M, "bf16", seed=30 + j)
            base[n] = (aq.aq_pack(torch.from_numpy(p.codes).cuda(), 4),
                       torch.from_numpy(p.scales).cuda(), torch.from_numpy(p.biases).cuda())
        self.W = [base] + [{n: tuple(t.clone() for t in w) for n, w in base.items()}
                           for _ in range(self.copies - 1)]
        self.xb = workloads.make_x(M, 5120, "bf16", seed=7)
        self.x = torch.from_numpy(self.xb.view(np.int16)).cuda().view(torch.bfloat16)
        self.xo = self.x.clone()
        self.h = torch.empty((M, 13824), dtype=torch.bfloat16, device="cuda")
        self.outs = {n: torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                     for n, N, _ in workloads.LAYER_PROJECTIONS}
        self.stream = torch.cuda.Stream()
        self.launches = 4 if fused else 7
        with torch.cuda.stream(self.stream):
            self.step(self.W[0], self.x)
        torch.cuda.synchronize()

    def step(self, d, xin):
        aq, outs, stream = self.aq, self.outs, self.stream
        if self.fused:
            aq.aq_matmul_multi(xin, [d["q"], d["k"], d["v"]], 4,
                               outs=[outs["q"], outs["k"], outs["v"]], stream=stream)
            aq.aq_matmul_bf16(self.xo, *d["o"], 4, out=outs["o"], stream=stream)
            aq.aq_matmul_gate_up(xin, d["gate"], d["up"], 4, out=self.h, stream=stream)
            aq.aq_matmul_bf16(self.h, *d["down"], 4, out=outs["down"], stream=stream)
            return
        for n in ("q", "k", "v"):
            aq.aq_matmul_bf16(xin, *d[n], 4, out=outs[n], stream=stream)
        aq.aq_matmul_bf16(self.xo, *d["o"], 4, out=outs["o"], stream=stream)
        aq.aq_matmul_bf16(xin, *d["gate"], 4, out=outs["gate"], stream=stream)
        aq.aq_matmul_bf16(xin, *d["up"], 4, out=outs["up"], stream=stream)
        aq.aq_matmul_bf16(self.h, *d["down"], 4, out=outs["down"], stream=stream)

    def call(self, i):
        self.step(self.W[i % self.copies], self.x)

    def timer(self, ncalls):
        return GraphTimer(self.torch, self.stream, self.call, ncalls, self.copies, chunk_max=64)

    def free(self):
        del self.W, self.x, self.xo, self.h, self.outs
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def per_config_layer_step(spec, args, torch, aq, l2, sampler, world):
    name, idx = parse_workload(spec)
    M, fused = LAYER_STEPS[name][idx]
    s = LayerSetup(M, fused, torch, aq, l2)
    n = max(args.steps, PER_CONFIG_MIN_CALLS)
    timer = s.timer(n)
    timer.warm(max(args.warmup, n))
    us_list, clocks = time_config_regions(timer, sampler, world)
    e = config_entry(f"{name}[{idx}]: one 5120-hidden decoder layer (7 projections), 4-bit, "
                     f"M={M}, " + ("fused: q/k/v multi, gate/up+SiLU" if fused
                                   else "seven separate calls"),
                     us_list, s.layer_bytes, 0, clocks,
                     {"unit_of_time": "us per layer step", "calls_per_region": n,
                      "regions": PER_CONFIG_REGIONS, "launches_per_call": s.launches})
    del timer
    s.free()
    return e


def run_layer_step(args, rank, world, local_rank, sampler):
    """One decoder-layer step of the 5120-hidden layer workload."""
    import torch
    import quantized_matmul_affine_gb300 as aq

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    name, idx = parse_workload(args.workload)
    M, fused = LAYER_STEPS[name][idx]
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    s = LayerSetup(M, fused, torch, aq, l2)
    steps = max(1, min(args.steps, 4096))
    timer = s.timer(steps)
    timer.warm(args.warmup)
    _barrier(world)
    t0 = time.time()
    ms = timer.time_ms()
    clocks = sampler.window(t0, time.time())
    us = reduce_max(ms * 1e3 / steps, "cuda")

    # end to end: pinned x in, the layer's last output (down) back to the host
    x_host = torch.from_numpy(s.xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((M, 5120), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(s.x)
    n_e2e = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s.stream):
        for i in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            s.step(s.W[i % s.copies], x_dev)
            y_host.copy_(s.outs["down"], non_blocking=True)
            s.stream.synchronize()
    e2e_us = reduce_max((time.perf_counter() - t0) * 1e6 / n_e2e, "cuda")

    hbm, _, src = peaks()
    achieved = s.layer_bytes / (us * 1e-6) / 1e9
    return {
        "metric": LAYER_METRIC,
        "value": round(whole_job_us_per_call(us, world), 3),
        "unit": "us/step",
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: one 5120-hidden decoder layer (q,k,v,o,gate,up,"
                               f"down), 4-bit, M={M}, "
                               + ("fused: q/k/v multi, gate/up+SiLU" if fused
                                  else "seven separate calls"),
                   "M": M, "fused": fused,
                   "l2": f"cold: {s.copies} rotating copies of the layer's weights "
                         f"({s.copies * s.wbytes / 1e6:.0f} MB > 2x L2)",
                   "timing": f"CUDA events on the launching stream around {steps} steps "
                             f"replayed from CUDA graphs of {timer.chunk} steps",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": peak_source(src),
                     "algorithmic_bytes_per_launch": s.layer_bytes},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/step",
                "h2d_bytes_per_step": M * 5120 * 2, "d2h_bytes_per_step": M * 5120 * 2,
                "path": "pinned x -> device, the layer's calls, down output -> pinned host, sync"},
        "gpu_launches": steps * s.launches,
        "clocks": clocks,
    }


# ---------------------------------------------------------------------------
# Other code widths and group sizes
# ---------------------------------------------------------------------------

WIDTHS_METRIC = ("µs/call and effective HBM GB/s (fraction of roofline), other code widths and "
                 "group sizes, y=x·Wᵀ")
# name -> list of (bits, group, N, K, M, x dtype)
WIDTH_WORKLOADS = {"widths": [(8, 64, 4096, 4096, 1, "bf16"), (2, 32, 4096, 4096, 1, "bf16"),
                              (6, 128, 4096, 4096, 1, "bf16"), (4, 128, 4096, 4096, 1, "bf16"),
                              (8, 32, 4096, 4096, 16, "fp16"), (8, 64, 4096, 4096, 64, "bf16"),
                              (8, 64, 8192, 8192, 256, "bf16"), (5, 32, 8192, 8192, 256, "fp16"),
                              (3, 64, 10240, 5120, 256, "fp16"), (8, 32, 4096, 4096, 4, "fp16"),
                              (8, 32, 4096, 4096, 8, "fp16"), (5, 64, 4096, 4096, 16, "bf16")]}


def run_widths(args, rank, world, local_rank, sampler):
    """aq_matmul_ex on a width / group size other than the 3/4-bit group-64
    format: device-timed calls over rotating weight copies (> 2x L2) and the
    same through host buffers."""
    import torch
    import quantized_matmul_affine_gb300 as aq

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

    def call(i):
        c = i % copies
        aq.aq_matmul_ex(x, *ws[c], bits, group, out=ys[c], stream=stream)

    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    aq.aq_stats_reset()
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    used = [aq.aq_variant_name(v) for v, c in enumerate(aq.aq_stats()) if c]
    steps = max(1, min(args.steps, 4096))
    timer = GraphTimer(torch, stream, call, steps, copies, chunk_max=256)
    timer.warm(args.warmup)
    _barrier(world)
    t0 = time.time()
    ms = timer.time_ms()
    clocks = sampler.window(t0, time.time())
    us = reduce_max(ms * 1e3 / steps, "cuda")
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
    by = wbytes + 2 * M * K + 2 * M * N
    fl = 2 * M * N * K
    bound, achieved, peak, unit, frac, src = roofline_of(by, fl, us)
    return {
        "metric": WIDTHS_METRIC,
        "value": round(whole_job_us_per_call(us, world), 3),
        "unit": "us/call",
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: {bits}-bit affine group-{group}, N={N}, K={K}, "
                               f"M={M}, x {dt}",
                   "bits": bits, "group": group, "M": M, "N": N, "K": K,
                   "variant": ",".join(used),
                   "l2": f"cold: {copies} rotating weight copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {steps} calls "
                             f"replayed from CUDA graphs of {timer.chunk}",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak,
                     "unit": unit, "frac": round(frac, 4), "traffic": None,
                     "peak_source": peak_source(src),
                     "algorithmic_bytes_per_launch": by, "flops_per_launch": fl},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * M * K, "d2h_bytes_per_step": 2 * M * N,
                "path": "pinned x -> device, aq_matmul_ex, y -> pinned host, sync"},
        "gpu_launches": steps,
        "clocks": clocks,
    }


# ---------------------------------------------------------------------------
# Decode attention over a quantised KV cache
# ---------------------------------------------------------------------------

ATTN_METRIC = ("µs/call and effective HBM GB/s (fraction of roofline), decode attention over "
               "an affine-quantised KV cache")
# name -> list of (H, KV, N, D, bits, group, q dtype)
ATTN_WORKLOADS = {"attention": [(16, 8, 8192, 256, 4, 64, "bf16"), (16, 8, 2048, 256, 4, 64, "bf16"),
                                (16, 8, 32768, 256, 4, 64, "bf16"), (16, 8, 8192, 256, 8, 64, "bf16"),
                                (32, 8, 8192, 128, 4, 64, "bf16"), (16, 8, 8192, 512, 4, 64, "bf16")]}
# the same shapes through aq_attention_decode_ws (a workspace: several
# clusters a KV head)
ATTN_WORKLOADS["attnws"] = list(ATTN_WORKLOADS["attention"])


def run_attention(args, rank, world, local_rank, sampler):
    """aq_attention_decode on one decode step of a quantised KV cache:
    device-timed calls over rotating cache copies (> 2x L2) and the same
    through host buffers (q in, o out)."""
    import torch
    import quantized_matmul_affine_gb300 as aq

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
    ws_mode = name == "attnws"
    ws_bytes = aq.aq_attention_workspace_bytes(H, KV, N, D, bits, group) if ws_mode else 0
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_mode else None

    def attend(qq, cc, out):
        if ws_mode:
            aq.aq_attention_decode_ws(qq, *cc, bits, group, workspace=ws, out=out, stream=stream)
        else:
            aq.aq_attention_decode(qq, *cc, bits, group, out=out, stream=stream)

    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    qb = workloads.make_x(H, D, dt, seed=71)
    q = torch.from_numpy(qb.view(np.int16)).cuda().view(tdt)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    cbytes = 2 * (R * D * bits // 8 + 4 * R * G)
    copies = max(2, -(-2 * l2 // cbytes) + 1)
    caches = [(tuple(t.clone() for t in k0), tuple(t.clone() for t in v0)) for _ in range(copies)]
    outs = [torch.empty((H, D), dtype=tdt, device="cuda") for _ in range(copies)]
    stream = torch.cuda.Stream()

    def call(i):
        c = i % copies
        attend(q, caches[c], outs[c])

    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 4096))
    timer = GraphTimer(torch, stream, call, steps, copies, chunk_max=256)
    timer.warm(args.warmup)
    _barrier(world)
    t0 = time.time()
    ms = timer.time_ms()
    clocks = sampler.window(t0, time.time())
    us = reduce_max(ms * 1e3 / steps, "cuda")
    q_host = torch.from_numpy(qb.view(np.int16)).view(tdt).pin_memory()
    o_host = torch.empty((H, D), dtype=tdt).pin_memory()
    q_dev = torch.empty_like(q)
    n_e2e = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            q_dev.copy_(q_host, non_blocking=True)
            attend(q_dev, caches[i % copies], outs[0])
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
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{name}[{idx}]: {H} query heads over {KV} KV heads of {D}, "
                               f"{N} cached rows, {bits}-bit group-{group} K and V, q {dt}",
                   "H": H, "KV": KV, "N": N, "D": D, "bits": bits, "group": group,
                   "l2": f"cold: {copies} rotating cache copies > 2x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA events on the launching stream around {steps} calls "
                             f"replayed from CUDA graphs of {timer.chunk}",
                   "launch": (aq.aq_attention_describe_ws(H, KV, N, D, bits, group, ws_bytes)
                              if ws_mode else aq.aq_attention_describe(H, KV, N, D, bits, group)),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": attn_traffic,
                     "peak_source": peak_source(src),
                     "algorithmic_bytes_per_launch": by},
        "e2e": {"value": round(whole_job_us_per_call(e2e_us, world), 3), "unit": "us/call",
                "h2d_bytes_per_step": 2 * H * D, "d2h_bytes_per_step": 2 * H * D,
                "path": "pinned q -> device, "
                        + ("aq_attention_decode_ws" if ws_mode else "aq_attention_decode")
                        + ", o -> pinned host, sync"},
        "gpu_launches": steps,
        "clocks": clocks,
    }


# ---------------------------------------------------------------------------
# The oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_columns_time(p, words, x, ncols, threads, rng):
    """Seconds for the oracle to compute `ncols` output columns (a random
    contiguous window, every activation row) on `threads` threads."""
    import oracle
    start = int(rng.integers(0, p.N - ncols + 1))
    c = slice(start, start + ncols)
    sub = np.ascontiguousarray(words[c])
    t0 = time.perf_counter()
    oracle.matmul(x, sub, p.scales[c], p.biases[c], p.bits, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(p, budget_s):
    """The oracle as it stands, timed on the host: all cores, then one core,
    each on a window of output columns sized to about budget_s/2 seconds and
    scaled by N / columns to one full call."""
    import oracle
    oracle.build()
    words = oracle.pack(p.codes, p.bits)
    x = p.x_f64()
    rng = np.random.default_rng(0)
    threads = os.cpu_count() or 1
    cal = min(p.N, 16)
    t_col = oracle_columns_time(p, words, x, cal, 1, rng) / cal  # one core, per column
    out = {}
    for name, th, floor in (("all_cores", threads, threads), ("one_core", 1, 1)):
        want = int((budget_s / 2) / max(t_col / th, 1e-9))
        if name == "one_core" and p.N >= 1024:
            want = max(want, 1024)
        ncols = int(min(p.N, max(floor, want)))
        dt = oracle_columns_time(p, words, x, ncols, th, rng)
        out[name] = {"value": round(dt * p.N / ncols * 1e6, 1), "unit": "us/call",
                     "cores": th, "kind": "oracle",
                     "sample": f"{ncols} of {p.N} output columns (all {p.M} rows), scaled by "
                               f"N/{ncols}" + ("" if ncols == p.N else " (extrapolated)")
                               + f"; {th} thread{'s' if th > 1 else ''}"}
    line = dict(out["all_cores"])
    line["one_core"] = out["one_core"]
    return line


def run_reference(args, rank, world):
    """The oracle on the host cores, as the reference arm: each step computes
    a random window of output columns on all cores and is scaled to a full
    call; the window is sized so the whole run takes about --ref-budget s."""
    import oracle
    oracle.build()
    name, idx = parse_workload(args.workload)
    p = workloads.workload(name, idx)
    words = oracle.pack(p.codes, p.bits)
    x = p.x_f64()
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    cal = min(p.N, max(threads, 16))
    t_col = oracle_columns_time(p, words, x, cal, threads, rng) / cal
    total = args.steps + args.warmup
    per_step_budget = args.ref_budget / max(1, total)
    ncols = int(min(p.N, max(threads, per_step_budget / max(t_col, 1e-9))))
    step_times = []
    for i in range(total):
        dt = oracle_columns_time(p, words, x, ncols, threads, rng)
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
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help=f"one workload alone (default: {DEFAULT_WORKLOAD} with per_config)")
    ap.add_argument("--cpu-budget", type=float, default=24.0,
                    help="seconds of host time for the cpu_baseline legs")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of host time for the whole reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all", action="store_true", help="one line per workload (not the default)")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only: skip the hot-L2, end-to-end and CPU legs")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the torch.matmul comparison leg of the matmul workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    per_config = args.workload is None and not args.all
    if args.workload is None:
        args.workload = DEFAULT_WORKLOAD

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    import torch
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    sampler = ClockSampler.for_device(torch, torch.cuda.current_device()).start()

    specs = [args.workload]
    if args.all:
        specs = [f"{n}:{i}" for n, c in workloads.WORKLOADS.items() for i in range(len(c))]
    try:
        for spec in specs:
            args.workload = spec
            kind = parse_workload(spec)[0]
            if kind in ATTN_WORKLOADS:
                line = run_attention(args, rank, world, local_rank, sampler)
            elif kind in WIDTH_WORKLOADS:
                line = run_widths(args, rank, world, local_rank, sampler)
            elif kind in LAYER_STEPS:
                line = run_layer_step(args, rank, world, local_rank, sampler)
            elif kind in workloads.QUANTIZE_WORKLOADS:
                line = run_quantize(args, rank, world, local_rank, sampler)
            else:
                line, p = run_ours(args, rank, world, local_rank, sampler, per_config)
                if (rank == 0 and world == 1 and not args.no_cpu_baseline and not args.all
                        and not args.quick):
                    line["cpu_baseline"] = cpu_baseline(p, args.cpu_budget)
            if rank == 0:
                print(json.dumps(line), flush=True)
    finally:
        sampler.stop()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

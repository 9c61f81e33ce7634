#!/usr/bin/env python
"""Throughput of the W4A4 + LoRA linear layer on GB300.

One step = the four linears of a Qwen3-style 1024-hidden decoder layer at
M = 700 tokens (qkv 1024->4096, o 2048->1024, gate_up 1024->6144,
down 3072->1024; group 64, LoRA rank 32), each as the path's two kernels:
w4a4_quantize_act (quantise + LoRA down) and w4a4_linear (GEMM + LoRA up +
column affine).  Weight packing is offline (done once, untimed).

Inputs are seeded synthetic data (synthetic.make_linear_case).  To keep the
timed inputs out of L2, the step cycles through R replicas of the layer
(distinct buffers, > 2x the 129 MB L2 in total).

Prints one JSON line (metric: effective TOPS = (2MNK + 2Mr(K+N)) / time).
  --impl reference : the CPU oracle timed on the host cores (bounded sample).
  --workload stack : instead, the 28-layer stack of those four linears with
                     RMSNorm glue (112 linears, one CUDA graph per forward pass).
  --workload decode : the small-M sweep, M in {1, 4, 16, 32, 76}, K = N = 4096.
  --workload prefill : the two M = 8192 prefill linears (4096->14336, 14336->4096).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import DECODER_LAYER_M700, make_linear_case  # noqa: E402
from w4a4_quantized_gemm_gb300 import metrics  # noqa: E402

METRIC = "W4A4+LoRA linear effective TOPS (decoder-layer linears, M=700)"
UNIT = "TOPS"
WORKLOAD = "qwen3_1024_decoder_layer_linears_M700"
STACK_METRIC = "W4A4+LoRA linear effective TOPS (28-layer stack, M=700, RMSNorm glue, CUDA graph)"
STACK_WORKLOAD = "qwen3_1024_28_layer_stack_M700"
PREFILL_METRIC = "W4A4+LoRA linear effective TOPS (prefill, M=8192: 4096->14336 and 14336->4096)"
PREFILL_WORKLOAD = "prefill_M8192_K4096_N14336_and_K14336_N4096"
L2_BYTES = 129 * 2 ** 20


def max_over_ranks(x: float, dev, world: int) -> float:
    """The largest of every rank's x: a job's time is its slowest rank's."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput (units per second): every rank runs its own replica of
    the step (weak scaling), and the step takes the slowest rank's time."""
    return world * units_per_rank_step / (ms_per_step * 1e-3)


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def int8_dense_peak_tops():
    """cuBLAS int8 GEMM throughput (torch._int_mm, 8192^3, best of 3 x 5 calls), in TOPS, or None.

    The spec fraction is quoted against the INT8 dense tensor rate, which
    this GPU runs far below its fp8 rate; the path itself uses the fp8 kind, so
    `roofline.peak` stays the fp8 dense rate and this is reported beside it."""
    import torch
    try:
        n = 8192
        a = torch.randint(-64, 64, (n, n), dtype=torch.int8, device="cuda")
        b = torch.randint(-64, 64, (n, n), dtype=torch.int8, device="cuda").t().contiguous().t()
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                torch._int_mm(a, b)
            e1.record()
            torch.cuda.synchronize()
            best = max(best, 5 * 2 * n ** 3 / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        del a, b
        return best
    except Exception:  # an int8 GEMM the library does not offer here: report nothing
        return None


def layer_ops() -> int:
    return sum(metrics.linear_ops(s["M"], s["N"], s["K"], s["r"]) for s in DECODER_LAYER_M700.values())


def base_config(extra=None):
    cfg = {"workload": WORKLOAD, "M": 700, "group": 64, "rank": 32,
           "linears": {k: [v["K"], v["N"]] for k, v in DECODER_LAYER_M700.items()}}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------- CPU oracle
def time_oracle(budget_s: float, max_rows: int = 700, chunk: int = 16):
    """Run the oracle on row chunks of every linear until `budget_s` elapses.
    Returns (ops done, seconds, rows per linear)."""
    import oracle
    oracle.build()
    cases = {k: make_linear_case(seed=i, **v) for i, (k, v) in enumerate(DECODER_LAYER_M700.items())}
    ops, rows, t0 = 0, 0, time.perf_counter()
    while rows < max_rows:
        n = min(chunk, max_rows - rows)
        for c in cases.values():
            oracle.linear(c.X[rows:rows + n], c.W, c.L_down, c.L_up, c.colscale, c.bias)
            ops += metrics.linear_ops(n, c.N, c.K, c.r)
        rows += n
        if time.perf_counter() - t0 >= budget_s:
            break
    return ops, time.perf_counter() - t0, rows


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    # each step: the oracle on a bounded row sample of every linear
    rows_per_step = args.ref_rows
    steps = []
    import oracle
    oracle.build()
    cases = {k: make_linear_case(seed=i, **v) for i, (k, v) in enumerate(DECODER_LAYER_M700.items())}
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        ops = 0
        r0 = (i * rows_per_step) % (700 - rows_per_step)
        for c in cases.values():
            oracle.linear(c.X[r0:r0 + rows_per_step], c.W, c.L_down, c.L_up, c.colscale, c.bias)
            ops += metrics.linear_ops(rows_per_step, c.N, c.K, c.r)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            steps.append((ops, dt))
    ops = sum(o for o, _ in steps)
    sec = sum(t for _, t in steps)
    value = ops / sec / 1e12
    sample = f"{rows_per_step} of 700 rows of each of the 4 linears per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64",
        "data": "synthetic", "config": base_config({"sample": sample}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) of the SM clock and the throttle
    reasons while the benchmark runs.  The caller keeps the GPU under the timed
    load for the whole sampling window (an untimed pre-roll of the same work,
    then the timed region, marked with mark_start / mark_end)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, inside = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
            if self.t_start is not None and self.t_end is not None and self.t_start <= t <= self.t_end:
                inside += 1
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unavailable"], "samples": 0}
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}
        if self.t_start is not None and self.t_end is not None:
            out.update(samples_in_timed_region=inside,
                       window="untimed pre-roll of the timed work, then the timed region")
        return out


def preroll(replay, seconds: float = 0.5, sync=None) -> int:
    """Untimed replays of the timed work for `seconds`, so that the GPU is under
    that load while the clock sampler starts (synchronising every 16 replays
    keeps the launch queue short).  Returns the number of replays."""
    if sync is None:
        import torch
        sync = torch.cuda.synchronize
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < seconds:
        replay(i)
        i += 1
        if i % 16 == 0:
            sync()
    sync()
    return i


# ------------------------------------------------------------ host and ncu facts
def host_cpu():
    """nproc and the CPU model name of this host (lscpu), for the oracle baseline."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def kernel_source_hash(name: str) -> str:
    """sha256 (first 16 hex digits) of one CUDA source file of the library."""
    import hashlib
    with open(os.path.join(ROOT, "w4a4_quantized_gemm_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the GEMM launches
# of one step, from the ncu capture summarised under profiles/, keyed by the
# hash of the kernel source they were taken on: once the kernel changes, the
# counters no longer describe it and traffic is reported as null.
NCU_TRAFFIC = {
    # the four decoder-layer GEMM launches (qkv, o, gate_up, down) at M = 700, one launch each,
    # read from HBM (24 input replicas cycled): 3,501,056 + 3,065,856 + 4,747,520 + 4,507,904 bytes read,
    # none written; Y stays in L2 within a launch (profiles/gemm_tc_traffic_decoder_layer_m700.md)
    (WORKLOAD, "958dd4c4b0f2e294"): {
        "bytes_per_pass": 15822336,
        "per_linear": {"qkv": 3501056, "o": 3065856, "gate_up": 4747520, "down": 4507904},
        "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch per linear "
                  "(profiles/gemm_tc_traffic_decoder_layer_m700.md)"},
    # the M = 8192 GEMMs, two launches per linear (the full rounds, then the last round split over K):
    # 4096 -> 14336 71.77 + 14.70 MB read, 208.04 MB written; 14336 -> 4096 160.96 + 37.75 MB read,
    # 53.07 MB written (profiles/gemm_tc_prefill_m8192.md)
    (PREFILL_WORKLOAD, "958dd4c4b0f2e294"): {
        "bytes_per_pass": 294509824 + 251788288,
        "per_linear": {"gate_up_style": 294509824, "down_style": 251788288},
        "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, both launches of each linear "
                  "(profiles/gemm_tc_prefill_m8192.md)"},
}


def gemm_launches(dispatch: str) -> int:
    """GEMM launches one w4a4_linear call makes (two when its last round of tiles runs split over K)."""
    return 2 if "round-robin, last" in dispatch else 1


def ncu_traffic(workload: str, source: str = "gemm_tc.cu"):
    rec = NCU_TRAFFIC.get((workload, kernel_source_hash(source)))
    return dict(rec) if rec else None


def step_stats(ms):
    """median, p10 and p90 of per-step times (ms)."""
    a = np.asarray(ms, np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "n": int(a.size)}


def decode_sweep(w4, dev, steps: int, warmup: int, Ms=(1, 4, 16, 32), R: int = 20, hbm: float = 6800.0):
    """The small-M calls (K = N = 4096, r = 32): per M, the whole call through
    w4a4_forward (from fp16 X to Y: the fused kernel up to M = 8, quantise + GEMM
    above), the same two steps as separate calls, and the GEMM alone, each in a
    CUDA graph over R weight replicas (> L2), so the weights come from HBM.
    GB/s = packed weights + scales (the bytes every call must stream) / time."""
    import torch
    from synthetic import SMALL_M_SWEEP
    base = make_linear_case(seed=0, **SMALL_M_SWEEP[-1])
    W = torch.from_numpy(base.W).to(dev)
    Ld = torch.from_numpy(base.L_down.view(np.float16).copy()).to(dev)
    Lu = torch.from_numpy(base.L_up.view(np.float16).copy()).to(dev)
    packed0 = torch.empty(w4.packed_weights_bytes(base.N, base.K, base.r), dtype=torch.uint8, device=dev)
    w4.w4a4_pack_weights(W, Ld, Lu, packed0, base.r)
    del W
    packs = [packed0.clone() for _ in range(R)]
    cs = torch.from_numpy(base.colscale.view(np.float16).copy()).to(dev)
    b = torch.from_numpy(base.bias.view(np.float16).copy()).to(dev)
    wbytes = metrics.weight_bytes(base.N, base.K)
    out = {}
    for M in Ms:
        X = torch.from_numpy(base.X[:M].view(np.float16).copy()).to(dev)
        ws = torch.empty(w4.act_workspace_bytes(M, base.K, base.r), dtype=torch.uint8, device=dev)
        Y = torch.empty((M, base.N), dtype=torch.float16, device=dev)
        w4.w4a4_quantize_act(X, packs[0], ws, base.r)
        w4.w4a4_linear(ws, packs[0], cs, b, Y, base.K, base.r)
        disp = w4.w4a4_last_dispatch()
        w4.w4a4_forward(X, packs[0], cs, b, Y, base.r, act_ws=ws)
        disp_f = w4.w4a4_last_dispatch()
        torch.cuda.synchronize()
        gf, gw, gg = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf):
            for p_ in packs:
                w4.w4a4_forward(X, p_, cs, b, Y, base.r, act_ws=ws, stream=torch.cuda.current_stream())
        with torch.cuda.graph(gw):
            for p_ in packs:
                st = torch.cuda.current_stream()
                w4.w4a4_quantize_act(X, p_, ws, base.r, st)
                w4.w4a4_linear(ws, p_, cs, b, Y, base.K, base.r, w4.KERNEL_AUTO, st)
        with torch.cuda.graph(gg):
            for p_ in packs:
                w4.w4a4_linear(ws, p_, cs, b, Y, base.K, base.r, w4.KERNEL_AUTO, torch.cuda.current_stream())
        torch.cuda.synchronize()

        def tm(graph):
            for _ in range(max(warmup, 3)):
                graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (steps * R)

        uf, uw, ug = tm(gf), tm(gw), tm(gg)
        out[M] = {"whole_call_us": uf, "whole_call_gbs": wbytes / (uf * 1e-6) / 1e9, "whole_call_dispatch": disp_f,
                  "two_calls_us": uw, "two_calls_gbs": wbytes / (uw * 1e-6) / 1e9,
                  "gemm_us": ug, "gemm_gbs": wbytes / (ug * 1e-6) / 1e9, "dispatch": disp}
    low = min(out, key=lambda m: out[m]["whole_call_gbs"])
    return {"per_M": out, "min_whole_call_gbs": out[low]["whole_call_gbs"], "at_M": low,
            "frac_hbm": out[low]["whole_call_gbs"] / hbm, "hbm_gbs": hbm, "weight_bytes_per_call": wbytes,
            "what": "whole call = one w4a4_forward from fp16 X (K = N = 4096, r = 32) per weight replica "
                    "(two_calls: w4a4_quantize_act + w4a4_linear); "
                    f"{R} replicas, {R * wbytes / 2**20:.0f} MiB > L2; min over M <= 32 is the headline"}


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from w4a4_quantized_gemm_gb300 import build as wbuild
    wbuild.build()
    import w4a4_quantized_gemm_gb300 as w4

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    names = list(DECODER_LAYER_M700)
    R = args.replicas
    L = {}
    for i, name in enumerate(names):
        s = DECODER_LAYER_M700[name]
        c = make_linear_case(seed=i, **s)
        X = torch.from_numpy(c.X.view(np.float16).copy()).to(dev)
        W = torch.from_numpy(c.W).to(dev)
        Ld = torch.from_numpy(c.L_down.view(np.float16).copy()).to(dev)
        Lu = torch.from_numpy(c.L_up.view(np.float16).copy()).to(dev)
        cs = torch.from_numpy(c.colscale.view(np.float16).copy()).to(dev)
        b = torch.from_numpy(c.bias.view(np.float16).copy()).to(dev)
        packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device=dev)
        w4.w4a4_pack_weights(W, Ld, Lu, packed, c.r)
        del W
        wsb = w4.act_workspace_bytes(c.M, c.K, c.r)
        L[name] = dict(
            c=c, X=[X.clone() for _ in range(R)], packed=[packed.clone() for _ in range(R)],
            cs=[cs.clone() for _ in range(R)], b=[b.clone() for _ in range(R)],
            ws=[torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in range(R)],
            Y=[torch.empty((c.M, c.N), dtype=torch.float16, device=dev) for _ in range(R)])
    torch.cuda.synchronize()
    footprint = sum(sum(t.numel() * t.element_size() for k in ("X", "packed", "ws", "Y") for t in d[k])
                    for d in L.values())

    def step(i, timers=None):
        rep = i % R
        for name in names:
            d = L[name]
            c = d["c"]
            if timers is not None:
                timers[name][0].record(stream)
            w4.w4a4_quantize_act(d["X"][rep], d["packed"][rep], d["ws"][rep], c.r, stream)
            if timers is not None:
                timers[name][1].record(stream)
            w4.w4a4_linear(d["ws"][rep], d["packed"][rep], d["cs"][rep], d["b"][rep], d["Y"][rep], c.K, c.r,
                           w4.KERNEL_AUTO, stream)
            if timers is not None:
                timers[name][2].record(stream)

    dispatch = {}
    for i in range(max(args.warmup, R)):  # every replica once (first-call kernel attributes set here)
        step(i)
    for name in names:  # record the kernel each linear uses
        d = L[name]
        w4.w4a4_linear(d["ws"][0], d["packed"][0], d["cs"][0], d["b"][0], d["Y"][0], d["c"].K, d["c"].r)
        dispatch[name] = w4.w4a4_last_dispatch()
    torch.cuda.synchronize()

    # One CUDA graph per replica holding one step's 8 launches (the pages' own
    # remedy for launch overhead, "W4A4 CUDA Kernel for Voice Clone", section 4).
    def capture(fn):
        graphs = []
        for rep in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(rep, torch.cuda.current_stream())
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs

    def step_on(rep, st):
        for name in names:
            d = L[name]
            c = d["c"]
            w4.w4a4_quantize_act(d["X"][rep], d["packed"][rep], d["ws"][rep], c.r, st)
            w4.w4a4_linear(d["ws"][rep], d["packed"][rep], d["cs"][rep], d["b"][rep], d["Y"][rep], c.K, c.r,
                           w4.KERNEL_AUTO, st)

    step_graphs = capture(step_on)

    def timed(graphs, steps):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # A step is P passes of the layer (each on the next replica), P chosen so that
    # the K timed steps last at least --min-timed-s: long enough for the clock
    # sampler (one sample per 200 ms) to see the timed region itself.
    t_pass = timed(step_graphs, 4 * R) / (4 * R)
    P = max(1, int(np.ceil(args.min_timed_s * 1e3 / (args.steps * t_pass))))

    def timed_steps(steps):
        for i in range(args.warmup * P):
            step_graphs[i % R].replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record()
        for k in range(steps):
            for j in range(P):
                step_graphs[(k * P + j) % R].replay()
            ev[k + 1].record()
        torch.cuda.synchronize()
        per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
        return ev[0].elapsed_time(ev[steps]), per

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.__enter__()
    preroll(lambda i: step_graphs[i % len(step_graphs)].replay())
    if sampler:
        sampler.mark_start()
    ms, per_step = timed_steps(args.steps)
    if sampler:
        sampler.mark_end()
        sampler.__exit__()
    ms = max_over_ranks(ms, dev, world)
    if world > 1:
        dist.barrier()
    ms_per_step = ms / args.steps
    value = job_rate(world, P * layer_ops(), ms_per_step) / 1e12
    stats = step_stats(per_step)
    stats.update({f"{k}_tops": P * layer_ops() / (stats[k] * 1e-3) / 1e12 for k in ("median", "p10", "p90")})

    # per-kernel durations.  Per step: one graph per replica holding the step's
    # four GEMMs (or four activation kernels), the same buffers as the step.
    # Per linear: one graph holding that linear's kernel over all R replicas
    # (per launch = graph time / R; the replicas of one linear may sit in L2).
    def launch(name, kind, rep, st):
        d = L[name]
        c = d["c"]
        if kind == "q":
            w4.w4a4_quantize_act(d["X"][rep], d["packed"][rep], d["ws"][rep], c.r, st)
        else:
            w4.w4a4_linear(d["ws"][rep], d["packed"][rep], d["cs"][rep], d["b"][rep], d["Y"][rep], c.K, c.r,
                           w4.KERNEL_AUTO, st)

    def kind_step(kind):
        return lambda rep, st: [launch(n, kind, rep, st) for n in names]

    def one_linear(name, kind):
        return lambda rep, st: [launch(name, kind, j, st) for j in range(R)]

    reps = max(args.steps, 2 * R)
    q_s = timed(capture(kind_step("q")), reps) / reps * 1e-3
    gemm_s = timed(capture(kind_step("g")), reps) / reps * 1e-3
    lin_reps = max(4, reps // R)
    q_us = {n: 1e3 * timed(capture(one_linear(n, "q"))[:1], lin_reps) / (lin_reps * R) for n in names}
    g_us = {n: 1e3 * timed(capture(one_linear(n, "g"))[:1], lin_reps) / (lin_reps * R) for n in names}
    # the gate_up linear with the SiLU(gate) * up epilogue (fused gate|up weights packed in
    # the epilogue's order, H [M, N/2] out), on the same activations, against its plain GEMM
    gu = L["gate_up"]
    cgu = gu["c"]
    Wgu = torch.from_numpy(cgu.W).to(dev)
    pk_silu = torch.empty_like(gu["packed"][0])
    w4.w4a4_pack_weights_gate_up(Wgu, torch.from_numpy(cgu.L_down.view(np.float16).copy()).to(dev),
                                 torch.from_numpy(cgu.L_up.view(np.float16).copy()).to(dev), pk_silu, cgu.r)
    del Wgu
    pks_silu = [pk_silu.clone() for _ in range(R)]
    Hs = [torch.empty((cgu.M, cgu.N // 2), dtype=torch.float16, device=dev) for _ in range(R)]
    w4.w4a4_linear_silu_mul(gu["ws"][0], pks_silu[0], gu["cs"][0], gu["b"][0], Hs[0], cgu.K, cgu.r)
    silu_dispatch = w4.w4a4_last_dispatch()
    silu_graph = capture(lambda rep, st: [w4.w4a4_linear_silu_mul(gu["ws"][j], pks_silu[j], gu["cs"][j], gu["b"][j],
                                                                   Hs[j], cgu.K, cgu.r, st) for j in range(R)])
    silu_us = 1e3 * timed(silu_graph[:1], lin_reps) / (lin_reps * R)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    if "bf16_tflops" in peaks:
        bf16, peak_src = float(peaks["bf16_tflops"]), "measured"
    else:
        bf16, peak_src = 1900.0, "fallback"
    fp8_peak = 2.0 * bf16  # FP8 tensor kind: measured bf16 burst x nominal fp8/bf16 ratio (4.5/2.25)
    achieved = layer_ops() / gemm_s / 1e12
    traffic = ncu_traffic(WORKLOAD)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": traffic["bytes_per_pass"] if traffic else None,
                "traffic_source": traffic["source"] if traffic else
                "null: no ncu capture of the current gemm_tc.cu source",
                "kernel": "w4a4_linear (GEMM + LoRA up + affine), 4 launches per layer pass",
                "peak_source": f"{peak_src} bf16 burst x 2 (fp8 kind)",
                "gemm_us_per_step": gemm_s * 1e6, "quantize_us_per_step": q_s * 1e6,
                "per_linear_gemm_us": g_us, "per_linear_quantize_us": q_us,
                "gate_up_silu_mul_us": silu_us, "gate_up_silu_mul_dispatch": silu_dispatch,
                "gemm_algorithmic_bytes": sum(metrics.gemm_bytes(**DECODER_LAYER_M700[n]) for n in names),
                "quantize_algorithmic_bytes": sum(metrics.act_bytes(DECODER_LAYER_M700[n]["M"],
                                                                    DECODER_LAYER_M700[n]["K"],
                                                                    DECODER_LAYER_M700[n]["r"]) for n in names)}
    roofline["quantize_gbs"] = roofline["quantize_algorithmic_bytes"] / q_s / 1e9
    i8 = int8_dense_peak_tops()
    roofline["int8_dense_tops_measured"] = i8
    roofline["frac_of_int8_dense"] = achieved / i8 if i8 else None

    # end to end through the public API: pinned host X in, Y back to pinned host (graph of copies + calls)
    e2e = None
    if not args.no_e2e:
        # A step's four inputs sit back to back in one pinned host buffer and in one device
        # buffer per replica, and so do its four outputs (qkv first): the copy engines move
        # a few large copies per step at close to their peak, where eight copies of 1.4-8.6 MB
        # ran at 90-180 GB/s.
        xsz = {n: L[n]["X"][0].numel() for n in names}
        ysz = {n: L[n]["Y"][0].numel() for n in names}
        Xh_all = torch.empty(sum(xsz.values()), dtype=torch.float16).pin_memory()
        Yh_all = torch.empty(sum(ysz.values()), dtype=torch.float16).pin_memory()
        XA = [torch.empty(sum(xsz.values()), dtype=torch.float16, device=dev) for _ in range(R)]
        YA = [torch.empty(sum(ysz.values()), dtype=torch.float16, device=dev) for _ in range(R)]

        def split(buf, sizes, like):
            out, o = {}, 0
            for n in names:
                out[n] = buf[o:o + sizes[n]].view(like[n].shape)
                o += sizes[n]
            return out

        Xv = [split(XA[rep], xsz, {n: L[n]["X"][0] for n in names}) for rep in range(R)]
        Yv = [split(YA[rep], ysz, {n: L[n]["Y"][0] for n in names}) for rep in range(R)]
        Xhv = split(Xh_all, xsz, {n: L[n]["X"][0] for n in names})
        for n in names:
            Xhv[n].copy_(L[n]["X"][0])
        h2d = Xh_all.numel() * 2
        d2h = Yh_all.numel() * 2
        first = names[0]
        rest_off = ysz[first]

        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        # The copies run on side streams and are pipelined across the E = 4R steps of one
        # graph (step k on replica k % R): the inputs are copied in ahead (one copy per step;
        # each step waits for its own, and a replica's input buffer is refilled only once the
        # step before on it has been quantised), the first linear's Y is copied out while the
        # other three compute, the other three Ys in one copy while the next step computes (a
        # replica's outputs are rewritten only once that copy has landed), and the graph ends
        # once the last copy has landed.  Every step copies its own inputs in and its own
        # outputs out inside the timed region.
        E = 4 * R

        def e2e_steps(_, st):
            start = torch.cuda.Event()
            start.record(st)
            s_in.wait_event(start)
            s_out.wait_event(start)
            arrived, consumed, copied = [], [], []
            for k in range(E):
                rep = k % R
                with torch.cuda.stream(s_in):
                    if k >= R:
                        s_in.wait_event(consumed[k - R])
                    XA[rep].copy_(Xh_all, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    arrived.append(ev)
                st.wait_event(arrived[k])
                if k >= R:
                    st.wait_event(copied[k - R])
                for n in names:
                    d = L[n]
                    c = d["c"]
                    w4.w4a4_quantize_act(Xv[rep][n], d["packed"][rep], d["ws"][rep], c.r, st)
                    if n == names[-1]:
                        ev = torch.cuda.Event()
                        ev.record(st)
                        consumed.append(ev)
                    w4.w4a4_linear(d["ws"][rep], d["packed"][rep], d["cs"][rep], d["b"][rep], Yv[rep][n], c.K,
                                   c.r, w4.KERNEL_AUTO, st)
                    if n == first or n == names[-1]:
                        done = torch.cuda.Event()
                        done.record(st)
                        s_out.wait_event(done)
                        with torch.cuda.stream(s_out):
                            if n == first:
                                Yh_all[:rest_off].copy_(YA[rep][:rest_off], non_blocking=True)
                            else:
                                Yh_all[rest_off:].copy_(YA[rep][rest_off:], non_blocking=True)
                                ev = torch.cuda.Event()
                                ev.record(s_out)
                                copied.append(ev)
            st.wait_stream(s_in)
            st.wait_stream(s_out)

        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_steps(0, torch.cuda.current_stream())
        torch.cuda.synchronize()
        reps_e2e = max(2, (args.steps + E - 1) // E)
        e_ms = max_over_ranks(timed([g_e2e], reps_e2e) / (reps_e2e * E), dev, world)
        e2e = {"value": job_rate(world, layer_ops(), e_ms) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "how": f"one CUDA graph of {E} steps over {R} replicas: per step, one H2D of the 4 inputs X (back to back in "
                      "pinned host memory; copy stream, all issued at the start, each step waits for its own), "
                      "the two C-ABI calls per linear, then on a second copy stream one D2H of the first "
                      "linear's Y while the others compute and one D2H of the other three Ys while the next "
                      "step computes; the graph ends when the last copy has landed"}

    # the small-M half of the metric: whole calls (activation kernel + GEMM) at M <= 32
    decode = None
    if not args.no_decode:
        hbm = float(peaks["hbm_gbs"]) if "hbm_gbs" in peaks else 6800.0
        decode = decode_sweep(w4, dev, max(args.steps, 20), args.warmup, hbm=hbm)
        decode["peak_source"] = "measured HBM copy bandwidth" if "hbm_gbs" in peaks else "fallback"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ops, sec, rows = time_oracle(args.cpu_budget)
        cpu = {"value": ops / sec / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of each of the 4 linears ({ops / 1e9:.2f} Gop, {sec:.1f} s)",
               **host_cpu()}

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    clocks = sampler.summary() if sampler else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 codes (fp8 e4m3 operands), fp32 accumulate, fp16 out",
        "data": "synthetic",
        "config": base_config({"replicas": R, "l2": f"inputs larger than L2: {footprint / 2**20:.0f} MiB cycled",
                               "passes_per_step": P, "dispatch": dispatch}),
        "step_ms": stats, "ms_per_pass": ms_per_step / P,
        "gpu_launches": args.steps * P * sum(1 + gemm_launches(dispatch[n]) for n in names),
        "roofline": roofline, "decode": decode, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ config 5: stack
def stack_ops(M: int = 700) -> int:
    from synthetic import STACK_LAYERS, STACK_LINEARS
    return STACK_LAYERS * sum(metrics.linear_ops(M, N, K, 32) for _, K, N in STACK_LINEARS)


def stack_config(extra=None):
    from synthetic import STACK_LAYERS, STACK_LINEARS
    cfg = {"workload": STACK_WORKLOAD, "M": 700, "group": 64, "rank": 32, "layers": STACK_LAYERS,
           "linears_per_layer": {n: [k, nn] for n, k, nn in STACK_LINEARS},
           "glue": "RMSNorm (unit gain, eps 1e-6, fp64-defined) of the columns the next linear reads, fused into "
                   "the next linear's activation kernel; the last output normalised by the glue kernel"}
    if extra:
        cfg.update(extra)
    return cfg


def time_stack_oracle(budget_s: float, max_rows: int = 8):
    """The oracle's chain through all 112 linears for a few rows, until the budget."""
    import oracle
    from synthetic import STACK_LAYERS, STACK_LINEARS, make_stack_input, make_stack_linear
    oracle.build()
    X = make_stack_input(700)[:max_rows]
    rows, ops, t0 = 0, 0, time.perf_counter()
    nl = len(STACK_LINEARS)
    for n in (1, 1, 2, 4):
        if rows >= max_rows or time.perf_counter() - t0 >= budget_s:
            break
        x = X[rows:rows + n]
        for i in range(STACK_LAYERS * nl):
            c = make_stack_linear(i // nl, i % nl)
            y = oracle.linear(x, c.W, c.L_down, c.L_up, c.colscale, c.bias)
            x = oracle.rmsnorm_f16(oracle.f64_to_f16_array(y), STACK_LINEARS[(i + 1) % nl][1])
            ops += metrics.linear_ops(n, c.N, c.K, c.r)
        rows += n
    return ops, time.perf_counter() - t0, rows


def run_stack_reference(args, rank, world):
    if rank != 0:
        return 0
    steps = []
    for i in range(args.warmup + args.steps):
        ops, sec, rows = time_stack_oracle(1e9, max_rows=1)
        if i >= args.warmup:
            steps.append((ops, sec))
    ops = sum(o for o, _ in steps)
    sec = sum(t for _, t in steps)
    value = ops / sec / 1e12
    sample = "1 of 700 rows through all 112 linears and their RMSNorm glue per step"
    print(json.dumps({
        "impl": "reference", "metric": STACK_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64",
        "data": "synthetic", "config": stack_config({"sample": sample}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def _reference_line(args, world, metric, unit, value, sec_per_step, config, sample):
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64",
        "data": "synthetic", "config": dict(config, sample=sample),
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_prefill_reference(args, rank, world, rows_per_step=2):
    """The oracle on the prefill workload: each step, `rows_per_step` rows of
    both M = 8192 linears (every call quantises the whole weight matrix)."""
    if rank != 0:
        return 0
    import oracle
    from synthetic import PREFILL
    oracle.build()
    cases = [make_linear_case(seed=i, **s) for i, s in enumerate(PREFILL.values())]
    ops, sec = 0, 0.0
    for i in range(args.warmup + args.steps):
        r0 = (i * rows_per_step) % (8192 - rows_per_step)
        t0 = time.perf_counter()
        for c in cases:
            oracle.linear(c.X[r0:r0 + rows_per_step], c.W, c.L_down, c.L_up, c.colscale, c.bias)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            ops += sum(metrics.linear_ops(rows_per_step, c.N, c.K, c.r) for c in cases)
            sec += dt
    config = {"workload": PREFILL_WORKLOAD, "M": 8192, "group": 64, "rank": 32,
              "linears": {n: [s["K"], s["N"]] for n, s in PREFILL.items()}}
    print(json.dumps(_reference_line(args, world, PREFILL_METRIC, UNIT, ops / sec / 1e12, sec / args.steps, config,
                                     f"{rows_per_step} of 8192 rows of both linears per step")), flush=True)
    return 0


def run_decode_reference(args, rank, world):
    """The oracle on the small-M sweep: each step, the whole M = 32 call (of the
    sweep's M <= 32, the one with the most work per weight byte, so the lowest
    bandwidth: the metric's binding case)."""
    if rank != 0:
        return 0
    import oracle
    from synthetic import SMALL_M_SWEEP
    oracle.build()
    c = make_linear_case(seed=0, **SMALL_M_SWEEP[-1])
    wbytes = metrics.weight_bytes(c.N, c.K)
    sec = 0.0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.linear(c.X[:32], c.W, c.L_down, c.L_up, c.colscale, c.bias)
        if i >= args.warmup:
            sec += time.perf_counter() - t0
    config = {"workload": "small_m_sweep_K4096_N4096", "group": 64, "rank": 32}
    value = wbytes * args.steps / sec / 1e9
    print(json.dumps(_reference_line(args, world, DECODE_METRIC, "GB/s", value, sec / args.steps, config,
                                     "the M = 32 call of the sweep, whole, per step")), flush=True)
    return 0


def run_stack(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from w4a4_quantized_gemm_gb300 import build as wbuild
    wbuild.build()
    import w4a4_quantized_gemm_gb300 as w4
    from synthetic import STACK_LAYERS, STACK_LINEARS, make_stack_input, make_stack_linear
    from w4a4_quantized_gemm_gb300.stack import W4A4Stack

    dev = torch.device("cuda", local_rank)
    nl = len(STACK_LINEARS)
    stack = W4A4Stack((make_stack_linear(l, j) for l in range(STACK_LAYERS) for j in range(nl)), 700, dev)
    X0h = torch.from_numpy(make_stack_input(700).view(np.float16).copy())
    stack.X0.copy_(X0h.to(dev))
    weight_bytes = sum(L["packed"].numel() for L in stack.layers)
    fwd = stack.capture()

    def gemm_only(st):
        for i, L in enumerate(stack.layers):
            w4.w4a4_linear(L["ws"], L["packed"], L["cs"], L["b"], L["Y"], L["K"], L["r"], w4.KERNEL_AUTO, st)

    def quant_only(st):  # the activation step of every linear (with the RMSNorm where it is fused)
        for i, L in enumerate(stack.layers):
            if stack.reads_previous_output(i):
                w4.w4a4_quantize_act_rmsnorm(stack.layers[i - 1]["Y"], L["K"], L["packed"], L["ws"], L["r"], st)
            else:
                w4.w4a4_quantize_act(L["X"], L["packed"], L["ws"], L["r"], st)

    def glue_only(st):  # the separate RMSNorm launches that remain
        for i in range(len(stack.layers)):
            if stack.has_glue(i):
                stack.run_glue(i, st)

    stack.forward()
    torch.cuda.synchronize()
    parts = {}
    for name, fn in (("gemm", gemm_only), ("quantize", quant_only), ("glue", glue_only)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        torch.cuda.synchronize()
        parts[name] = g
    g_gemm = parts["gemm"]

    def timed(graph, steps):
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.__enter__()
    preroll(lambda i: fwd.replay())
    if sampler:
        sampler.mark_start()
    ms = timed(fwd, args.steps)
    if sampler:
        sampler.mark_end()
        sampler.__exit__()
    ms = max_over_ranks(ms, dev, world)
    ms_per_step = ms / args.steps
    ops = stack_ops()
    value = job_rate(world, ops, ms_per_step) / 1e12
    gemm_s = timed(g_gemm, args.steps) / args.steps * 1e-3
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    bf16, peak_src = (float(peaks["bf16_tflops"]), "measured") if "bf16_tflops" in peaks else (1900.0, "fallback")
    achieved = ops / gemm_s / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": 2.0 * bf16, "unit": "TFLOP/s",
                "frac": achieved / (2.0 * bf16), "traffic": None,
                "kernel": "w4a4_linear (GEMM + LoRA up + affine), 112 launches per forward",
                "peak_source": f"{peak_src} bf16 burst x 2 (fp8 kind)",
                "gemm_us_per_step": gemm_s * 1e6, "forward_us": ms_per_step * 1e3,
                "quantize_us_per_step": timed(parts["quantize"], args.steps) / args.steps * 1e3,
                "glue_us_per_step": timed(parts["glue"], args.steps) / args.steps * 1e3,
                "packed_weight_bytes": weight_bytes}
    i8 = int8_dense_peak_tops()
    roofline["int8_dense_tops_measured"] = i8
    roofline["frac_of_int8_dense"] = achieved / i8 if i8 else None

    e2e = None
    if not args.no_e2e:
        Xh = X0h.pin_memory()
        Oh = torch.empty_like(stack.out, device="cpu").pin_memory()
        g_e2e = torch.cuda.CUDAGraph()
        stack.forward()
        torch.cuda.synchronize()
        with torch.cuda.graph(g_e2e):
            stack.X0.copy_(Xh, non_blocking=True)
            stack.forward(torch.cuda.current_stream())
            Oh.copy_(stack.out, non_blocking=True)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(timed(g_e2e, args.steps) / args.steps, dev, world)
        e2e = {"value": job_rate(world, ops, e_ms) / 1e12, "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": Xh.numel() * 2, "d2h_bytes_per_step": Oh.numel() * 2,
               "how": "one CUDA graph: H2D of the stack input from pinned host, the 336 C-ABI launches, D2H of the output"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c_ops, c_sec, c_rows = time_stack_oracle(args.cpu_budget)
        cpu = {"value": c_ops / c_sec / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{c_rows} of 700 rows through all 112 linears and their glue ({c_sec:.1f} s)"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    print(json.dumps({
        "metric": STACK_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 codes (fp8 e4m3 operands), fp32 accumulate, fp16 out",
        "data": "synthetic",
        "config": stack_config({"l2": f"packed weights {weight_bytes / 2**20:.0f} MiB > L2, streamed every pass"}),
        "gpu_launches": args.steps * stack.launches_per_forward(),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": sampler.summary() if sampler else None}), flush=True)
    return 0


# ------------------------------------------------------- config 3: small M
DECODE_METRIC = "W4A4+LoRA linear packed-weight GB/s of the whole call (K=N=4096, small M; min over M<=32)"


def run_decode(args, rank, world, local_rank):
    """Config 3: M in {1, 4, 16, 32, 76}, K = N = 4096.  Each timed GEMM call
    reads a different replica of the packed weights (20 replicas > L2), so the
    weights come from HBM; value = the lowest weight bandwidth over M <= 32
    (with N ranks: every rank streams its own weights, the job's bandwidth)."""
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from w4a4_quantized_gemm_gb300 import build as wbuild
    wbuild.build()
    import w4a4_quantized_gemm_gb300 as w4
    from synthetic import SMALL_M_SWEEP

    dev = torch.device("cuda", local_rank)
    R = 20
    results = {}
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm, hbm_src = (float(peaks["hbm_gbs"]), "measured") if "hbm_gbs" in peaks else (6800.0, "fallback")
    base = make_linear_case(seed=0, **SMALL_M_SWEEP[-1])
    W = torch.from_numpy(base.W).to(dev)
    Ld = torch.from_numpy(base.L_down.view(np.float16).copy()).to(dev)
    Lu = torch.from_numpy(base.L_up.view(np.float16).copy()).to(dev)
    packed0 = torch.empty(w4.packed_weights_bytes(base.N, base.K, base.r), dtype=torch.uint8, device=dev)
    w4.w4a4_pack_weights(W, Ld, Lu, packed0, base.r)
    del W
    packs = [packed0.clone() for _ in range(R)]
    # the same weights as asymmetric group-128 codes (fp16 scale + zero point), for the W4A16 variant
    W = torch.from_numpy(base.W).to(dev)
    packed_a = torch.empty_like(packed0)
    w4.w4a16_pack_weights_asym(W, Ld, Lu, packed_a, base.r)
    packs_a = [packed_a.clone() for _ in range(R)]
    # LoRA from the quantisation error (offline): one K=N=4096, r=32 layer, 3 rounds, 16 power steps
    torch.cuda.synchronize()
    t_svd = time.perf_counter()
    _, _, svd_errs = w4.w4a4_pack_weights_svd(W, base.r, torch.empty_like(packed0), rounds=3, power_iters=16)
    torch.cuda.synchronize()
    svd_s = time.perf_counter() - t_svd
    del W
    cs = torch.from_numpy(base.colscale.view(np.float16).copy()).to(dev)
    b = torch.from_numpy(base.bias.view(np.float16).copy()).to(dev)
    wbytes = metrics.weight_bytes(base.N, base.K)
    sampler = ClockSampler(local_rank)
    sampler.__enter__()
    e2e = None
    for s_ in SMALL_M_SWEEP:
        M = s_["M"]
        X = torch.from_numpy(base.X[:M].view(np.float16).copy()).to(dev)
        ws = torch.empty(w4.act_workspace_bytes(M, base.K, base.r), dtype=torch.uint8, device=dev)
        Y = torch.empty((M, base.N), dtype=torch.float16, device=dev)
        w4.w4a4_quantize_act(X, packs[0], ws, base.r)
        w4.w4a4_linear(ws, packs[0], cs, b, Y, base.K, base.r)
        disp = w4.w4a4_last_dispatch()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for p_ in packs:
                w4.w4a4_linear(ws, p_, cs, b, Y, base.K, base.r, w4.KERNEL_AUTO, torch.cuda.current_stream())
        gq = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gq):
            for p_ in packs:
                w4.w4a4_quantize_act(X, p_, ws, base.r, torch.cuda.current_stream())
        torch.cuda.synchronize()
        def tm(graph):
            for _ in range(max(args.warmup, 3)):
                graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (args.steps * R)
        gw = torch.cuda.CUDAGraph()  # the W4A16 linear on the same weights: fp16 X straight in, one kernel
        with torch.cuda.graph(gw):
            for p_ in packs:
                w4.w4a16_linear(X, p_, cs, b, Y, base.r, torch.cuda.current_stream())
        ga = torch.cuda.CUDAGraph()  # the W4A16 linear on asymmetric group-128 weights
        with torch.cuda.graph(ga):
            for p_ in packs_a:
                w4.w4a16_linear_asym(X, p_, cs, b, Y, base.r, torch.cuda.current_stream())
        torch.cuda.synchronize()
        us, uq, uw, ua = (max_over_ranks(tm(x), dev, world) for x in (g, gq, gw, ga))
        gbs = job_rate(world, wbytes, us * 1e-3) / 1e9
        results[M] = {"gemm_us": us, "quantize_us": uq, "weight_gbs": gbs,
                      "frac_hbm": gbs / (world * hbm), "dispatch": disp,
                      "w4a16_linear_us": uw, "w4a16_weight_gbs": job_rate(world, wbytes, uw * 1e-3) / 1e9,
                      "w4a16_asym_g128_us": ua, "w4a16_asym_g128_weight_gbs": job_rate(world, wbytes, ua * 1e-3) / 1e9}
        if M == 32 and not args.no_e2e:
            # end to end through the public API at the metric's binding M: pinned host X in, the two
            # C-ABI calls per weight replica, Y back to pinned host, all in one graph
            Xh = torch.empty((M, base.K), dtype=torch.float16).pin_memory()
            Xh.copy_(X.cpu())
            Yh = torch.empty((M, base.N), dtype=torch.float16).pin_memory()
            Xd = [torch.empty_like(X) for _ in packs]
            Yd = [torch.empty_like(Y) for _ in packs]
            s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge):
                st = torch.cuda.current_stream()
                start = torch.cuda.Event()
                start.record(st)
                s_in.wait_event(start)
                s_out.wait_event(start)
                arrived = []
                with torch.cuda.stream(s_in):  # every call's input copied in from the start
                    for j in range(len(packs)):
                        Xd[j].copy_(Xh, non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(s_in)
                        arrived.append(ev)
                for j, p_ in enumerate(packs):
                    st.wait_event(arrived[j])
                    w4.w4a4_forward(Xd[j], p_, cs, b, Yd[j], base.r, act_ws=ws, stream=st)
                    done = torch.cuda.Event()
                    done.record(st)
                    s_out.wait_event(done)
                    with torch.cuda.stream(s_out):  # each result copied out while the next call computes
                        Yh.copy_(Yd[j], non_blocking=True)
                st.wait_stream(s_in)
                st.wait_stream(s_out)
            torch.cuda.synchronize()
            ue = max_over_ranks(tm(ge), dev, world)
            e2e = {"value": job_rate(world, wbytes, ue * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": M * base.K * 2,
                   "d2h_bytes_per_step": M * base.N * 2, "us_per_call": ue, "M": M,
                   "how": "per call: H2D of X from pinned host (copy stream), w4a4_forward through the C-ABI, "
                          "D2H of Y (second copy stream, overlapping the next call); CUDA graph over the weight "
                          "replicas"}
    # whole calls (activation kernel + GEMM back to back): the headline
    whole = decode_sweep(w4, dev, args.steps, args.warmup, Ms=tuple(s_["M"] for s_ in SMALL_M_SWEEP), R=R, hbm=hbm)
    sampler.__exit__()
    for m_, v in whole["per_M"].items():
        v["whole_call_us"] = max_over_ranks(v["whole_call_us"], dev, world)
        v["whole_call_gbs"] = job_rate(world, wbytes, v["whole_call_us"] * 1e-3) / 1e9
        results[m_].update(whole_call_us=v["whole_call_us"], whole_call_gbs=v["whole_call_gbs"],
                           frac_hbm_whole_call=v["whole_call_gbs"] / (world * hbm),
                           whole_call_dispatch=v["whole_call_dispatch"], two_calls_us=v["two_calls_us"])
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    low = min(v["whole_call_gbs"] for m, v in results.items() if m <= 32)
    low_gemm = min(v["weight_gbs"] for m, v in results.items() if m <= 32)
    m32 = results[32]
    print(json.dumps({
        "metric": DECODE_METRIC, "value": low, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m32["whole_call_us"] * 1e-3, "higher_is_better": True,
        "scaling": "weak", "gemm_only_min_gbs": low_gemm,
        "vs_baseline": None, "dtype": "int4 codes (fp8 e4m3 operands), fp32 accumulate, fp16 out",
        "data": "synthetic",
        "config": {"workload": "small_m_sweep_K4096_N4096", "group": 64, "rank": 32, "replicas": R,
                   "l2": f"{R} weight replicas, {R * wbytes / 2**20:.0f} MiB > L2", "per_M": results,
                   "svd_lora": {"seconds_per_layer": svd_s, "rounds": 3, "power_iters": 16,
                                "residual_per_round": svd_errs,
                                "what": "w4a4_pack_weights_svd on the K=N=4096 weights, r=32 (offline)"}},
        "gpu_launches": args.steps * R * sum(1 if "linear_fused" in v.get("whole_call_dispatch", "") else 2
                                             for v in results.values()),
        "e2e": e2e, "clocks": sampler.summary(),
        "roofline": {"bound": "hbm", "achieved": low_gemm / world, "peak": hbm, "unit": "GB/s",
                     "frac": low_gemm / world / hbm, "traffic": None,
                     "kernel": "w4a4_linear (small-M weight-streaming kernel; the value above is the whole call)",
                     "peak_source": f"{hbm_src} HBM copy bandwidth",
                     "algorithmic_bytes_per_call": wbytes}}), flush=True)
    return 0


def run_prefill(args, rank, world, local_rank):
    """Config 4: one step = the gate/up-style (K=4096, N=14336) and the down-style
    (K=14336, N=4096) linear at M = 8192, each as quantize + GEMM.  Every step
    writes 470 MB of Y, so no input stays in L2 from one step to the next; two
    replicas of every buffer are cycled all the same."""
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from w4a4_quantized_gemm_gb300 import build as wbuild
    wbuild.build()
    import w4a4_quantized_gemm_gb300 as w4
    from synthetic import PREFILL

    dev = torch.device("cuda", local_rank)
    names = list(PREFILL)
    R = 2
    L = {}
    for i, name in enumerate(names):
        c = make_linear_case(seed=i, **PREFILL[name])
        W = torch.from_numpy(c.W).to(dev)
        Ld = torch.from_numpy(c.L_down.view(np.float16).copy()).to(dev)
        Lu = torch.from_numpy(c.L_up.view(np.float16).copy()).to(dev)
        packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device=dev)
        w4.w4a4_pack_weights(W, Ld, Lu, packed, c.r)
        del W
        X = torch.from_numpy(c.X.view(np.float16).copy()).to(dev)
        cs = torch.from_numpy(c.colscale.view(np.float16).copy()).to(dev)
        b = torch.from_numpy(c.bias.view(np.float16).copy()).to(dev)
        wsb = w4.act_workspace_bytes(c.M, c.K, c.r)
        L[name] = dict(c=c, X=[X] + [X.clone() for _ in range(R - 1)],
                       packed=[packed] + [packed.clone() for _ in range(R - 1)], cs=cs, b=b,
                       ws=[torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in range(R)],
                       Y=[torch.empty((c.M, c.N), dtype=torch.float16, device=dev) for _ in range(R)])
    torch.cuda.synchronize()
    ops = sum(metrics.linear_ops(PREFILL[n]["M"], PREFILL[n]["N"], PREFILL[n]["K"], PREFILL[n]["r"]) for n in names)
    footprint = sum(sum(t.numel() * t.element_size() for k in ("X", "packed", "ws", "Y") for t in d[k])
                    for d in L.values())

    def launch(name, kind, rep, st, Xsrc=None):
        d = L[name]
        c = d["c"]
        if kind in ("q", "qg"):
            w4.w4a4_quantize_act(d["X"][rep] if Xsrc is None else Xsrc, d["packed"][rep], d["ws"][rep], c.r, st)
        if kind in ("g", "qg"):
            w4.w4a4_linear(d["ws"][rep], d["packed"][rep], d["cs"], d["b"], d["Y"][rep], c.K, c.r,
                           w4.KERNEL_AUTO, st)

    dispatch = {}
    for rep in range(R):
        for n in names:
            launch(n, "qg", rep, torch.cuda.current_stream())
            dispatch[n] = w4.w4a4_last_dispatch()
    torch.cuda.synchronize()

    def capture(fn):
        graphs = []
        for rep in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(rep, torch.cuda.current_stream())
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs

    def timed(graphs, steps):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    step_graphs = capture(lambda rep, st: [launch(n, "qg", rep, st) for n in names])
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.__enter__()
    preroll(lambda i: step_graphs[i % len(step_graphs)].replay())
    if sampler:
        sampler.mark_start()
    ms = timed(step_graphs, args.steps)
    if sampler:
        sampler.mark_end()
        sampler.__exit__()
    ms_per_step = max_over_ranks(ms, dev, world) / args.steps
    value = job_rate(world, ops, ms_per_step) / 1e12

    # per linear: graphs holding that linear's GEMM (or activation kernel) alone, replicas alternating
    g_us = {n: 1e3 * timed(capture(lambda rep, st, n=n: launch(n, "g", rep, st)), args.steps) / args.steps
            for n in names}
    q_us = {n: 1e3 * timed(capture(lambda rep, st, n=n: launch(n, "q", rep, st)), args.steps) / args.steps
            for n in names}
    gemm_s = sum(g_us.values()) * 1e-6
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    if "bf16_tflops" in peaks:
        bf16, peak_src = float(peaks["bf16_tflops"]), "measured"
    else:
        bf16, peak_src = 1900.0, "fallback"
    fp8_peak = 2.0 * bf16  # FP8 tensor kind: measured bf16 burst x nominal fp8/bf16 ratio (4.5/2.25)
    achieved = ops / gemm_s / 1e12
    traffic = ncu_traffic(PREFILL_WORKLOAD)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": traffic["bytes_per_pass"] if traffic else None,
                "traffic_per_linear": traffic["per_linear"] if traffic else None,
                "traffic_source": traffic["source"] if traffic else
                "null: no ncu capture of the current gemm_tc.cu source",
                "kernel": "w4a4_linear (GEMM + LoRA up + affine), "
                          f"{sum(gemm_launches(dispatch[n]) for n in names)} launches per step",
                "peak_source": f"{peak_src} bf16 burst x 2 (fp8 kind)",
                "per_linear_gemm_us": g_us, "per_linear_quantize_us": q_us,
                "per_linear_gemm_tops": {n: metrics.linear_ops(PREFILL[n]["M"], PREFILL[n]["N"], PREFILL[n]["K"],
                                                               PREFILL[n]["r"]) / (g_us[n] * 1e-6) / 1e12
                                         for n in names},
                "gemm_algorithmic_bytes": sum(metrics.gemm_bytes(**PREFILL[n]) for n in names),
                "quantize_algorithmic_bytes": sum(metrics.act_bytes(PREFILL[n]["M"], PREFILL[n]["K"],
                                                                    PREFILL[n]["r"]) for n in names)}
    roofline["quantize_gbs"] = roofline["quantize_algorithmic_bytes"] / (sum(q_us.values()) * 1e-6) / 1e9
    i8 = int8_dense_peak_tops()
    roofline["int8_dense_tops_measured"] = i8
    roofline["frac_of_int8_dense"] = achieved / i8 if i8 else None

    # end to end through the public API: pinned host X in (copy stream), the two C-ABI calls per
    # linear once its X has landed, Y back to pinned host (second copy stream)
    e2e = None
    if not args.no_e2e:
        Xh = {n: torch.empty_like(L[n]["X"][0], device="cpu").pin_memory() for n in names}
        Yh = {n: torch.empty_like(L[n]["Y"][0], device="cpu").pin_memory() for n in names}
        for n in names:
            Xh[n].copy_(L[n]["X"][0])
        h2d = sum(Xh[n].numel() * 2 for n in names)
        d2h = sum(Yh[n].numel() * 2 for n in names)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        # pipelined across the E = 4R steps of one graph (step k on replica k % R), as in the
        # layer workload: a replica's input is refilled only once the step before on it has
        # read it, its output rewritten only once that output has been copied out; every step
        # copies its own inputs in and its own outputs out inside the timed region
        E = 4 * R

        def e2e_steps(st):
            start = torch.cuda.Event()
            start.record(st)
            s_in.wait_event(start)
            s_out.wait_event(start)
            arrived, consumed, copied = {}, {}, {}
            for k in range(E):
                rep = k % R
                with torch.cuda.stream(s_in):
                    for n in names:
                        if k >= R:
                            s_in.wait_event(consumed[k - R, n])
                        L[n]["X"][rep].copy_(Xh[n], non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(s_in)
                        arrived[k, n] = ev
                for n in names:
                    st.wait_event(arrived[k, n])
                    if k >= R:
                        st.wait_event(copied[k - R, n])
                    launch(n, "qg", rep, st)
                    done = torch.cuda.Event()
                    done.record(st)
                    consumed[k, n] = done
                    s_out.wait_event(done)
                    with torch.cuda.stream(s_out):
                        Yh[n].copy_(L[n]["Y"][rep], non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(s_out)
                        copied[k, n] = ev
            st.wait_stream(s_in)
            st.wait_stream(s_out)

        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_steps(torch.cuda.current_stream())
        torch.cuda.synchronize()
        reps_e2e = max(2, (args.steps + E - 1) // E)
        e_ms = max_over_ranks(timed([g_e2e], reps_e2e) / (reps_e2e * E), dev, world)
        e2e = {"value": job_rate(world, ops, e_ms) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "how": f"one CUDA graph of {E} steps over {R} replicas: per step, H2D of both inputs X from pinned "
                      "host (copy stream, ahead of the compute; each linear waits for its own), the two C-ABI calls "
                      "per linear, D2H of each Y on a second copy stream while the following linear (of this step "
                      "or the next) computes; the graph ends when the last copy has landed"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        done, rows, t0 = 0, 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_budget and rows < 64:
            for n in names:
                c = L[n]["c"]
                oracle.linear(c.X[rows:rows + 4], c.W, c.L_down, c.L_up, c.colscale, c.bias)
                done += metrics.linear_ops(4, c.N, c.K, c.r)
            rows += 4
        sec = time.perf_counter() - t0
        cpu = {"value": done / sec / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of both linears, 4 rows per call ({done / 1e9:.1f} Gop, {sec:.1f} s)"}

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 codes (fp8 e4m3 operands), fp32 accumulate, fp16 out",
        "data": "synthetic",
        "config": {"workload": PREFILL_WORKLOAD, "M": 8192, "group": 64, "rank": 32,
                   "linears": {n: [PREFILL[n]["K"], PREFILL[n]["N"]] for n in names}, "replicas": R,
                   "l2": f"inputs larger than L2: {footprint / 2**20:.0f} MiB cycled", "dispatch": dispatch},
        "gpu_launches": args.steps * sum(1 + gemm_launches(dispatch[n]) for n in names),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": sampler.summary() if sampler else None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="layer workload: skip the small-M sub-record")
    ap.add_argument("--min-timed-s", type=float, default=0.5,
                    help="layer workload: passes per step chosen so that the timed steps last at least this long")
    ap.add_argument("--workload", choices=["layer", "stack", "decode", "prefill"], default="layer")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.workload == "decode":
        if args.impl == "reference":
            return run_decode_reference(args, rank, world)
        return run_decode(args, rank, world, local_rank)
    if args.workload == "prefill":
        if args.impl == "reference":
            return run_prefill_reference(args, rank, world)
        return run_prefill(args, rank, world, local_rank)
    if args.workload == "stack":
        if args.impl == "reference":
            return run_stack_reference(args, rank, world)
        return run_stack(args, rank, world, local_rank)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())

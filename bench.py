"""Benchmark of the FP4 block-scaled quantized linear hot path on GB300.

One step = the whole hot path over one batch of the 1.2B Transformer FFN
workload (T = 8192 tokens; linears 2048 -> 6144 and 6144 -> 2048): for each
linear, the five quantized operands (X rowwise and X^T colwise + RHT16 from one
pass over X, W 16x16 in both orientations, dY rowwise SR and dY^T colwise +
RHT16 + SR from one pass over dY; each preceded by its tensor amax, computed on
a second stream while the previous operand is converted) and the three
block-scaled NVFP4 GEMMs (Fprop, Dgrad, Wgrad).

`value` is fwd+bwd GEMM TFLOP/s of the whole step (6 T N K per linear divided
by the step time, quantization included) with inputs resident in HBM; `e2e`
is the same metric through the public API (Fp4Linear.step_host) with the
inputs copied from pinned host memory and the outputs copied back inside the
timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1.2b|8b|12b|tiny]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample
    python bench.py --kernels              # single library calls, each against its roofline
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP4 linear fwd+bwd TFLOP/s; quantize GB/s (% of FP4/HBM roofline)"
# Nominal dense-rate ratio FP4 : BF16 on GB300 (13.5 : 2.25 PFLOP/s).
FP4_OVER_BF16 = 6.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Algorithmic bytes per input element of the step's quantizations, current
# scaling (one amax pass and one conversion pass over the BF16 input, E2M1 codes
# plus one 8-bit scale per 16 values written per operand): X and dY each yield a
# rowwise and a colwise operand, W yields W and W^T -- all 2 * 2 + 2 * (1/2 + 1/16).
BYTES_TWO_OPERANDS = 5.125


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle sample
_INPUT_CACHE: dict = {}


def oracle_sample(workload, tokens: int = 16, feats: int = 256) -> dict:
    """Time the oracle on a bounded sample of one step: for every linear, the
    first `tokens` tokens and the first `feats` output and input features.
    Quantization covers X and dY on those tokens (rowwise and colwise + RHT16)
    and the W / W^T rows the sampled GEMM outputs need (with the tensor amax of
    the whole weight); the three GEMMs produce Y[tokens x feats],
    dX[tokens x feats] (summing over all N) and dW[feats x feats]. Returns the
    GEMM FLOPs covered and the elapsed seconds."""
    import oracle
    from workloads import linear_inputs

    oracle.build()
    flops, elapsed = 0.0, 0.0
    for which, lin in enumerate(workload.linears):
        key = (workload.name, which)
        if key not in _INPUT_CACHE:
            _INPUT_CACHE[key] = linear_inputs(workload, which)
        inp = _INPUT_CACHE[key]
        Ts, Fs = tokens, feats
        x = inp["x"][:Ts].copy()
        dy = inp["dy"][:Ts].copy()
        t0 = time.perf_counter()
        qx = oracle.quantize(x, tensor_id=8 * which + 0)
        qxt = oracle.quantize(x, colwise=True, rht=True, seed=workload.rht_seed, tensor_id=8 * which + 1,
                              op_rows=(0, Fs))
        qw = oracle.quantize(inp["w"], block=oracle.BLOCK_16x16, tensor_id=8 * which + 2, op_rows=(0, Fs))
        qwt = oracle.quantize(inp["w"], block=oracle.BLOCK_16x16, colwise=True, tensor_id=8 * which + 2,
                              op_rows=(0, Fs))
        qdy = oracle.quantize(dy, sr=True, seed=workload.sr_seed, tensor_id=8 * which + 3)
        qdyt = oracle.quantize(dy, colwise=True, rht=True, sr=True, seed=workload.sr_seed,
                               tensor_id=8 * which + 4, op_rows=(0, Fs))
        oracle.gemm(qx["codes"], qx["scales"], qx["s_dec"], qw["codes"], qw["scales"], qw["s_dec"])
        oracle.gemm(qdy["codes"], qdy["scales"], qdy["s_dec"], qwt["codes"], qwt["scales"], qwt["s_dec"])
        oracle.gemm(qdyt["codes"], qdyt["scales"], qdyt["s_dec"], qxt["codes"], qxt["scales"], qxt["s_dec"])
        elapsed += time.perf_counter() - t0
        flops += 2.0 * (Ts * Fs * lin.k_in + Ts * Fs * lin.n_out + Fs * Fs * Ts)
    return {"flops": flops, "seconds": elapsed}


def cpu_baseline_entry(workload, tokens: int, feats: int, min_seconds: float = 10.0) -> dict:
    flops = secs = 0.0
    reps = 0
    while secs < min_seconds and reps < 20:
        s = oracle_sample(workload, tokens, feats)
        flops += s["flops"]
        secs += s["seconds"]
        reps += 1
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x (every linear of the step on {tokens} tokens and {feats} x {feats} output/input "
                      f"features: quantizations of those slices plus the three GEMMs), single-threaded C oracle, "
                      f"{secs:.1f} s"}


# --------------------------------------------------------------------------- distributed
def dist_setup():
    """One process per GPU (torchrun env vars). Replicas only: the ranks exchange
    nothing but a barrier and the max of their timings. NCCL on GPUs, gloo on CPU."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
        return dist, dist.get_rank(), world
    return None, 0, 1


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- reference arm
def run_reference(args, workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    times, flops = [], 0.0
    for _ in range(args.warmup):
        oracle_sample(workload, args.ref_tokens, args.ref_feats)
    for _ in range(args.steps):
        s = oracle_sample(workload, args.ref_tokens, args.ref_feats)
        times.append(s["seconds"])
        flops = s["flops"]
    total = sum(times)
    value = flops * len(times) / total / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (oracle)", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": workload.name, "sample_tokens": args.ref_tokens,
                       "sample_features": args.ref_feats},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: every linear on {args.ref_tokens} tokens and "
                                       f"{args.ref_feats} x {args.ref_feats} features, single-threaded C oracle"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, workload):
    import numpy as np
    import torch

    import fp4_block_scaled_02_gb300 as fb
    from workloads import linear_inputs

    dist, rank, world = dist_setup()
    dev = torch.cuda.current_device()
    fb._lib.load()
    stream = torch.cuda.current_stream()

    # inputs: seeded synthetic BF16, uploaded once (resident in HBM)
    layers, host = [], []
    for which, lin in enumerate(workload.linears):
        inp = linear_inputs(workload, which)
        dev_in = {k: torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16) for k, v in inp.items()}
        L = fb.Fp4Linear(lin.tokens, lin.k_in, lin.n_out, rht=workload.rht, seed=workload.rht_seed, layer=which)
        outs = {"y": torch.empty((lin.tokens, lin.n_out), dtype=torch.bfloat16, device="cuda"),
                "dx": torch.empty((lin.tokens, lin.k_in), dtype=torch.bfloat16, device="cuda"),
                "dw": torch.empty((lin.n_out, lin.k_in), dtype=torch.float32, device="cuda")}
        layers.append((lin, L, dev_in, outs))
        host.append({k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
                     for k, v in inp.items()})

    gemm_flops = sum(3 * 2.0 * lin.tokens * lin.k_in * lin.n_out for lin, *_ in layers)
    quant_bytes = sum(BYTES_TWO_OPERANDS * (lin.tokens * (lin.k_in + lin.n_out) + lin.n_out * lin.k_in)
                      for lin, *_ in layers)
    # per linear: 3 x (amax + quantize) + 3 GEMMs; with the amaxes on a side
    # stream, each amax launch becomes two (tile pass + finalize)
    launches_per_step = sum(12 if L.side is not None else 9 for _, L, _, _ in layers)
    q_launches = launches_per_step - 3 * len(layers)

    def step(ev=None):
        for lin, L, di, o in layers:
            if ev is not None:
                ev.append(torch.cuda.Event(enable_timing=True))
                ev[-1].record(stream)
            L.quantize_all(di["x"], di["w"], di["dy"], stream=stream)
            if ev is not None:
                ev.append(torch.cuda.Event(enable_timing=True))
                ev[-1].record(stream)
            L.gemms(o["y"], o["dx"], o["dw"], stream=stream)
            if ev is not None:
                ev.append(torch.cuda.Event(enable_timing=True))
                ev[-1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = fb.fp4_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    # ---- device-resident timed region
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, start.elapsed_time(end))
    # the quantize / GEMM split for the roofline: the same steps again with
    # events between the groups (kept out of the timed steps above: an event
    # between two kernels stops the second from launching early)
    evs = []
    for _ in range(args.steps):
        step(evs)
    torch.cuda.synchronize()
    clk = clocks.stop()
    q_ms = sum(evs[i].elapsed_time(evs[i + 1]) for i in range(0, len(evs), 3))
    g_ms = sum(evs[i + 1].elapsed_time(evs[i + 2]) for i in range(0, len(evs), 3))
    ms_step = ms / args.steps
    value = world * gemm_flops / (ms_step * 1e-3) / 1e12
    gemm_tflops = gemm_flops * args.steps / (g_ms * 1e-3) / 1e12
    quant_gbs = quant_bytes * args.steps / (q_ms * 1e-3) / 1e9
    status = fb.fp4_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # ---- end to end through the public API: pinned host inputs in, outputs back
    h2d = sum(t.numel() * t.element_size() for h in host for t in h.values())
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
                for (_, _, _, o) in layers]
    d2h = sum(t.numel() * t.element_size() for h in host_out for t in h.values())

    # Fp4Linear.step_host: input copies, the step and output copies on their own
    # streams, so one linear's copies overlap the other's compute
    def e2e_step():
        for (lin, L, di, o), h, ho in zip(layers, host, host_out):
            L.step_host(h["x"], h["w"], h["dy"], ho["y"], ho["dx"], ho["dw"], stream=stream)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _, L, _, _ in layers:
        L.h2d_stream.wait_event(e0)  # no copy starts before the timed region
    for _ in range(args.steps):
        e2e_step()
    for _, L, _, _ in layers:
        stream.wait_event(L.ev_out)  # ... and the last output copies end inside it
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * gemm_flops / (e_ms * 1e-3) / 1e12

    if rank != 0:
        return
    peaks, src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    hbm_peak = peaks["hbm_gbs"]
    traffic = load_traffic()
    gemm_roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": fp4_peak, "unit": "TFLOP/s",
                 "frac": gemm_tflops / fp4_peak, "traffic": traffic.get("gemm"),
                 "peak_source": f"{src} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)",
                 "kernel": "gemm_nvfp4_kernel (6 launches per step)"}
    quant_roof = {"bound": "hbm", "achieved": quant_gbs, "peak": hbm_peak, "unit": "GB/s",
                  "frac": quant_gbs / hbm_peak, "traffic": traffic.get("quantize"),
                  "peak_source": f"{src} hbm_gbs",
                  "kernel": f"amax + quantize kernels ({q_launches} launches per step)"}
    dominant, other = (gemm_roof, quant_roof) if g_ms >= q_ms else (quant_roof, gemm_roof)
    cpu = cpu_baseline_entry(workload, args.ref_tokens, args.ref_feats) if not args.no_cpu_baseline else None
    lin_desc = [[l.k_in, l.n_out] for l in workload.linears]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload.name, "tokens": workload.linears[0].tokens, "linears_k_n": lin_desc,
                   "recipe": "NVFP4: 1x16 E4M3 acts/grads, 16x16 weights, current scaling, SR on dY, "
                             "RHT16 on Wgrad inputs",
                   "l2": "inputs larger than L2 (%.0f MB of BF16 inputs per step)" % (h2d / 1e6),
                   "parallelism": f"replicas x{world}"},
        "gemm_tflops": gemm_tflops, "quantize_gbs": quant_gbs,
        "ms_gemm_per_step": g_ms / args.steps, "ms_quantize_per_step": q_ms / args.steps,
        "roofline": dominant, "roofline_other": other,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def load_traffic() -> dict:
    """Per-launch DRAM bytes from the committed ncu summary (profiles/traffic.json), if present."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f)
        except (OSError, ValueError):
            pass
    return {}


# --------------------------------------------------------------------------- per-kernel timings
def run_kernels(args):
    """`--kernels`: median CUDA-event time of single library calls (10 reps, L2
    flushed before each by writing 256 MB), with each call's roofline fraction:
    GEMMs against the FP4 dense peak (the emulated UE5M3 path against BF16),
    quantizer calls against the HBM copy peak with their algorithmic bytes.
    GEMM operands are random codes with block scales of moderate size; quantizer
    inputs random normal BF16. `--only REGEX` keeps the calls whose key matches
    (for a profiler capture of one kind of call). Prints one JSON line."""
    import torch

    import fp4_block_scaled_02_gb300 as fb

    fb._lib.load()
    torch.manual_seed(0)
    peaks, src = load_peaks()
    fp4_peak, bf16_peak, hbm_peak = peaks["bf16_tflops"] * FP4_OVER_BF16, peaks["bf16_tflops"], peaks["hbm_gbs"]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def time_ms(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ts.sort()
        return ts[len(ts) // 2]

    def operand(rows, cols, fmt, per_row=False):
        t = fb.QTensor.empty(rows, cols, fmt, per_row=per_row)
        t.codes.copy_(torch.randint(0, 256, t.codes.shape, dtype=torch.uint8, device="cuda"))
        lo = {fb.FP4_SCALE_E4M3: 0x30, fb.FP4_SCALE_UE5M3: 0x70, fb.FP4_SCALE_UE8M0: 0x7C}[fmt]
        t.scales.copy_(torch.randint(lo, lo + 16, t.scales.shape, dtype=torch.uint8, device="cuda"))
        t.s_dec.fill_(1.0)
        return t

    res = {}
    gemms = [("nvfp4", fb.FP4_SCALE_E4M3, "8b_fprop", (8192, 21504, 4096)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "8b_dgrad", (8192, 4096, 21504)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "8b_wgrad", (21504, 4096, 8192)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "12b_fprop", (8192, 12288, 4608)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "12b_dgrad", (8192, 4608, 12288)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "1p2b_fprop", (8192, 6144, 2048)),
             ("nvfp4", fb.FP4_SCALE_E4M3, "1p2b_dgrad", (8192, 2048, 6144)),
             ("nvfp4_rowscale", fb.FP4_SCALE_E4M3, "1p2b_fprop", (8192, 6144, 2048)),
             ("mxfp4", fb.FP4_SCALE_UE8M0, "8b_fprop", (8192, 21504, 4096)),
             ("mxfp4", fb.FP4_SCALE_UE8M0, "1p2b_fprop", (8192, 6144, 2048)),
             ("ue5m3_emulated", fb.FP4_SCALE_UE5M3, "sweep", (8192, 4096, 4096)),
             ("ue5m3_rebiased", fb.FP4_SCALE_UE5M3, "sweep", (8192, 4096, 4096))]
    only = re.compile(args.only) if args.only else None

    def wanted(key):
        return only is None or only.search(key) is not None

    for kind, fmt, name, (M, N, K) in gemms:
        if not wanted(f"gemm_{kind}_{name}_bf16"):
            continue
        a, b = operand(M, K, fmt, per_row=kind == "nvfp4_rowscale"), operand(N, K, fmt)
        d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(fb.fp4_gemm_workspace_bytes(a, b), dtype=torch.uint8, device="cuda") \
            if kind == "ue5m3_rebiased" else None
        ms = time_ms(lambda: fb.fp4_gemm(a, b, d, ws=ws))
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        peak = bf16_peak if kind == "ue5m3_emulated" else fp4_peak
        res[f"gemm_{kind}_{name}_bf16"] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peak, 3)}
        del a, b, d, ws
    T, C = 8192, 6144
    x = torch.randn((T, C), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(8192, dtype=torch.float32, device="cuda")
    E, SR = fb.FP4_SCALE_E4M3, fb.FP4_ROUND_SR
    quants = {
        "rows_rne": (lambda: fb.fp4_quantize(fb.QuantConfig(), x, o_r, ws=ws), 4.5625),
        "rows_sr": (lambda: fb.fp4_quantize(fb.QuantConfig(round=SR), x, o_r, ws=ws), 4.5625),
        "cols_rht_sr": (lambda: fb.fp4_quantize(fb.QuantConfig(round=SR, orient=fb.FP4_ORIENT_COLWISE, rht=True),
                                                x, o_c, ws=ws), 4.5625),
        "dual_rne_rht": (lambda: fb.fp4_quantize_dual(fb.QuantConfig(), fb.QuantConfig(
            orient=fb.FP4_ORIENT_COLWISE, rht=True), x, o_r, o_c, ws=ws), 5.125),
        "dual_sr_rht": (lambda: fb.fp4_quantize_dual(fb.QuantConfig(round=SR), fb.QuantConfig(
            round=SR, orient=fb.FP4_ORIENT_COLWISE, rht=True), x, o_r, o_c, ws=ws), 5.125),
        "mxfp4_rows": (lambda: fb.fp4_quantize(fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE8M0, block=fb.FP4_BLOCK_1x32),
                                               x, o_mx), 2.53125),
        # per-row tensor scales: one pass, so the input is read once (2 + 0.5625 B/elem)
        "rows_rowscale_rne": (lambda: fb.fp4_quantize(fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW), x, o_rr), 2.5625),
        "rows_rowscale_sr": (lambda: fb.fp4_quantize(fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW, round=SR), x, o_rr),
                             2.5625),
        "tensor_amax_dual_rht": (lambda: fb.fp4_tensor_amax_dual(fb.QuantConfig(), fb.QuantConfig(
            orient=fb.FP4_ORIENT_COLWISE, rht=True), x, st_r, st_c, ws), 2.0),
    }
    o_r, o_c = fb.QTensor.empty(T, C), fb.QTensor.empty(C, T)
    o_mx = fb.QTensor.empty(T, C, fb.FP4_SCALE_UE8M0)
    o_rr = fb.QTensor.empty(T, C, per_row=True)
    st_r, st_c = fb.AmaxState(), fb.AmaxState()
    for name, (fn, bpe) in quants.items():
        if not wanted(f"quantize_{name}_{T}x{C}"):
            continue
        ms = time_ms(fn)
        gbs = bpe * T * C / (ms * 1e-3) / 1e9
        res[f"quantize_{name}_{T}x{C}"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 3)}
    if wanted("quantize_2d_both_12288x4608"):
        w = torch.randn((12288, 4608), dtype=torch.bfloat16, device="cuda")
        o1, o2 = fb.QTensor.empty(12288, 4608), fb.QTensor.empty(4608, 12288)
        ms = time_ms(lambda: fb.fp4_quantize(fb.QuantConfig(block=fb.FP4_BLOCK_16x16, emit_transpose=True), w, o1,
                                             o2, ws=ws))
        gbs = 5.125 * w.numel() / (ms * 1e-3) / 1e9
        res["quantize_2d_both_12288x4608"] = {"ms": round(ms, 4), "gbs": round(gbs, 1),
                                              "frac": round(gbs / hbm_peak, 3)}
    status = fb.fp4_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    print(json.dumps({"kernels": res, "peaks": {"fp4_tflops": fp4_peak, "bf16_tflops": bf16_peak,
                                                "hbm_gbs": hbm_peak, "source": src},
                      "method": "median of 10 CUDA-event timed calls, L2 flushed before each"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="1.2b")
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--ref-feats", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernels", action="store_true", help="time single library calls instead of the step")
    ap.add_argument("--only", default=None, help="with --kernels: time only the calls whose key matches this regex")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    from workloads import WORKLOADS
    workload = WORKLOADS[args.workload]
    if args.kernels:
        run_kernels(args)
    elif args.impl == "reference":
        run_reference(args, workload)
    else:
        run_gpu(args, workload)


if __name__ == "__main__":
    main()

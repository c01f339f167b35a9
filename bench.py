"""Benchmark of the FP4 block-scaled quantized linear hot path on GB300.

One step = the whole hot path over one batch of a workload's linears. By
default that is the 8B hybrid FFN workload (T = 8192 tokens; linears
4096 -> 21504 and 21504 -> 4096), the largest configuration of the pages'
models that the quantizer and GEMM targets are set on. For each linear: the
five quantized operands (X rowwise and X^T colwise + RHT16 from one pass over
X, W 16x16 in both orientations, dY rowwise SR and dY^T colwise + RHT16 + SR
from one pass over dY; each preceded by its tensor amax, computed on a second
stream while the previous operand is converted) and the three block-scaled
NVFP4 GEMMs (Fprop, Dgrad, Wgrad). `--workload ue5m3_sweep` runs the UE5M3
held-amax sweep instead: one 4096 -> 4096 linear whose gradient drifts x10^+-3
over 100 steps, UE5M3 block scales, the held amax refreshed every 50 steps,
and the rebiased native GEMMs.

`value` is fwd+bwd GEMM TFLOP/s of the whole step (6 T N K per linear divided
by the step time, quantization included) with inputs resident in HBM (larger
than L2); `e2e` is the same metric through the public API (Fp4Linear.step_host)
with the inputs copied from pinned host memory and the outputs copied back
inside the timed region. `roofline` is the dominant kernel, the block-scaled
GEMM, timed with CUDA events on its own launches in a second pass of the same
steps; `roofline_quantize` the dominant quantizer kernel (the one-read rowwise
+ colwise quantizer) the same way. `cpu_baseline` is the CPU oracle on this
machine's cores: every operand of the step quantized in full, GEMM outputs
sampled and scaled to the full outputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b|12b|1.2b|tiny|ue5m3_sweep]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample of each step
    python bench.py --kernels              # single library calls, each against its roofline
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
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
# Algorithmic bytes per input element of one quantize call that reads its input
# once and writes two operands (E2M1 codes + one 8-bit scale per 16 values
# each): the one-read rowwise + colwise call and the 16x16 call emitting W and
# W^T, with the tensor amax given (its own pass is a separate launch) -- 2 + 2 *
# (1/2 + 1/16). A call that also reads the input for its amax adds 2.
BYTES_ONE_PASS_TWO_OPERANDS = 3.125
BYTES_AMAX_PASS = 2.0
GEMM_LABELS = ("fprop", "dgrad", "wgrad")
QUANT_LABELS = ("w", "x", "dy")


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


# --------------------------------------------------------------------------- CPU oracle
_INPUT_CACHE: dict = {}


def workload_inputs(workload, which: int) -> dict:
    from workloads import linear_inputs
    key = (workload.name, which)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE[key] = linear_inputs(workload, which)
    return _INPUT_CACHE[key]


def _operand_specs(workload, which: int):
    """The step's quantized operands of linear `which`: (name, input key,
    oracle quantize options, operand rows). Tensor ids follow the layer's: 8 *
    layer + {0 X, 1 X^T, 2 W and W^T, 3 dY, 4 dY^T}."""
    import oracle
    lin = workload.linears[which]
    T, K, N = lin.tokens, lin.k_in, lin.n_out
    fmt = oracle.FMT_UE5M3 if workload.scale_fmt == "ue5m3" else oracle.FMT_E4M3
    base = dict(scale_fmt=fmt, seed=workload.sr_seed)
    rht = dict(rht=workload.rht, seed=workload.rht_seed)
    t = 8 * which
    return [
        ("x", "x", dict(base, tensor_id=t + 0), T),
        ("xt", "x", dict(base, colwise=True, tensor_id=t + 1, **rht), K),
        ("w", "w", dict(base, block=oracle.BLOCK_16x16, tensor_id=t + 2), N),
        ("wt", "w", dict(base, block=oracle.BLOCK_16x16, colwise=True, tensor_id=t + 2), K),
        ("dy", "dy", dict(base, sr=True, tensor_id=t + 3), T),
        ("dyt", "dy", dict(base, colwise=True, sr=True, tensor_id=t + 4, **rht), N),
    ]


def oracle_step(workload, quant_frac: float, gemm_samples: int, threads: int, seed: int = 0) -> dict:
    """Time the CPU oracle on a sample of one step of `workload` with `threads`
    host threads (the oracle is C behind ctypes, which releases the GIL, so the
    threads run in parallel) and scale it to the whole step.

    Quantization: the first `quant_frac` of every operand's rows, split into
    row bands over the threads. Each operand's tensor amax is computed first (a
    timed pass over the whole tensor, as current scaling does) and handed to the
    band calls as a held amax, which gives the same scale as current scaling, so
    the bands do not each repeat it. GEMMs: `gemm_samples` outputs of each of
    the step's three GEMMs per linear, at random inside the quantized rows,
    split over the threads; each GEMM's time is scaled by (outputs of the GEMM
    / outputs sampled). Returns the step's GEMM FLOPs, the measured and the
    whole-step (scaled) seconds, and a description of the sample."""
    import numpy as np

    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    pool = cf.ThreadPoolExecutor(max_workers=threads)
    t_quant = t_quant_scaled = t_gemm = t_gemm_scaled = 0.0
    flops = 0.0
    n_gemm = 0
    for which, lin in enumerate(workload.linears):
        inp = workload_inputs(workload, which)
        specs = _operand_specs(workload, which)
        q = {}
        # every operand's tensor amax over the whole tensor (one pass each, in parallel)
        t0 = time.perf_counter()
        amaxes = list(pool.map(lambda sp: oracle.tensor_amax(inp[sp[1]], colwise=sp[2].get("colwise", False),
                                                             rht=sp[2].get("rht", False), seed=sp[2].get("seed", 0)),
                               specs))
        dt_amax = time.perf_counter() - t0
        t0 = time.perf_counter()
        for (name, src, kw, R), amax in zip(specs, amaxes):
            bits = inp[src]
            rows = max(16, int(R * quant_frac) // 16 * 16)
            nb = max(1, min(threads, rows // 16))
            edges = [rows * i // nb // 16 * 16 for i in range(nb)] + [rows]

            def band(r0, r1, bits=bits, kw=kw, amax=amax):
                st = oracle.HeldState()
                st.amax[0], st.valid[0], st.last[0] = amax, 1, 0
                # held amax, step 1 (not a refresh step): the tensor scale of current scaling
                return oracle.quantize(bits, held=True, state=st, step=1, op_rows=(r0, r1), **kw)

            parts = list(pool.map(lambda e: band(*e), zip(edges[:-1], edges[1:])))
            q[name] = ({k: np.concatenate([p[k] for p in parts]) for k in ("codes", "scales")}
                       | {"s_dec": parts[0]["s_dec"]}, rows)
        dt = time.perf_counter() - t0
        t_quant += dt_amax + dt
        t_quant_scaled += dt_amax + dt / quant_frac
        for ka, kb in (("x", "w"), ("dy", "wt"), ("dyt", "xt")):
            (ra, ma), (rb, nbr) = q[ka], q[kb]
            M = {"x": lin.tokens, "dy": lin.tokens, "dyt": lin.n_out}[ka]
            N = {"w": lin.n_out, "wt": lin.k_in, "xt": lin.k_in}[kb]
            K = ra["codes"].shape[1] * 2
            ms = rng.integers(0, ma, gemm_samples)
            ns = rng.integers(0, nbr, gemm_samples)
            chunks = np.array_split(np.arange(gemm_samples), threads)
            fmt = oracle.FMT_UE5M3 if workload.scale_fmt == "ue5m3" else oracle.FMT_E4M3
            t0 = time.perf_counter()
            list(pool.map(lambda c: oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"],
                                                rb["s_dec"], scale_fmt=fmt, pairs=(ms[c], ns[c])),
                          [c for c in chunks if c.size]))
            dt = time.perf_counter() - t0
            t_gemm += dt
            t_gemm_scaled += dt * (M * N) / gemm_samples
            flops += 2.0 * M * N * K
            n_gemm += 1
    pool.shutdown()
    return {"flops": flops, "seconds_measured": t_quant + t_gemm, "seconds_step": t_quant_scaled + t_gemm_scaled,
            "quant_seconds_step": t_quant_scaled, "gemm_seconds_step": t_gemm_scaled,
            "sample": f"{quant_frac:g} of every operand's rows quantized (tensor amax over the whole tensor) and "
                      f"{gemm_samples} sampled outputs of each of the {n_gemm} GEMMs, scaled to the whole step"}


def cpu_baseline_entry(workload) -> dict:
    """The oracle on this machine's host cores: every operand quantized in full
    and GEMM outputs sampled (all cores); plus the same on one thread over a
    sixteenth of the rows, for the single-thread figure."""
    cores = os.cpu_count() or 1
    full = oracle_step(workload, 1.0, 256 * cores, cores)
    one = oracle_step(workload, 1.0 / 16, 64, 1, seed=1)
    return {"value": full["flops"] / full["seconds_step"] / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "sample": full["sample"] + f"; {full['seconds_measured']:.1f} s measured on "
                                                          f"{cores} threads",
            "step_seconds": full["seconds_step"], "quantize_seconds_per_step": full["quant_seconds_step"],
            "single_thread": {"value": one["flops"] / one["seconds_step"] / 1e12, "cores": 1,
                              "sample": one["sample"] + f"; {one['seconds_measured']:.1f} s measured"}}


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
    """The CPU oracle as the reference arm: each step quantizes a sixteenth of
    every operand's rows and samples GEMM outputs on all host cores, scaled to
    the whole step. Rank 0 alone runs it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    frac, samples = 1.0 / 16, 16 * cores
    for i in range(args.warmup):
        oracle_step(workload, frac, samples, cores, seed=100 + i)
    steps = [oracle_step(workload, frac, samples, cores, seed=i) for i in range(args.steps)]
    flops = steps[0]["flops"]
    sec = sum(s["seconds_step"] for s in steps) / len(steps)
    value = flops / sec / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * sec, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 steps, f64 GEMM sums (oracle)",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload.name, "tokens": workload.linears[0].tokens,
                       "linears_k_n": [[l.k_in, l.n_out] for l in workload.linears]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": steps[0]["sample"] + f", {cores} threads; each step "
                                                            f"{sum(s['seconds_measured'] for s in steps) / len(steps):.1f} s measured"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, workload):
    import numpy as np
    import torch

    import fp4_block_scaled_02_gb300 as fb

    dist, rank, world = dist_setup()
    dev = torch.cuda.current_device()
    fb._lib.load()
    stream = torch.cuda.current_stream()
    sweep = workload.held
    ue = workload.scale_fmt == "ue5m3"
    target_T = workload.targets[0]

    def upload(bits):
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    # inputs: seeded synthetic BF16, uploaded once (resident in HBM)
    layers, host = [], []
    for which, lin in enumerate(workload.linears):
        inp = workload_inputs(workload, which)
        dev_in = {k: upload(v) for k, v in inp.items()}
        if sweep:
            # the sweep's gradient of step s: the base gradient times
            # 10^(-3 + 6 s / (steps - 1)) rounded to BF16 (FP32 product, RNE)
            base = dev_in["dy"].float()
            dev_in["dy_steps"] = [(base * torch.tensor(10.0 ** (-3.0 + 6.0 * s / (workload.steps - 1)),
                                                       dtype=torch.float32, device="cuda")).to(torch.bfloat16)
                                  for s in range(workload.steps)]
            del base
        L = fb.Fp4Linear(lin.tokens, lin.k_in, lin.n_out, rht=workload.rht, seed=workload.rht_seed, layer=which,
                         scale_fmt=fb.FP4_SCALE_UE5M3 if ue else fb.FP4_SCALE_E4M3, held=sweep, target_T=target_T)
        outs = {"y": torch.empty((lin.tokens, lin.n_out), dtype=torch.bfloat16, device="cuda"),
                "dx": torch.empty((lin.tokens, lin.k_in), dtype=torch.bfloat16, device="cuda"),
                "dw": torch.empty((lin.n_out, lin.k_in), dtype=torch.float32, device="cuda")}
        layers.append((lin, L, dev_in, outs))
        h = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in inp.items()}
        if sweep:
            # two pinned gradients (steps 0 and 99) alternate in the end-to-end run
            h["dy_steps"] = [dev_in["dy_steps"][0].cpu().pin_memory(), dev_in["dy_steps"][-1].cpu().pin_memory()]
        host.append(h)

    gemm_flops = workload.gemm_flops_per_step()
    # kernels launched per step: per linear, each quantize call is an amax launch
    # plus a conversion launch (with the amaxes on the side stream: a tile pass and
    # a finalize kernel each); the UE5M3 GEMMs run the rebias pass, the native
    # kernel and the emulated fallback (which returns at once) each
    per_linear = (12 if layers[0][1].side is not None else 6 + (9 if ue else 3))
    launches_per_step = per_linear * len(layers)

    def dy_of(di, i):
        return di["dy_steps"][i % workload.steps] if sweep else di["dy"]

    def step(i, mark=None):
        for lin, L, di, o in layers:
            L.step(di["x"], di["w"], dy_of(di, i), o["y"], o["dx"], o["dw"], step=i if sweep else 0,
                   stream=stream, mark=mark)

    it = 0
    for _ in range(args.warmup):
        step(it)
        it += 1
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
    timed_steps = list(range(it, it + args.steps))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in timed_steps:
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, start.elapsed_time(end))
    it += args.steps
    # per-kernel times: the same steps again with an event before and after each
    # launch on the stream (kept out of the timed steps above: an event between
    # two kernels stops the second from launching early)
    evs = []

    def mark(label):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        evs.append((label, e))

    per_label = {}
    for n in range(args.steps):
        evs.clear()
        step(timed_steps[n], mark=mark)
        torch.cuda.synchronize()
        open_ = {}
        li = 0
        for label, e in evs:
            if label.endswith("/end"):
                name = label[:-4]
                per_label.setdefault((li // 6, name), []).append(open_.pop(name).elapsed_time(e))
                li += 1
            else:
                open_[label] = e
    clk = clocks.stop()
    status = fb.fp4_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms_step = ms / args.steps
    value = world * gemm_flops / (ms_step * 1e-3) / 1e12

    # the dominant kernels against their rooflines
    def gemm_shape(lin, name):
        return {"fprop": (lin.tokens, lin.n_out, lin.k_in), "dgrad": (lin.tokens, lin.k_in, lin.n_out),
                "wgrad": (lin.n_out, lin.k_in, lin.tokens)}[name]

    g_flop = g_ms = q_bytes = q_ms = 0.0
    g_n = q_n = 0
    for (li, name), times in per_label.items():
        lin = layers[li][0]
        t = sum(times)
        if name in GEMM_LABELS:
            M, N, K = gemm_shape(lin, name)
            g_flop += 2.0 * M * N * K * len(times)
            g_ms += t
            g_n += len(times)
        elif name in ("x", "dy"):
            elems = lin.tokens * (lin.k_in if name == "x" else lin.n_out)
            for s in timed_steps:
                # held scaling reads the input a second time for its amax on refresh steps
                refresh = sweep and s % 50 == 0
                q_bytes += elems * (BYTES_ONE_PASS_TWO_OPERANDS + (BYTES_AMAX_PASS if refresh else 0.0))
            q_ms += t
            q_n += len(times)
    all_quant_ms = sum(sum(v) for (li, n), v in per_label.items() if n in QUANT_LABELS)
    gemm_tflops = g_flop / (g_ms * 1e-3) / 1e12
    dual_gbs = q_bytes / (q_ms * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host inputs in, outputs back
    def h2d_bytes():
        return sum(t.numel() * t.element_size() for h in host for k, t in h.items() if k != "dy_steps")

    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
                for (_, _, _, o) in layers]
    h2d = h2d_bytes()
    d2h = sum(t.numel() * t.element_size() for h in host_out for t in h.values())

    # Fp4Linear.step_host: input copies, the step and output copies on their own
    # streams, so one linear's copies overlap the other's compute
    def e2e_step(i):
        for (lin, L, di, o), h, ho in zip(layers, host, host_out):
            dy_h = h["dy_steps"][i % 2] if sweep else h["dy"]
            L.step_host(h["x"], h["w"], dy_h, ho["y"], ho["dx"], ho["dw"], step=i if sweep else 0, stream=stream)

    for _ in range(max(1, args.warmup)):
        e2e_step(it)
        it += 1
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _, L, _, _ in layers:
        L.h2d_stream.wait_event(e0)  # no copy starts before the timed region
    for _ in range(args.steps):
        e2e_step(it)
        it += 1
    for _, L, _, _ in layers:
        stream.wait_event(L.ev_out)  # ... and the last output copies end inside it
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * gemm_flops / (e_ms * 1e-3) / 1e12
    if fb.fp4_device_status() != 0:
        raise RuntimeError("device status after the end-to-end run")

    if rank != 0:
        return
    counts = event_counts(workload, layers, dy_of)
    peaks, src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    hbm_peak = peaks["hbm_gbs"]
    traffic = load_traffic()
    wl = args.workload
    gemm_roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": fp4_peak, "unit": "TFLOP/s",
                 "frac": gemm_tflops / fp4_peak, "traffic": traffic.get(f"gemm_nvfp4_kernel@{wl}"),
                 "peak_source": f"{src} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)",
                 "kernel": f"gemm_nvfp4_kernel ({g_n // args.steps} launches per step: Fprop, Dgrad, Wgrad of each "
                           f"linear), CUDA events around each launch",
                 "ms_per_launch": g_ms / max(1, g_n)}
    quant_roof = {"bound": "hbm", "achieved": dual_gbs, "peak": hbm_peak, "unit": "GB/s",
                  "frac": dual_gbs / hbm_peak, "traffic": traffic.get(f"quantize_dual_kernel@{wl}"),
                  "peak_source": f"{src} hbm_gbs",
                  "kernel": f"quantize_dual_kernel ({q_n // args.steps} launches per step: X and dY of each linear, "
                            f"{BYTES_ONE_PASS_TWO_OPERANDS} B per input element"
                            + (", + 2 on held-amax refresh steps" if sweep else ", tensor amax given") + ")",
                  "ms_per_launch": q_ms / max(1, q_n)}
    cpu = None if args.no_cpu_baseline else cpu_baseline_entry(workload)
    lin_desc = [[l.k_in, l.n_out] for l in workload.linears]
    recipe = ("UE5M3: 1x16 UE5M3 acts/grads, 16x16 weights, held amax refreshed every 50 steps "
              f"(T = {target_T:g}), SR on dY, no RHT, rebiased native GEMMs"
              if sweep else "NVFP4: 1x16 E4M3 acts/grads, 16x16 weights, current scaling, SR on dY, "
                            "RHT16 on Wgrad inputs")
    cfg = {"workload": workload.name, "tokens": workload.linears[0].tokens, "linears_k_n": lin_desc,
           "recipe": recipe,
           "l2": "inputs larger than L2 (%.0f MB of BF16 inputs per step)" % (h2d / 1e6),
           "parallelism": f"replicas x{world}"}
    if sweep:
        cfg["sweep_steps_timed"] = [timed_steps[0], timed_steps[-1]]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1 (fp32 accumulate)", "data": "synthetic",
        "config": cfg,
        "gemm_tflops": gemm_tflops, "quantize_dual_gbs": dual_gbs,
        "ms_gemm_per_step": g_ms / args.steps, "ms_quantize_calls_per_step": all_quant_ms / args.steps,
        "roofline": gemm_roof, "roofline_quantize": quant_roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "event_counts": counts,
    }
    print(json.dumps(line), flush=True)


COUNTER_ORDER = ["elem_sat", "elem_underflow", "scale_sat", "scale_underflow"]
LAYER_ROWS = ["x", "xt", "w", "dy", "dyt"]  # Fp4Linear.counters rows (W: both orientations, each element once)


def event_counts(workload, layers, dy_of):
    """The four event counters of every quantized tensor, outside the timed
    region (the pages argue from saturation and underflow events). Fixed-shape
    workloads: one step's counters per tensor with the step's own recipe, and
    the MXFP4 1x32 power-of-two-scale quantizer (rowwise) on the same X, W and dY.
    The held-amax sweep: a fresh layer per target T, stepped through every step
    of the sweep in order, dY's rowwise and colwise counters at each step."""
    import torch

    import fp4_block_scaled_02_gb300 as fb

    out = {"order": COUNTER_ORDER}
    if not workload.held:
        nv, mx, elems = [], [], []
        for lin, L, di, o in layers:
            L.counters.zero_()
            L.step(di["x"], di["w"], di["dy"], o["y"], o["dx"], o["dw"], step=0)
            torch.cuda.synchronize()
            c = L.counters.cpu().tolist()
            nv.append({name: c[i] for i, name in enumerate(LAYER_ROWS)})
            m = {}
            for name in ("x", "w", "dy"):
                t = di[name]
                q = fb.QTensor.empty(t.shape[0], t.shape[1], fb.FP4_SCALE_UE8M0)
                cnt = torch.zeros(4, dtype=torch.int64, device="cuda")
                fb.fp4_quantize(fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE8M0, block=fb.FP4_BLOCK_1x32), t, q,
                                counters=cnt, ws=L.ws)
                m[name] = cnt.cpu().tolist()
                del q
            mx.append(m)
            elems.append({"x": lin.tokens * lin.k_in, "w": lin.n_out * lin.k_in, "dy": lin.tokens * lin.n_out})
        out.update({"nvfp4": nv, "mxfp4_1x32_rowwise": mx, "elements": elems})
    else:
        lin, L0, di, o = layers[0]
        per_T = {}
        for T in workload.targets:
            L = fb.Fp4Linear(lin.tokens, lin.k_in, lin.n_out, rht=workload.rht, seed=workload.rht_seed,
                             scale_fmt=L0.scale_fmt, held=True, target_T=T)
            rows = {"dy": [], "dyt": []}
            for s in range(workload.steps):
                L.counters.zero_()
                L.step(di["x"], di["w"], dy_of(di, s), o["y"], o["dx"], o["dw"], step=s)
                c = L.counters.cpu().tolist()
                rows["dy"].append(c[3])
                rows["dyt"].append(c[4])
            per_T[f"{T:g}"] = rows
            del L
        out.update({"steps": workload.steps, "per_step": per_T,
                    "elements": {"dy": lin.tokens * lin.n_out}})
    if fb.fp4_device_status() != 0:
        raise RuntimeError("device status after the event-count pass")
    return out


def load_traffic() -> dict:
    """Per-launch DRAM bytes (kernel@workload) from the committed ncu summaries
    (profiles/traffic.json), if present."""
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
        # the conversion pass alone (tensor amax given, as in the step)
        "dual_sr_rht_given": (lambda: fb.fp4_quantize_dual(
            fb.QuantConfig(round=SR, tscale=fb.FP4_TSCALE_GIVEN),
            fb.QuantConfig(round=SR, orient=fb.FP4_ORIENT_COLWISE, rht=True, tscale=fb.FP4_TSCALE_GIVEN),
            x, o_r, o_c, st_r, st_c), 3.125),
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
    # held scaling ([UE] method details): refreshed at step 0, then timed on step 1, a
    # non-refresh step -- one pass over the input, the amax pass only a guard launch
    HELD = dict(tscale=fb.FP4_TSCALE_HELD, refresh_every=50)
    sh_r, sh_c, sh_d = fb.AmaxState(), fb.AmaxState(), fb.AmaxState()
    if wanted(f"quantize_rows_held_rne_step1_{T}x{C}"):
        fb.fp4_quantize(fb.QuantConfig(step=0, **HELD), x, o_r, state=sh_r, ws=ws)
    if wanted(f"quantize_dual_held_sr_rht_step1_{T}x{C}"):
        fb.fp4_quantize_dual(fb.QuantConfig(step=0, round=SR, **HELD),
                             fb.QuantConfig(step=0, round=SR, orient=fb.FP4_ORIENT_COLWISE, rht=True, **HELD),
                             x, o_r, o_c, sh_d, sh_c, ws=ws)
    quants["rows_held_rne_step1"] = (lambda: fb.fp4_quantize(fb.QuantConfig(step=1, **HELD), x, o_r, state=sh_r,
                                                             ws=ws), 2.5625)
    quants["dual_held_sr_rht_step1"] = (lambda: fb.fp4_quantize_dual(
        fb.QuantConfig(step=1, round=SR, **HELD),
        fb.QuantConfig(step=1, round=SR, orient=fb.FP4_ORIENT_COLWISE, rht=True, **HELD),
        x, o_r, o_c, sh_d, sh_c, ws=ws), 3.125)
    # the given-amax calls read the records a tensor-amax call leaves
    fb.fp4_tensor_amax_dual(fb.QuantConfig(), fb.QuantConfig(orient=fb.FP4_ORIENT_COLWISE, rht=True), x, st_r, st_c,
                            ws)
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
    if wanted("quantize_2d_plain_12240x4608"):
        # rows not a multiple of 64: the 16x16 kernel without TMA tiles (plain scale layout)
        w = torch.randn((12240, 4608), dtype=torch.bfloat16, device="cuda")
        lay = dict(layout=fb.FP4_LAYOUT_PLAIN)
        o1, o2 = fb.QTensor.empty(12240, 4608, **lay), fb.QTensor.empty(4608, 12240, **lay)
        ms = time_ms(lambda: fb.fp4_quantize(fb.QuantConfig(block=fb.FP4_BLOCK_16x16, emit_transpose=True, **lay), w,
                                             o1, o2, ws=ws))
        gbs = 5.125 * w.numel() / (ms * 1e-3) / 1e9
        res["quantize_2d_plain_12240x4608"] = {"ms": round(ms, 4), "gbs": round(gbs, 1),
                                               "frac": round(gbs / hbm_peak, 3)}
    if wanted(f"dequantize_{T}x{C}"):
        fb.fp4_quantize(fb.QuantConfig(), x, o_r, ws=ws)
        y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
        ms = time_ms(lambda: fb.fp4_dequantize(o_r, y))
        gbs = (0.5625 + 2.0) * T * C / (ms * 1e-3) / 1e9  # codes + scales read, BF16 written
        res[f"dequantize_{T}x{C}"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 3)}
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
    ap.add_argument("--workload", default="8b")
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

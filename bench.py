#!/usr/bin/env python
"""BRA forward throughput on B300: tokens/s, roofline fraction, CPU oracle.

One step is one BRA forward (bra_forward through the C ABI: routing, then
routed attention + LePE) over one batch of the workload. The headline
workload is the BiFormer stage-1 shape (B=64, 56x56, C=64, 2 heads, S=7,
top-1, LePE 5x5, bf16); the line's `workloads` key measures all five
workload shapes the same way (configs 1..5 in the order the workload
statement lists them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Timing: inputs resident in HBM; K steps replayed from CUDA graphs over
rotating input sets whose footprint exceeds the 126 MB L2, bracketed by a
barrier and a synchronize, timed with CUDA events, max over ranks. Under
torchrun each rank runs its own shard of images (weak scaling, no collective
on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import bra_synth  # noqa: E402

METRIC = "BRA forward tokens/s on 1 B300 (bf16) and % of roofline; vs CPU oracle"
L2_BYTES = 126 * 1024 * 1024
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "vision_transformer_sparse_route_b300", "csrc")

# Config numbers of the five workloads, in the order the workload statement
# lists them.
CONFIG_NUMBER = {"tiny_f32": 1, "stage1_bf16": 2, "stage2_bf16": 3, "stage3_bf16": 4,
                 "seg512_bf16": 5}

# Unit counts of a B300 SM for the ALU and MUFU ceilings: 128 float32 FMA
# lanes (2 flops each) and 16 ex2 results per clock (the bf16x2 form returns
# two exponentials per result).
FP32_LANES_PER_SM = 128
EX2_PER_SM_CLK = 16
SM_FALLBACK, MHZ_FALLBACK = 148, 2032.0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="stage1_bf16", choices=list(bra_synth.WORKLOADS))
    p.add_argument("--workloads", default="all",
                   help="workloads measured for the `workloads` key: all, none or a "
                        "comma-separated list")
    p.add_argument("--sets", type=int, default=0, help="rotating input sets (0: auto)")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--kernel-steps", type=int, default=200)
    p.add_argument("--load-seconds", type=float, default=1.5,
                   help="identical untimed steps before the timed region (clock samples)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--cpu-seconds-each", type=float, default=2.5,
                   help="oracle seconds per (workload, thread count) of the `workloads` key")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    return p.parse_args(argv)


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sources_digest(files=None) -> str:
    """Digest of the given kernel sources (names under csrc/), by default of
    every .cu/.cuh file there."""
    names = files if files is not None else sorted(
        n for n in os.listdir(CSRC) if n.endswith((".cu", ".cuh")))
    h = hashlib.sha256()
    for name in sorted(names):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def kernel_sources(kernel: str, workload: str) -> list:
    """The source files that define the device kernel `kernel` ("route" or
    "attend") runs as for a workload: the kernel's own header and the headers
    it includes. A recorded DRAM byte count stays valid while these are
    unchanged."""
    wl = bra_synth.WORKLOADS[workload]
    small = wl.dtype == "bf16" and wl.H // wl.S * (wl.W // wl.S) <= 8
    if kernel == "route":
        if small and wl.S * wl.S <= 64 and wl.C // 64 in (1, 2, 4) and wl.C % 64 == 0:
            # the per-chunk routing kernel of the small-map path
            return ["forward_image.cuh", "attend_image.cuh", "attend_bf16.cuh", "route.cuh",
                    "ptx.cuh"]
        return ["route.cuh", "ptx.cuh"]
    if wl.dtype == "f32":
        return ["attend_f32.cuh", "ptx.cuh"]
    if wl.H // wl.S * (wl.W // wl.S) < 16:  # regions under 16 tokens: image-resident kernel
        return ["attend_image.cuh", "attend_bf16.cuh", "ptx.cuh"]
    return ["attend_bf16.cuh", "ptx.cuh"]


def algorithmic_bytes(wl: bra_synth.Workload) -> dict:
    """Bytes each kernel must move at least (inputs read once, outputs
    written once); LePE weights and the routing index are below 0.1%."""
    e = 4 if wl.dtype == "f32" else 2
    t = wl.B * wl.H * wl.W * wl.C * e
    return {"route": 2 * t, "attend": 4 * t, "forward": 4 * t}


def algorithmic_work(wl: bra_synth.Workload) -> dict:
    """Algorithmic work of each kernel and of the whole forward: bytes (inputs
    read once, output written once), contraction flops of q k^T and p v,
    other float32 flops (LePE 2 ks^2 per output element, affinity 2 R^2 C
    and region pooling 2 N C per image) and exponentials (one per query and
    routed key and head). The float32 path runs its contractions on the FMA
    pipe, so there they count as ALU flops."""
    N, R, n = wl.H * wl.W, wl.R, wl.n
    b = algorithmic_bytes(wl)
    contraction = 4 * wl.B * N * wl.topk * n * wl.C
    lepe = 2 * wl.ks * wl.ks * wl.B * N * wl.C
    affinity = 2 * wl.B * R * R * wl.C
    pooling = 2 * wl.B * N * wl.C
    exps = wl.B * N * wl.heads * wl.topk * n
    tc = contraction if wl.dtype == "bf16" else 0
    alu_c = 0 if wl.dtype == "bf16" else contraction
    route = {"bytes": b["route"], "tensor_flops": 0, "alu_flops": affinity + pooling, "exps": 0}
    attend = {"bytes": b["attend"], "tensor_flops": tc, "alu_flops": lepe + alu_c, "exps": exps}
    fwd = {"bytes": b["forward"], "tensor_flops": tc,
           "alu_flops": lepe + alu_c + affinity + pooling, "exps": exps}
    return {"route": route, "attend": attend, "forward": fwd}


def projection_work(wl: bra_synth.Workload) -> dict:
    """Algorithmic work of the Q/K/V projection of one batch: x read once, q,
    k and v written once, the [3C, C] weight read once (bf16), and
    2 M C 3C contraction flops."""
    M, C = wl.B * wl.H * wl.W, wl.C
    return {"bytes": 4 * M * C * 2 + 3 * C * C * 2, "tensor_flops": 6 * M * C * C,
            "alu_flops": 0, "exps": 0}


def block_work(wl: bra_synth.Workload) -> dict:
    """Algorithmic work of the block's attention branch y = x + bra(norm1(x))
    as its four steps run it: LayerNorm (x read, x_n written), projection (x_n
    read, q, k, v written, weight read), forward (q, k, v read, out written),
    residual add (x and out read, y written): 13 M C elements; flops of the
    projection and the forward."""
    M, C = wl.B * wl.H * wl.W, wl.C
    fwd = algorithmic_work(wl)["forward"]
    return {"bytes": 13 * M * C * 2 + 3 * C * C * 2,
            "tensor_flops": fwd["tensor_flops"] + 6 * M * C * C,
            "alu_flops": fwd["alu_flops"], "exps": fwd["exps"]}


def ffn_work(wl: bra_synth.Workload) -> dict:
    """Algorithmic work of the block's ConvFFN branch y = x + fc2(GELU(
    dwconv3x3(fc1(norm2(x))))) as its four steps run it: LayerNorm 2 M C,
    fc1 M C + 3 M C, the convolution and GELU 3 M C + 3 M C, fc2 3 M C + M C
    (residual) + M C elements (bf16), the weights once; contraction flops of
    fc1 and fc2, float32 flops of the 3 x 3 convolution."""
    M, C = wl.B * wl.H * wl.W, wl.C
    return {"bytes": 17 * M * C * 2 + 2 * 3 * C * C * 2 + 10 * 3 * C * 4,
            "tensor_flops": 2 * 6 * M * C * C, "alu_flops": 2 * 9 * 3 * M * C, "exps": 0}


def backward_work(wl: bra_synth.Workload) -> dict:
    """Algorithmic work of the backward of attend (the routing fixed): q, k,
    v and dout read once and dq, dk, dv written once (float32), the LePE
    weights; the six contractions of the attention's backward (the logits and
    O again, dout v^T, P^T dout, dS k and dS^T q: 2 k n d each per query and
    head), on the tensor pipe for bf16 and the FMA pipe for float32; the
    LePE's input and weight gradients (2 ks^2 each per element); one
    exponential per query, routed key and head."""
    e = 4 if wl.dtype == "f32" else 2
    T = wl.B * wl.H * wl.W * wl.C
    nk = wl.topk * wl.n
    contraction = 6 * 2 * (wl.B * wl.H * wl.W) * nk * wl.C
    lepe = 4 * wl.ks * wl.ks * T
    return {"bytes": 4 * T * e + 3 * T * 4 + 2 * wl.C * wl.ks * wl.ks * 4,
            "tensor_flops": contraction if wl.dtype == "bf16" else 0,
            "alu_flops": lepe + (contraction if wl.dtype == "f32" else 0),
            "exps": wl.B * wl.H * wl.W * wl.heads * nk}


def peaks(sm_count: int | None = None, sm_mhz: float | None = None) -> dict:
    """Roofline denominators: HBM GB/s and bf16 tensor TFLOP/s measured on
    the B300s (MEASURED_PEAKS.json, burst figures for kernels timed
    alone), float32 ALU TFLOP/s and exponentials/s derived from the SM's unit
    counts and its maximum clock."""
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        hbm, tc, kind = float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1800.0)), "measured"
        mhz = sm_mhz or float(p.get("sm_max_mhz", MHZ_FALLBACK))
    except (OSError, KeyError, ValueError):
        hbm, tc, kind = 6400.0, 1800.0, "fallback"
        mhz = sm_mhz or MHZ_FALLBACK
    sms = sm_count or SM_FALLBACK
    clk = mhz * 1e6
    return {"hbm_gbs": hbm, "tensor_tflops": tc,
            "alu_tflops": sms * FP32_LANES_PER_SM * 2 * clk / 1e12,
            "ex2_per_s_f32": sms * EX2_PER_SM_CLK * clk,
            "ex2_per_s_bf16": 2 * sms * EX2_PER_SM_CLK * clk,
            "source": kind, "sm_count": sms, "sm_mhz": mhz}


def measured_peaks():
    p = peaks()
    return p["hbm_gbs"], p["source"]


def roofline(work: dict, pk: dict, dtype: str, seconds: float) -> dict:
    """Roofline of one kernel (or the whole forward) that took `seconds`:
    the slowest of bytes at HBM bandwidth, contraction flops at the tensor
    peak, ALU flops at the float32 peak and exponentials at the MUFU rate;
    `bound` names it, and achieved / peak are in its unit."""
    ex2 = pk["ex2_per_s_bf16"] if dtype == "bf16" else pk["ex2_per_s_f32"]
    terms = {
        "hbm": (work["bytes"] / (pk["hbm_gbs"] * 1e9), work["bytes"] / 1e9, pk["hbm_gbs"],
                "GB/s"),
        "tensor": (work["tensor_flops"] / (pk["tensor_tflops"] * 1e12),
                   work["tensor_flops"] / 1e12, pk["tensor_tflops"], "TFLOP/s"),
        "alu": (work["alu_flops"] / (pk["alu_tflops"] * 1e12), work["alu_flops"] / 1e12,
                pk["alu_tflops"], "TFLOP/s"),
        "mufu": (work["exps"] / ex2, work["exps"] / 1e9, ex2 / 1e9, "G exp/s"),
    }
    bound = max(terms, key=lambda k: terms[k][0])
    t_roof, amount, peak, unit = terms[bound]
    achieved = amount / seconds if seconds > 0 else 0.0
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": t_roof / seconds if seconds > 0 else 0.0, "roof_us": t_roof * 1e6,
            "measured_us": seconds * 1e6,
            "terms_us": {k: v[0] * 1e6 for k, v in terms.items()}}


class ClockSampler:
    """nvidia-smi samples (100 ms) from start() to stop(), with timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", self.gpu_id, "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [f.strip() for f in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float, window: str) -> dict:
        rows = [r for t, r in self.rows if len(r) >= 9]
        timed = [r for t, r in self.rows if len(r) >= 9 and t0 <= t <= t1]
        use = timed if len(timed) >= 3 else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        mx = [num(r[2]) for r in use if num(r[2]) is not None]
        pw = [num(r[3]) for r in use if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(use),
                "window": window if len(timed) >= 3 else window + " (timed region too short; "
                "samples span the load phase before it)"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("sources") != sources_digest(kernel_sources(kernel, workload)):
        return None
    return e.get("dram_bytes_per_launch")


def selected_workloads(spec: str) -> list:
    if spec in ("", "none"):
        return []
    if spec == "all":
        return list(bra_synth.WORKLOADS)
    names = [s.strip() for s in spec.split(",") if s.strip()]
    for n in names:
        if n not in bra_synth.WORKLOADS:
            raise SystemExit(f"unknown workload {n}")
    return names


# ------------------------------------------------------------- CPU oracle
def time_oracle(wl: bra_synth.Workload, x: bra_synth.Inputs, seconds: float, cores: int,
                images: int | None = None):
    """Runs the oracle forward on the first `images` images until `seconds`
    have passed; returns (tokens/s, images per call, calls)."""
    import oracle
    oracle.build()
    if images is None:
        t = time.perf_counter()
        oracle.forward(x.q[:1], x.k[:1], x.v[:1], wl.heads, wl.S, wl.topk, x.lepe_w,
                       x.lepe_b, threads=cores)
        per_img = max(time.perf_counter() - t, 1e-4)
        images = int(max(1, min(x.q.shape[0], seconds / 4 / per_img)))
    q, k, v = x.q[:images], x.k[:images], x.v[:images]
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(q, k, v, wl.heads, wl.S, wl.topk, x.lepe_w, x.lepe_b, threads=cores)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    tokens = calls * images * wl.H * wl.W
    return tokens / el, images, calls


def reference_arm(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    x = bra_synth.make_inputs(wl, seed=0, batch=slice(0, 1))
    import oracle
    oracle.build()
    step = lambda: oracle.forward(x.q, x.k, x.v, wl.heads, wl.S, wl.topk, x.lepe_w,
                                  x.lepe_b, threads=cores)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    tokens = args.steps * wl.H * wl.W
    value = tokens / el
    sample = f"one image ({wl.H}x{wl.W} tokens) of {wl.name} per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64/Box-Muller, region offsets + token noise)",
            "config": dict(workload=wl.name, **wl.describe()),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- ours
class Setup:
    """Device buffers, CUDA graphs and timers for one workload."""

    def __init__(self, wl, dev, stream, x, sets_arg: int, use_graph: bool):
        import torch
        import vision_transformer_sparse_route_b300 as bra
        self.torch, self.bra, self.wl, self.dev, self.stream = torch, bra, wl, dev, stream
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.tdt = tdt
        cast = lambda a: torch.from_numpy(a).to(tdt)
        self.host = [cast(a).pin_memory() for a in (x.q, x.k, x.v)]
        self.w = torch.from_numpy(x.lepe_w).to(dev)
        self.b = torch.from_numpy(x.lepe_b).to(dev)
        ab = algorithmic_bytes(wl)
        self.set_bytes = ab["forward"] + wl.B * wl.R * wl.topk * 4
        self.sets = sets_arg or max(2, -(-3 * L2_BYTES // self.set_bytes) + 1)
        self.bufs = []
        for _ in range(self.sets):
            q, k, v = (h.to(dev, non_blocking=True) for h in self.host)
            out = torch.empty_like(q)
            idx = torch.empty((wl.B, wl.R, wl.topk), dtype=torch.int32, device=dev)
            self.bufs.append((q, k, v, out, idx))
        torch.cuda.synchronize()
        self.graphs = self.capture(self.fwd) if use_graph else []

    def fwd(self, s):
        q, k, v, out, idx = self.bufs[s % self.sets]
        self.bra.forward(q, k, v, self.wl.heads, self.wl.S, self.wl.topk, self.w, self.b,
                         out=out, idx=idx, stream=self.stream)

    def launches(self) -> int:
        wl = self.wl
        return self.bra.forward_launches(wl.B, wl.H, wl.W, wl.C, wl.heads, wl.S, wl.topk,
                                         wl.ks, 1 if wl.dtype == "bf16" else 0)

    def route(self, s):
        q, k, v, out, idx = self.bufs[s % self.sets]
        self.bra.route(q, k, self.wl.S, self.wl.topk, idx=idx, stream=self.stream)

    def attend(self, s):
        q, k, v, out, idx = self.bufs[s % self.sets]
        self.bra.attend(q, k, v, idx, self.wl.heads, self.wl.S, self.w, self.b, out=out,
                        stream=self.stream)

    def attend_tc(self, s):
        q, k, v, out, idx = self.bufs[s % self.sets]
        self.bra.attend_tc(q, k, v, idx, self.wl.heads, self.wl.S, self.w, self.b, out=out,
                           stream=self.stream)

    def capture(self, launch):
        """One CUDA graph per input set (launch overhead off the step)."""
        torch = self.torch
        gs = []
        with torch.cuda.stream(self.stream):
            for s in range(self.sets):
                launch(s)  # warm the library (tensor-map entry point, attributes)
            self.stream.synchronize()
            for s in range(self.sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    launch(s)
                gs.append(g)
        torch.cuda.synchronize()
        return gs

    def step(self, i):
        if self.graphs:
            self.graphs[i % self.sets].replay()
        else:
            self.fwd(i)

    def time_steps(self, n: int) -> float:
        """ms for n forward steps, CUDA events on the launching stream."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for i in range(n):
                self.step(i)
            e1.record(self.stream)
            e1.synchronize()
        return e0.elapsed_time(e1)

    def time_kernel(self, launch, steps: int) -> float:
        """ms per launch of one kernel, replayed alone from its own CUDA graphs
        over the rotating input sets."""
        torch = self.torch
        gs = self.capture(launch)
        with torch.cuda.stream(self.stream):
            for i in range(3):
                gs[i % self.sets].replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for i in range(steps):
                gs[i % self.sets].replay()
            e1.record(self.stream)
            e1.synchronize()
        return e0.elapsed_time(e1) / steps

    def release(self):
        self.graphs = []
        self.bufs = []
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def time_projection(wl, dev, stream, steps: int) -> float:
    """ms per bra_qkv_project launch over the workload's tokens, from CUDA
    graphs over rotating input sets larger than L2."""
    import torch
    import vision_transformer_sparse_route_b300 as bra
    M, C = wl.B * wl.H * wl.W, wl.C
    x, w, b = bra_synth.make_projection_inputs(M, C, 0)
    wd = torch.from_numpy(w).to(torch.bfloat16).to(dev)
    bd = torch.from_numpy(b).to(dev)
    per_set = 4 * M * C * 2
    sets = max(2, -(-3 * L2_BYTES // per_set) + 1)
    xh = torch.from_numpy(x).to(torch.bfloat16)
    bufs = [(xh.to(dev), torch.empty((M, C), dtype=torch.bfloat16, device=dev),
             torch.empty((M, C), dtype=torch.bfloat16, device=dev),
             torch.empty((M, C), dtype=torch.bfloat16, device=dev)) for _ in range(sets)]
    graphs = []
    with torch.cuda.stream(stream):
        for xs, q, k, v in bufs:
            bra.qkv_project(xs, wd, bd, q, k, v, stream=stream)
        stream.synchronize()
        for xs, q, k, v in bufs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                bra.qkv_project(xs, wd, bd, q, k, v, stream=stream)
            graphs.append(g)
        for i in range(3):
            graphs[i % sets].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % sets].replay()
        e1.record(stream)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graphs, bufs
    torch.cuda.empty_cache()
    return ms


def time_block(wl, dev, stream, steps: int) -> float:
    """ms per bra_block_attention call (four launches) on the workload's map,
    from CUDA graphs over rotating input sets larger than L2."""
    import numpy as np
    import torch
    import vision_transformer_sparse_route_b300 as bra
    B, H, W, C = wl.B, wl.H, wl.W, wl.C
    M = B * H * W
    x, w, b = bra_synth.make_projection_inputs(M, C, 0)
    rng = np.random.default_rng(0)
    wd = torch.from_numpy(w).to(torch.bfloat16).to(dev)
    bd = torch.from_numpy(b).to(dev)
    lnw = torch.from_numpy((1 + 0.1 * rng.standard_normal(C)).astype(np.float32)).to(dev)
    lnb = torch.from_numpy((0.1 * rng.standard_normal(C)).astype(np.float32)).to(dev)
    lw = torch.from_numpy((0.02 * rng.standard_normal((C, wl.ks, wl.ks))).astype(np.float32)).to(dev)
    lb = torch.from_numpy((0.02 * rng.standard_normal(C)).astype(np.float32)).to(dev)
    ws_bytes = bra._load().bra_block_attention_workspace_bytes(B, H, W, C, wl.S, wl.topk)
    per_set = 2 * M * C * 2 + ws_bytes
    sets = max(2, -(-3 * L2_BYTES // per_set) + 1)
    xh = torch.from_numpy(x).to(torch.bfloat16).reshape(B, H, W, C)
    bufs = [(xh.to(dev), torch.empty((B, H, W, C), dtype=torch.bfloat16, device=dev),
             torch.empty(ws_bytes, dtype=torch.uint8, device=dev)) for _ in range(sets)]
    def call(xs, y, ws):
        bra.block_attention(xs, lnw, lnb, wd, bd, wl.heads, wl.S, wl.topk, lw, lb, out=y,
                            workspace=ws, stream=stream)
    graphs = []
    with torch.cuda.stream(stream):
        for t in bufs:
            call(*t)
        stream.synchronize()
        for t in bufs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(*t)
            graphs.append(g)
        for i in range(3):
            graphs[i % sets].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % sets].replay()
        e1.record(stream)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graphs, bufs
    torch.cuda.empty_cache()
    return ms


def time_block_ffn(wl, dev, stream, steps: int) -> float:
    """ms per bra_block_ffn call (four launches) on the workload's map, from
    CUDA graphs over rotating input sets larger than L2."""
    import numpy as np
    import torch
    import vision_transformer_sparse_route_b300 as bra
    B, H, W, C = wl.B, wl.H, wl.W, wl.C
    M = B * H * W
    rng = np.random.default_rng(1)
    d = lambda a, t=torch.float32: torch.from_numpy(a.astype(np.float32)).to(t).to(dev)  # noqa
    lnw, lnb = d(1 + 0.1 * rng.standard_normal(C)), d(0.1 * rng.standard_normal(C))
    w1 = d(rng.standard_normal((3 * C, C)) / np.sqrt(C), torch.bfloat16)
    b1 = d(0.02 * rng.standard_normal(3 * C))
    cw, cb = d(rng.standard_normal((3 * C, 3, 3)) / 3), d(0.02 * rng.standard_normal(3 * C))
    w2 = d(rng.standard_normal((C, 3 * C)) / np.sqrt(3 * C), torch.bfloat16)
    b2 = d(0.02 * rng.standard_normal(C))
    ws_bytes = bra._load().bra_block_ffn_workspace_bytes(B, H, W, C)
    per_set = 2 * M * C * 2 + ws_bytes
    sets = max(2, -(-3 * L2_BYTES // per_set) + 1)
    x, _, _ = bra_synth.make_projection_inputs(M, C, 0)
    xh = torch.from_numpy(x).to(torch.bfloat16).reshape(B, H, W, C)
    bufs = [(xh.to(dev), torch.empty((B, H, W, C), dtype=torch.bfloat16, device=dev),
             torch.empty(ws_bytes, dtype=torch.uint8, device=dev)) for _ in range(sets)]
    def call(xs, y, ws):
        bra.block_ffn(xs, lnw, lnb, w1, b1, cw, cb, w2, b2, out=y, workspace=ws, stream=stream)
    graphs = []
    with torch.cuda.stream(stream):
        for t in bufs:
            call(*t)
        stream.synchronize()
        for t in bufs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(*t)
            graphs.append(g)
        for i in range(3):
            graphs[i % sets].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % sets].replay()
        e1.record(stream)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graphs, bufs
    torch.cuda.empty_cache()
    return ms


def time_backward(wl, dev, stream, steps: int) -> float:
    """ms per bra_attend_backward call (the gradients of attend for a given
    dout, the routing fixed) on the workload, from CUDA graphs over rotating
    input sets larger than L2."""
    import numpy as np
    import torch
    import vision_transformer_sparse_route_b300 as bra
    x = bra_synth.make_inputs(wl, seed=0)
    cast = (lambda a: torch.from_numpy(a).to(torch.bfloat16)) if wl.dtype == "bf16" else \
        (lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)))
    q, k, v = (cast(a).to(dev) for a in (x.q, x.k, x.v))
    w = torch.from_numpy(x.lepe_w).to(dev)
    rng = np.random.default_rng(5)
    dout = cast(rng.standard_normal((wl.B, wl.H, wl.W, wl.C)).astype(np.float32)).to(dev)
    idx = bra.route(q, k, wl.S, wl.topk)
    e = 4 if wl.dtype == "f32" else 2
    T = wl.B * wl.H * wl.W * wl.C
    per_set = 4 * T * e + 3 * T * 4
    sets = max(2, -(-3 * L2_BYTES // per_set) + 1)
    bufs = [(q.clone(), k.clone(), v.clone(), dout.clone()) + tuple(
        torch.empty((wl.B, wl.H, wl.W, wl.C), dtype=torch.float32, device=dev) for _ in range(3))
        for _ in range(sets)]
    dw = torch.empty(x.lepe_w.shape, dtype=torch.float32, device=dev)
    db = torch.empty(wl.C, dtype=torch.float32, device=dev)
    lib = bra._load()
    code = bra.BRA_BF16 if wl.dtype == "bf16" else bra.BRA_F32

    def call(qs, ks, vs, gs, dq, dk, dv):
        rc = lib.bra_attend_backward(qs.data_ptr(), ks.data_ptr(), vs.data_ptr(), idx.data_ptr(),
                                     wl.B, wl.H, wl.W, wl.C, wl.heads, wl.S, wl.topk,
                                     w.data_ptr(), wl.ks, gs.data_ptr(), code, dq.data_ptr(),
                                     dk.data_ptr(), dv.data_ptr(), dw.data_ptr(), db.data_ptr(),
                                     stream.cuda_stream)
        if rc != bra.BRA_OK:
            raise RuntimeError(f"bra_attend_backward: {rc}")
    graphs = []
    with torch.cuda.stream(stream):
        for t in bufs:
            call(*t)
        stream.synchronize()
        for t in bufs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(*t)
            graphs.append(g)
        for i in range(3):
            graphs[i % sets].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % sets].replay()
        e1.record(stream)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graphs, bufs
    torch.cuda.empty_cache()
    return ms


def launch_floor(torch, stream, reps: int = 2000) -> dict:
    """Replay cost of a CUDA graph holding one near-empty kernel (a
    one-element fill) and one holding two of them in a chain, back to back
    on one stream: the floor under any one- or two-kernel forward."""
    z = torch.zeros(1, device=stream.device)
    out = {}
    for nk in (1, 2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            z.fill_(0.0)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(nk):
                    z.fill_(1.0)
            for _ in range(10):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        out[f"graph_{nk}_kernel_us"] = e0.elapsed_time(e1) * 1e3 / reps
    return out


def measure_workload(wl, dev, stream, pk, kernel_steps: int, cpu_seconds: float,
                     no_cpu: bool, use_graph: bool) -> dict:
    """The `workloads` entry of one workload: forward ms/step, each kernel's
    launch time, rooflines and the oracle at one thread and all cores."""
    import torch
    x = bra_synth.make_inputs(wl, seed=0)
    st = Setup(wl, dev, stream, x, 0, use_graph)
    for i in range(5):
        st.step(i)
    probe = st.time_steps(20) / 20
    n = int(min(20000, max(200, 0.3 / max(probe * 1e-3, 1e-7))))
    ms = st.time_steps(n) / n
    route_ms = st.time_kernel(st.route, kernel_steps)
    attend_ms = st.time_kernel(st.attend, kernel_steps)
    fwd_ms = st.time_kernel(st.fwd, kernel_steps)
    # the tcgen05 formulation of the attend step, where its shape applies
    # (8 x 8 regions, 64 channels, top-k <= 4)
    tc_ms = None
    if (wl.dtype == "bf16" and wl.C == 64 and wl.heads == 2 and wl.H // wl.S == 8
            and wl.W // wl.S == 8 and wl.topk <= 4 and wl.ks in (1, 3, 5)):
        tc_ms = st.time_kernel(st.attend_tc, kernel_steps)
    # the Q/K/V projection that produces this workload's q, k, v (bf16, C a
    # multiple of 64 up to 256)
    proj_ms = block_ms = None
    if wl.dtype == "bf16" and wl.C % 64 == 0 and wl.C <= 256:
        proj_ms = time_projection(wl, dev, stream, kernel_steps)
        # the block's attention branch, x + bra(norm1(x)), projections included
        block_ms = time_block(wl, dev, stream, kernel_steps)
    ffn_ms = None
    if wl.dtype == "bf16" and wl.C in (64, 128):
        # the block's ConvFFN branch (its fc2 takes K = 3C up to 384)
        ffn_ms = time_block_ffn(wl, dev, stream, kernel_steps)
    # the backward of attend (the routing fixed)
    bwd_ms = time_backward(wl, dev, stream, max(10, kernel_steps // 4))
    work = algorithmic_work(wl)
    ok = st.bra.device_status(stream)
    launches = st.launches()
    st.release()
    del st
    entry = {"config": CONFIG_NUMBER.get(wl.name), "ms_per_step": ms, "steps_timed": n,
             "tokens_per_s": wl.tokens / (ms * 1e-3), "forward_launches": launches,
             "forward_us": fwd_ms * 1e3, "route_us": route_ms * 1e3,
             "attend_us": attend_ms * 1e3,
             "step_roofline": roofline(work["forward"], pk, wl.dtype, ms * 1e-3),
             "route_roofline": roofline(work["route"], pk, wl.dtype, route_ms * 1e-3),
             "attend_roofline": roofline(work["attend"], pk, wl.dtype, attend_ms * 1e-3),
             **({"qkv_project_us": proj_ms * 1e3,
                 "qkv_project_roofline": roofline(projection_work(wl), pk, wl.dtype,
                                                  proj_ms * 1e-3)}
                if proj_ms is not None else {}),
             **({"block_attention_us": block_ms * 1e3,
                 "block_attention_roofline": roofline(block_work(wl), pk, wl.dtype,
                                                      block_ms * 1e-3)}
                if block_ms is not None else {}),
             **({"block_ffn_us": ffn_ms * 1e3,
                 "block_ffn_roofline": roofline(ffn_work(wl), pk, wl.dtype, ffn_ms * 1e-3)}
                if ffn_ms is not None else {}),
             "backward_us": bwd_ms * 1e3,
             "backward_roofline": roofline(backward_work(wl), pk, wl.dtype, bwd_ms * 1e-3),
             **({"attend_tc_us": tc_ms * 1e3,
                 "attend_tc_roofline": roofline(work["attend"], pk, wl.dtype, tc_ms * 1e-3)}
                if tc_ms is not None else {}),
             "device_status": ok}
    if not no_cpu:
        cores = os.cpu_count() or 1
        v1, i1, _ = time_oracle(wl, x, cpu_seconds, 1)
        va, ia, _ = time_oracle(wl, x, cpu_seconds, cores)
        entry["oracle_tokens_per_s"] = {"threads_1": v1, f"threads_{cores}": va,
                                        "images_sampled": [i1, ia], "cores": cores}
    del x
    torch.cuda.empty_cache()
    return entry


def our_arm(args, wl):
    import torch
    import vision_transformer_sparse_route_b300 as bra

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    pk = peaks(props.multi_processor_count)

    # this rank's shard of a world * B image batch (weak scaling)
    wl_global = wl.replace(B=wl.B * world)
    x = bra_synth.make_inputs(wl_global, seed=0, batch=bra_synth.rank_slice(wl.B, rank))
    stream = torch.cuda.Stream(device=dev)
    st = Setup(wl, dev, stream, x, args.sets, not args.no_graph)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or "0")
    sampler = ClockSampler(gpu_id)
    sampler.start()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            st.step(i)
        # untimed load phase: same steps, so clock samples reflect this load
        stream.synchronize()
        t_load = time.time()
        i = 0
        while time.time() - t_load < args.load_seconds:
            for _ in range(200):
                st.step(i)
                i += 1
            stream.synchronize()
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            st.step(i)
        ev1.record(stream)
        ev1.synchronize()
        t1 = time.time()
        barrier()
    sampler.stop()
    clocks = sampler.summary(t0, t1, "timed region")
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    tokens = world * args.steps * wl.tokens
    value = tokens / (ms / 1e3)

    # per-kernel durations: each kernel captured alone in a CUDA graph per input
    # set and replayed back to back over the rotating sets
    ks = max(1, args.kernel_steps)
    route_ms = st.time_kernel(st.route, ks)
    attend_ms = st.time_kernel(st.attend, ks)
    launches = st.launches()
    fwd_ms = st.time_kernel(st.fwd, ks) if launches == 1 else None

    # end to end through the public API with pinned host buffers: copies in,
    # forward and copies out of consecutive batches overlapped (HostPipeline)
    host = st.host
    pipe = bra.HostPipeline(host[0].shape, st.tdt, wl.S, wl.topk, dev)
    outs_h = [torch.empty(host[0].shape, dtype=st.tdt).pin_memory() for _ in range(2)]
    es = max(1, args.e2e_steps)
    for i in range(3):
        pipe.submit(*host, wl.heads, wl.S, wl.topk, st.w, st.b, outs_h[i % 2])
    pipe.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.copy_in)
    for i in range(es):
        pipe.submit(*host, wl.heads, wl.S, wl.topk, st.w, st.b, outs_h[i % 2])
    e1.record(pipe.copy_out)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * es * wl.tokens / (e2e_ms / 1e3)
    ok = bra.device_status(stream)
    sets, set_bytes = st.sets, st.set_bytes
    del pipe, outs_h
    st.release()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    work = algorithmic_work(wl)
    if launches == 1:  # the forward is one kernel (routing inside it)
        dom, dom_ms = "forward", fwd_ms
    else:
        dom = "attend" if attend_ms >= route_ms else "route"
        dom_ms = attend_ms if dom == "attend" else route_ms
    rl = roofline(work[dom], pk, wl.dtype, dom_ms * 1e-3)
    step_ms = ms / args.steps
    elem = 2 if wl.dtype == "bf16" else 4
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded SplitMix64/Box-Muller: per-region N(0,1) offsets + "
                "per-token N(0,0.5^2); LePE weights N(0,0.02^2))",
        "config": {"workload": wl.name, "config_number": CONFIG_NUMBER.get(wl.name),
                   **wl.describe(), "global_batch": wl.B * world,
                   "l2": f"{sets} rotating input sets, {sets * set_bytes / 2**20:.0f} MiB "
                         f"> {L2_BYTES // 2**20} MiB L2",
                   "launch": "eager" if args.no_graph else "cuda_graph",
                   "parallelism": f"batch shards x{world}, no collective"},
        "roofline": {**{k: rl[k] for k in ("bound", "achieved", "peak", "unit", "frac")},
                     "traffic": recorded_traffic(dom, wl.name), "kernel": f"bra_{dom}",
                     "algorithmic_bytes": work[dom]["bytes"], "kernel_ms": dom_ms,
                     "terms_us": rl["terms_us"],
                     "peak_source": f"MEASURED_PEAKS.json ({pk['source']}) for HBM and "
                                    "tensor; ALU and MUFU from unit counts x max clock"},
        "step_roofline": roofline(work["forward"], pk, wl.dtype, step_ms * 1e-3),
        "kernel_ms": {"bra_route": route_ms, "bra_attend": attend_ms,
                      **({"bra_forward": fwd_ms} if fwd_ms is not None else {})},
        "forward_launches": launches,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": 3 * wl.tokens * wl.C * elem,
                "d2h_bytes_per_step": wl.tokens * wl.C * elem,
                "ms_per_step": e2e_ms / es},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "device_status": ok,
        "peaks": pk,
    }
    if world == 1:
        line["launch_floor"] = launch_floor(torch, stream)
        table = {}
        for name in selected_workloads(args.workloads):
            table[name] = measure_workload(bra_synth.WORKLOADS[name], dev, stream, pk,
                                           ks, args.cpu_seconds_each, args.no_cpu,
                                           not args.no_graph)
        if table:
            line["workloads"] = table
    if not args.no_cpu and world == 1:
        cores = os.cpu_count() or 1
        v_cpu, imgs, calls = time_oracle(wl, x, args.cpu_seconds, cores)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"first {imgs} image(s) of {wl.name}, {calls} "
                                          f"oracle forward call(s), ~{args.cpu_seconds:.0f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    wl = bra_synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, wl)
    else:
        our_arm(args, wl)


if __name__ == "__main__":
    main()

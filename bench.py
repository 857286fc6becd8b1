#!/usr/bin/env python
"""BRA forward throughput on B300: tokens/s, roofline fraction, CPU oracle.

One step is one BRA forward (bra_route + bra_attend through the C ABI) over
one batch of the workload. Default workload: the BiFormer stage-1 shape
(B=64, 56x56, C=64, 2 heads, S=7, top-1, LePE 5x5, bf16).

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


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="stage1_bf16", choices=list(bra_synth.WORKLOADS))
    p.add_argument("--sets", type=int, default=0, help="rotating input sets (0: auto)")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--kernel-steps", type=int, default=200)
    p.add_argument("--load-seconds", type=float, default=1.5,
                   help="identical untimed steps before the timed region (clock samples)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sources_digest() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(wl: bra_synth.Workload) -> dict:
    """Bytes each kernel must move at least (inputs read once, outputs
    written once); LePE weights and the routing index are below 0.1%."""
    e = 4 if wl.dtype == "f32" else 2
    t = wl.B * wl.H * wl.W * wl.C * e
    return {"route": 2 * t, "attend": 4 * t, "forward": 4 * t}


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


def measured_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p["hbm_gbs"], "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("sources") != sources_digest():
        return None
    return e.get("dram_bytes_per_launch")


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

    # this rank's shard of a world * B image batch (weak scaling)
    wl_global = wl.replace(B=wl.B * world)
    x = bra_synth.make_inputs(wl_global, seed=0, batch=bra_synth.rank_slice(wl.B, rank))
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    cast = lambda a: torch.from_numpy(a).to(tdt)
    host = [cast(a).pin_memory() for a in (x.q, x.k, x.v)]
    w = torch.from_numpy(x.lepe_w).to(dev)
    b = torch.from_numpy(x.lepe_b).to(dev)

    ab = algorithmic_bytes(wl)
    set_bytes = ab["forward"] + wl.B * wl.R * wl.topk * 4
    sets = args.sets or max(2, -(-3 * L2_BYTES // set_bytes) + 1)
    bufs = []
    for s in range(sets):
        q, k, v = (h.to(dev, non_blocking=True) for h in host)
        out = torch.empty_like(q)
        idx = torch.empty((wl.B, wl.R, wl.topk), dtype=torch.int32, device=dev)
        bufs.append((q, k, v, out, idx))
    torch.cuda.synchronize()

    def fwd(s, stream=None):
        q, k, v, out, idx = bufs[s % sets]
        bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b, out=out, idx=idx, stream=stream)

    # one CUDA graph per input set (launch overhead off the step)
    stream = torch.cuda.Stream(device=dev)
    graphs = []
    if not args.no_graph:
        with torch.cuda.stream(stream):
            for s in range(sets):
                fwd(s, stream)  # warm the library (tensor-map entry point, attributes)
            stream.synchronize()
            for s in range(sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fwd(s, stream)
                graphs.append(g)
    torch.cuda.synchronize()

    def step(i):
        if graphs:
            graphs[i % sets].replay()
        else:
            fwd(i, stream)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or "0")
    sampler = ClockSampler(gpu_id)
    sampler.start()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        # untimed load phase: same steps, so clock samples reflect this load
        stream.synchronize()
        t_load = time.time()
        i = 0
        while time.time() - t_load < args.load_seconds:
            for _ in range(200):
                step(i)
                i += 1
            stream.synchronize()
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
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
    # set and replayed back to back over the rotating sets (no host work between
    # launches); CUDA events on the launching stream bracket the replays
    ks = max(1, args.kernel_steps)

    def kernel_graphs(launch):
        gs = []
        with torch.cuda.stream(stream):
            for s in range(sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    launch(s)
                gs.append(g)
        return gs

    def time_graphs(gs):
        with torch.cuda.stream(stream):
            for i in range(3):
                gs[i % sets].replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(ks):
                gs[i % sets].replay()
            e1.record(stream)
            e1.synchronize()
        return e0.elapsed_time(e1) / ks

    def launch_route(s):
        q, k, v, out, idx = bufs[s]
        bra.route(q, k, wl.S, wl.topk, idx=idx, stream=stream)

    def launch_attend(s):
        q, k, v, out, idx = bufs[s]
        bra.attend(q, k, v, idx, wl.heads, wl.S, w, b, out=out, stream=stream)

    route_ms = time_graphs(kernel_graphs(launch_route))
    attend_ms = time_graphs(kernel_graphs(launch_attend))

    # end to end through the public API with pinned host buffers: copies in,
    # forward and copies out of consecutive batches overlapped (HostPipeline)
    pipe = bra.HostPipeline(host[0].shape, tdt, wl.S, wl.topk, dev)
    outs_h = [torch.empty(host[0].shape, dtype=tdt).pin_memory() for _ in range(2)]
    es = max(1, args.e2e_steps)
    for i in range(3):
        pipe.submit(*host, wl.heads, wl.S, wl.topk, w, b, outs_h[i % 2])
    pipe.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.copy_in)
    for i in range(es):
        pipe.submit(*host, wl.heads, wl.S, wl.topk, w, b, outs_h[i % 2])
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

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    dom = "attend" if attend_ms >= route_ms else "route"
    dom_ms = attend_ms if dom == "attend" else route_ms
    achieved = ab[dom] / (dom_ms / 1e3) / 1e9
    step_ms = ms / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded SplitMix64/Box-Muller: per-region N(0,1) offsets + "
                "per-token N(0,0.5^2); LePE weights N(0,0.02^2))",
        "config": {"workload": wl.name, **wl.describe(), "global_batch": wl.B * world,
                   "l2": f"{sets} rotating input sets, {sets * set_bytes / 2**20:.0f} MiB "
                         f"> {L2_BYTES // 2**20} MiB L2",
                   "launch": "cuda_graph" if graphs else "eager",
                   "parallelism": f"batch shards x{world}, no collective"},
        "roofline": {"bound": "hbm", "kernel": f"bra_{dom}", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(dom, wl.name),
                     "algorithmic_bytes": ab[dom], "kernel_ms": dom_ms,
                     "peak_source": f"hbm_gbs of MEASURED_PEAKS ({peak_kind})"},
        "step_roofline": {"bytes": ab["forward"], "achieved_gbs": ab["forward"] / (step_ms / 1e3)
                          / 1e9, "frac": ab["forward"] / (step_ms / 1e3) / 1e9 / peak},
        "kernel_ms": {"bra_route": route_ms, "bra_attend": attend_ms},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": 3 * wl.tokens * wl.C * (2 if wl.dtype == "bf16" else 4),
                "d2h_bytes_per_step": wl.tokens * wl.C * (2 if wl.dtype == "bf16" else 4),
                "ms_per_step": e2e_ms / es},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "device_status": ok,
    }
    if not args.no_cpu and world == 1:
        cores = os.cpu_count() or 1
        xs = bra_synth.Inputs(x.q, x.k, x.v, x.lepe_w, x.lepe_b)
        v_cpu, imgs, calls = time_oracle(wl, xs, args.cpu_seconds, cores)
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

#!/usr/bin/env python3
"""Benchmark of the decode-linear weight stream on GB300.

A step is one pass of the hot path over one batch: the four linears of one
Qwen2.5-72B-shaped decoder layer (QKV 8192->10240 with bias, O 8192->8192,
gate_up 8192->59136, down 29568->8192) at M=1 with bf16 weights -- ~1.75 GB of
weights streamed from HBM per step, far more than the 129 MB L2, so no weight
byte is ever an L2 hit between steps.  The metric is achieved HBM bandwidth:
algorithmic bytes (weights + scales + x + y + bias) / device time, reported
absolutely and as a fraction of the measured HBM copy bandwidth.

`--workload fp8_m6` times the same four shapes with weight-only FP8
block-128 weights at M=6; `--workload decode_stream` times the whole-model
weight stream (80 FP8 layers + bf16 lm_head, M=1) as ms/token.

`--impl reference` times the CPU oracle (the only other arm: no reference
implementation exists) on a bounded sample of the same workload.

Prints ONE JSON line on rank 0.  Multi-GPU (torchrun): every rank streams its
own replica of the workload (no data exchange), times are reduced with MAX.
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

METRIC = "achieved HBM GB/s and % of GB300 peak per decode linear; ms/token weight stream"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["weight_streaming_skinny_gb300/csrc/dl_kernel.cuh",
                  "weight_streaming_skinny_gb300/csrc/dl_device.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it is current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("traffic", {}).get(workload, {}).get(kernel)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the workload runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu_index, self.period_ms = gpu_index, period_ms
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def layer_specs(workload: str):
    from weight_streaming_skinny_gb300 import inputs
    shapes = inputs.QWEN72B_SHAPES
    if workload == "qwen72b_layer_bf16_m1":
        return [(inputs.DTYPE_BF16, 1, *shapes[n][:2], shapes[n][2], n) for n in shapes], 1
    if workload == "qwen72b_layer_fp8_m6":
        return [(inputs.DTYPE_FP8_B128, 6, *shapes[n][:2], shapes[n][2], n) for n in shapes], 2
    raise ValueError(workload)


def build_layers(workload, dev):
    from weight_streaming_skinny_gb300 import inputs
    specs, cfg = layer_specs(workload)
    out = []
    for i, (dt, M, N, K, bias, name) in enumerate(specs):
        L = inputs.make_layer(dt, M, N, K, bias=bias, config_id=cfg, layer_idx=i, device=dev)
        out.append((name, L))
    return out


def launch(dl, L, y, ws, stream):
    if L.dtype == "bf16":
        dl.linear_bf16(L.x, L.w, L.bias, out=y, workspace=ws, stream=stream)
    else:
        dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out=y, workspace=ws, stream=stream)


def run_ours(args, rank, world, dist):
    import torch
    import weight_streaming_skinny_gb300 as dl
    from weight_streaming_skinny_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dl.load()
    workload = args.workload
    layers = build_layers(workload, dev)
    ys = [torch.empty((L.M, L.N), dtype=torch.bfloat16, device=dev) for _, L in layers]
    ws = dl.Workspace.for_shapes(
        [(L.M, L.N, L.K, dl.BF16 if L.dtype == "bf16" else dl.FP8_B128) for _, L in layers], dev)
    stream = torch.cuda.Stream(dev)
    nbytes = [L.algorithmic_bytes for _, L in layers]
    step_bytes = sum(nbytes)
    torch.cuda.synchronize(dev)

    def step(evs=None):
        for j, (_, L) in enumerate(layers):
            if evs is not None:
                evs[j].record(stream)
            launch(dl, L, ys[j], ws, stream)
        if evs is not None:
            evs[len(layers)].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()

    # ---- timed region: exactly K steps, per-kernel events on the launching stream
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(layers) + 1)] for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.05)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for k in range(K):
            step(evs[k])
        t1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    # keep the same load running (untimed) until the clock record has samples
    extra_steps = 0
    deadline = time.time() + 3.0
    while len(sampler.lines) < 5 and time.time() < deadline:
        with torch.cuda.stream(stream):
            for _ in range(20):
                step()
        stream.synchronize()
        extra_steps += 20
    sampler.stop()
    total_ms = t0.elapsed_time(t1)
    per_layer_ms = [sum(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(K)) / K
                    for j in range(len(layers))]
    if dist is not None:
        import torch.distributed as tdist
        t = torch.tensor([total_ms], dtype=torch.float64)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / K
    value = step_bytes * world * K / (total_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.skip_e2e:
        hx = [L.x.cpu().pin_memory() for _, L in layers]
        hy = [torch.empty((L.M, L.N), dtype=torch.bfloat16).pin_memory() for _, L in layers]
        dx = [torch.empty_like(L.x) for _, L in layers]
        h2d = sum(x.numel() * 2 for x in hx)
        d2h = sum(y.numel() * 2 for y in hy)
        E = max(3, min(K, 50))

        def e2e_step():
            for j, (_, L) in enumerate(layers):
                dx[j].copy_(hx[j], non_blocking=True)
                Lj = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, dx[j], L.w, L.scales, L.bias)
                launch(dl, Lj, ys[j], ws, stream)
                hy[j].copy_(ys[j], non_blocking=True)
            stream.synchronize()

        with torch.cuda.stream(stream):
            for _ in range(2):
                e2e_step()
            if dist is not None:
                dist.barrier()
            a = time.perf_counter()
            for _ in range(E):
                e2e_step()
            el = time.perf_counter() - a
        if dist is not None:
            import torch.distributed as tdist
            t = torch.tensor([el], dtype=torch.float64)
            tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
            el = float(t.item())
        e2e = {"value": round(step_bytes * world * E / el / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(el / E * 1e3, 4), "steps": E,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "x copied host->device and y device->host every step; weights resident in HBM"}

    # ---- roofline of the dominant kernel (all four layers run one kernel instance)
    peak, peak_kind = measured_peak()
    kname = "linear_kernel"
    k_bytes = sum(nbytes)
    k_ms = sum(per_layer_ms)
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": recorded_traffic(workload, kname),
                "kernel": kname, "bytes_per_launch_avg": int(k_bytes / len(layers)),
                "avg_launch_us": round(k_ms / len(layers) * 1e3, 3)}
    per_layer = {name: {"us": round(ms * 1e3, 3), "bytes": b,
                        "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                        "frac_measured": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
                 for (name, _), ms, b in zip(layers, per_layer_ms, nbytes)}
    return {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 5), "e2e": e2e,
        "roofline": roofline, "per_layer": per_layer, "clocks": sampler.summary(),
        "clock_window": f"timed region + {extra_steps} untimed steps of the same workload",
        "gpu_launches": len(layers) * K, "step_bytes": step_bytes,
    }, layers


def cpu_oracle_gbs(layers_host, budget_s: float, row_frac: float = 1.0):
    """Oracle GB/s over a bounded sample: row_frac of every layer's rows, repeated
    passes until budget_s of CPU time (at least one pass)."""
    import numpy as np
    import oracle
    from weight_streaming_skinny_gb300 import inputs
    prepared = []
    for name, L in layers_host:
        n = max(1, int(L.N * row_frac))
        rows = np.linspace(0, L.N - 1, n).astype(np.int64)
        xb = inputs.bf16_bits(L.x)
        bb = None if L.bias is None else inputs.bf16_bits(L.bias)
        if L.dtype == "bf16":
            args = (oracle.BF16, xb, inputs.bf16_bits(L.w), None, bb)
            wbytes = 2 * n * L.K
        else:
            args = (oracle.FP8_B128, xb, inputs.u8_codes(L.w), L.scales.cpu().numpy(), bb)
            wbytes = n * L.K + 4 * ((n + 127) // 128) * (L.K // 128)
        prepared.append((args, rows, wbytes + 2 * L.M * L.K + 2 * L.M * n + (2 * n if bb is not None else 0)))
    threads = oracle.default_threads()
    passes, t_total, b_total = 0, 0.0, 0
    while passes == 0 or t_total < budget_s:
        for args, rows, b in prepared:
            a = time.perf_counter()
            oracle.linear(*args[:3], scales=args[3], bias_bits=args[4], rows=rows, with_abs=False,
                          threads=threads)
            t_total += time.perf_counter() - a
            b_total += b
        passes += 1
    return b_total / t_total / 1e9, threads, passes, t_total


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen72b_layer_bf16_m1",
                    choices=["qwen72b_layer_bf16_m1", "qwen72b_layer_fp8_m6"])
    ap.add_argument("--skip-e2e", action="store_true", help="omit the end-to-end leg")
    ap.add_argument("--skip-cpu-baseline", action="store_true", help="omit the oracle timing leg")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("gloo")
        dist = tdist

    specs, _ = layer_specs(args.workload)
    config = {"workload": args.workload,
              "layers": [{"name": s[5], "dtype": s[0], "M": s[1], "N": s[2], "K": s[3],
                          "bias": s[4]} for s in specs],
              "l2": "inputs larger than L2: every step streams all four weight matrices "
                    "(>= 0.88 GB) through a 129 MB L2",
              "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        if rank != 0:
            return
        import torch
        layers = build_layers(args.workload, "cpu")
        sample_frac = 0.25
        for _ in range(args.warmup):
            cpu_oracle_gbs(layers, 0.0, sample_frac)
        vals, t_all = [], 0.0
        for _ in range(args.steps):
            v, threads, _, t = cpu_oracle_gbs(layers, 0.0, sample_frac)
            vals.append(v)
            t_all += t
        value = statistics.mean(vals)
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(t_all / args.steps * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": specs[0][0], "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                                 "kind": "oracle",
                                 "sample": f"{int(sample_frac * 100)}% of the output rows of each "
                                           "of the four linears (all K), one pass per step"},
                "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        del torch
        return

    res, layers = run_ours(args, rank, world, dist)
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        host_layers = [(n, L.to("cpu")) for n, L in layers]
        v, threads, passes, t = cpu_oracle_gbs(host_layers, args.cpu_budget_s, 1.0)
        cpu = {"value": round(v, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"the whole step (all rows of the four linears), {passes} pass(es), "
                         f"{t:.1f} s of oracle time"}
    if rank == 0:
        line = {"metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": specs[0][0], "data": "synthetic (seeded; no trained weights)",
                "config": config, "roofline": res["roofline"], "cpu_baseline": cpu,
                "e2e": res["e2e"], "clocks": res["clocks"], "clock_window": res["clock_window"],
                "gpu_launches": res["gpu_launches"], "per_layer": res["per_layer"],
                "step_bytes": res["step_bytes"], "kernel_hash": kernel_hash()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the decode-linear weight stream on GB300.

A step is one pass of the hot path over one batch.  The default workload is
the whole-model decode weight stream of one token: 80 Qwen2.5-72B-shaped
decoder layers with weight-only FP8 block-128 weights (QKV 8192->10240 with
bias, O 8192->8192, gate_up 8192->59136 with the fused SwiGLU epilogue, down
29568->8192), chained as the model chains them, then the bf16 lm_head
8192->152064 with the fused argmax, M=1 -- 72.7 GB of weights per token, far
more than the 129 MB L2, so no weight byte is ever an L2 hit between steps.
The metric is achieved HBM bandwidth: algorithmic bytes (weights + scales + x
+ y + bias) / device time, reported absolutely, as a fraction of the measured
HBM copy bandwidth, and as ms per token against the bandwidth ceiling.

A step runs through the layer-list entry point (dl_decode_stream), replayed as
a cached CUDA graph (`--mode graph`, default); `--mode calls` issues one API
call per layer.  After the timed region the line also carries: the same K
steps timed again (two runs must agree within 0.5 %), the per-step
distribution (median, p10, p90), isolated single calls of every layer shape
(an event pair around each call), the bf16 layer (M=1) and FP8 layer (M=6)
workloads with each layer's in-stream cost, and the 1024x1024 bf16 GEMV
latency.

`--workload qwen72b_layer_bf16_m1` / `qwen72b_layer_fp8_m6` / the token sweep
`qwen72b_mlp_{bf16,fp8}_m{1,2,4,6,8,16}` time those layer sets on their own.

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

MLP_TOKENS = (1, 2, 4, 6, 8, 16)
# The token sweep: the two largest linears of a decoder layer (gate_up, down)
# at M = 1..16 tokens, each dtype.
# qwen72b_decoder_fp8_m1 / qwen72b_lm_head_bf16_m1: one decoder layer and the
# lm_head of the whole-model stream on their own (small cases of its launches).
# gemv_bf16_1024_m1: the 1024 x 1024 bf16 GEMV with bias alone (a latency
# case whose 2.1 MB stay in L2; its own workload so that profilers can take it).
WORKLOADS = ["qwen72b_layer_bf16_m1", "qwen72b_layer_fp8_m6", "qwen72b_model_fp8_m1",
             "qwen72b_decoder_fp8_m1", "qwen72b_lm_head_bf16_m1", "gemv_bf16_1024_m1"] + [
    f"qwen72b_mlp_{dt}_m{m}" for dt in ("bf16", "fp8") for m in MLP_TOKENS]


def layer_specs(workload: str):
    """[(dtype, M, N, K, bias, name, act)], config id.  act = 1: gate_up with the
    fused SwiGLU epilogue (y holds N/2 columns); act = 2: lm_head with the fused
    argmax (y holds the M token indices, no logits are written)."""
    from weight_streaming_skinny_gb300 import inputs
    shapes = inputs.QWEN72B_SHAPES
    if workload == "qwen72b_layer_bf16_m1":
        return [(inputs.DTYPE_BF16, 1, *shapes[n][:2], shapes[n][2], n, 0) for n in shapes], 1
    if workload == "qwen72b_layer_fp8_m6":
        return [(inputs.DTYPE_FP8_B128, 6, *shapes[n][:2], shapes[n][2], n, 0) for n in shapes], 2
    if workload in ("qwen72b_model_fp8_m1", "qwen72b_decoder_fp8_m1"):
        specs = []
        for layer in range(inputs.QWEN72B_LAYERS if workload == "qwen72b_model_fp8_m1" else 1):
            for n in shapes:
                specs.append((inputs.DTYPE_FP8_B128, 1, *shapes[n][:2], shapes[n][2], f"{n}.{layer}",
                              1 if n == "gate_up" else 0))
        if workload == "qwen72b_model_fp8_m1":
            N, K, b = inputs.QWEN72B_LM_HEAD
            specs.append((inputs.DTYPE_BF16, 1, N, K, b, "lm_head", 2))
        return specs, 4
    if workload == "qwen72b_lm_head_bf16_m1":
        N, K, b = inputs.QWEN72B_LM_HEAD
        return [(inputs.DTYPE_BF16, 1, N, K, b, "lm_head", 2)], 4
    if workload == "gemv_bf16_1024_m1":
        return [(inputs.DTYPE_BF16, 1, 1024, 1024, True, "gemv", 0)], 0
    if workload.startswith("qwen72b_mlp_"):
        _, _, dt, m = workload.split("_")
        dtype = inputs.DTYPE_BF16 if dt == "bf16" else inputs.DTYPE_FP8_B128
        return [(dtype, int(m[1:]), *shapes[n][:2], shapes[n][2], n, 0) for n in ("gate_up", "down")], 3
    raise ValueError(workload)


def out_cols(L) -> int:
    """Columns of a layer's y (N, or N/2 with the SwiGLU epilogue)."""
    return L.N // 2 if getattr(L, "act", 0) == 1 else L.N


def out_buffer(L, dev):
    """y of a layer: bf16 [M, out_cols], or int32 [M] token indices (argmax)."""
    import torch
    if getattr(L, "act", 0) == 2:
        return torch.empty((L.M,), dtype=torch.int32, device=dev)
    return torch.empty((L.M, out_cols(L)), dtype=torch.bfloat16, device=dev)


def out_bytes(L) -> int:
    """Algorithmic bytes of a layer: weights (+ scales) + x + its outputs (+ bias)."""
    act = getattr(L, "act", 0)
    y = 4 * L.M if act == 2 else 2 * L.M * out_cols(L)
    return L.algorithmic_bytes - 2 * L.M * L.N + y


def build_layers(workload, dev):
    """Seeded layers on `dev` (each LayerInputs gets an `act` attribute).  In the
    whole-model stream a layer reads the previous layer's output where the
    model does: down -> next QKV, O -> gate_up, gate_up (SwiGLU) -> down, last
    down -> lm_head.  Attention is not part of this path, so O reads a fixed
    activation buffer."""
    from weight_streaming_skinny_gb300 import inputs
    specs, cfg = layer_specs(workload)
    out = []
    for i, (dt, M, N, K, bias, name, act) in enumerate(specs):
        L = inputs.make_layer(dt, M, N, K, bias=bias, config_id=cfg, layer_idx=i, device=dev)
        L.act = act
        out.append((name, L))
    if workload in ("qwen72b_model_fp8_m1", "qwen72b_decoder_fp8_m1"):
        for i in range(1, len(out)):
            prev, cur = out[i - 1][1], out[i][1]
            if out_cols(prev) == cur.K and prev.M == cur.M and out[i][0].split(".")[0] != "o":
                cur.x = None          # chained: filled with the previous layer's y below
    return out


def launch(dl, L, y, ws, stream):
    if getattr(L, "act", 0) == 1:
        dl.linear_swiglu(L.x, L.w, L.scales, L.bias, out=y, workspace=ws, stream=stream)
    elif getattr(L, "act", 0) == 2:
        dl.linear_argmax(L.x, L.w, L.scales, L.bias, out_idx=y, workspace=ws, stream=stream)
    elif L.dtype == "bf16":
        dl.linear_bf16(L.x, L.w, L.bias, out=y, workspace=ws, stream=stream)
    else:
        dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out=y, workspace=ws, stream=stream)


def replica_rate(local_s: float, bytes_per_rank: float, dist, world: int):
    """Whole-job throughput of `world` independent replicas (weak scaling):
    the bytes every rank processed over the slowest rank's time.  Returns
    (seconds, GB/s); with torch.distributed the local time is reduced with MAX
    over the ranks (gloo, CPU tensors)."""
    if dist is not None:
        import torch
        t = torch.tensor([local_s], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local_s = float(t.item())
    return local_s, bytes_per_rank * world / local_s / 1e9


def _pctl(vals, q):
    """q-quantile (0..1) of a list, linear interpolation."""
    v = sorted(vals)
    if not v:
        return None
    i = q * (len(v) - 1)
    lo = int(i)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (i - lo)


def _dist_us(ms_list):
    """median / p10 / p90 in microseconds of per-call (or per-step) times in ms."""
    return {"median_us": round(statistics.median(ms_list) * 1e3, 3),
            "p10_us": round(_pctl(ms_list, 0.1) * 1e3, 3),
            "p90_us": round(_pctl(ms_list, 0.9) * 1e3, 3), "n": len(ms_list)}


def make_dl_layers(dl, layers, ys):
    return [dl.Layer(dl.BF16 if L.dtype == "bf16" else dl.FP8_B128, L.x, L.w, ys[j],
                     L.scales, L.bias, act=L.act) for j, (_, L) in enumerate(layers)]


def time_steps(torch, step, stream, steps, per_step=True):
    """CUDA-event timing of `steps` calls of step() on `stream`: (total ms, per-step ms list)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1 if per_step else 2)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for k in range(steps):
            step()
            if per_step:
                evs[k + 1].record(stream)
        if not per_step:
            evs[1].record(stream)
    stream.synchronize()
    total = evs[0].elapsed_time(evs[-1])
    each = [evs[k].elapsed_time(evs[k + 1]) for k in range(steps)] if per_step else []
    return total, each


def single_call_times(torch, dl, calls, stream, reps):
    """Isolated call times: an event pair around every call (events break the
    overlap with the neighbouring launches), calls cycled through `calls`
    (distinct weights, together at least 3 x L2, keep L2 cold).  A short spin
    kernel before each pair keeps the GPU busy while the host enqueues the
    call, so that the pair measures the call on the device, not the host's
    submission.  Returns per-call ms."""
    n = len(calls)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    with torch.cuda.stream(stream):
        for r in range(reps):
            torch.cuda._sleep(100_000)
            evs[r][0].record(stream)
            calls[r % n]()
            evs[r][1].record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def layer_call(dl, L, y, ws, stream):
    return lambda: launch(dl, L, y, ws, stream)


def stream_rate(torch, dl, layers, ys, stream, steps, warmup):
    """GB/s and ms per step of the layers as one decode stream (graph replay)."""
    dls = make_dl_layers(dl, layers, ys)
    ws = dl.Workspace.for_stream(dls)
    step = lambda: dl.decode_stream(dls, ws, use_graph=True, stream=stream)  # noqa: E731
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    total, each = time_steps(torch, step, stream, steps)
    nbytes = sum(out_bytes(L) for _, L in layers)
    return total / steps, each, nbytes


def cold_copies(L, l2_bytes) -> int:
    """Distinct copies of a layer that single calls rotate over so that each
    call finds none of its bytes in L2: ceil(3 x L2 / the layer's bytes)."""
    return max(1, -(-3 * l2_bytes // L.algorithmic_bytes))


def layer_config_summary(torch, dl, workload, dev, stream, peak, steps=60, warmup=5, repeats=8):
    """An untimed-by-the-contract summary of one of the layer workloads: the
    configured step (its 4 layers as one graph replay); each layer's in-stream
    cost, measured inside a stream of `repeats` copies of the layer set
    (distinct weights, one graph, as consecutive decoder layers of a decode
    step run) as (the stream's time - the time of the same stream without
    every copy of that layer) / repeats, and also the same difference in the
    4-layer graph alone, where the first layer pays the graph's start; and
    each layer's isolated single call, rotated over the copies (some of these
    layers are smaller than L2)."""
    from weight_streaming_skinny_gb300 import inputs
    specs, cfg = layer_specs(workload)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layers = build_layers(workload, dev)
    ys = [out_buffer(L, dev) for _, L in layers]
    ms, each, nbytes = stream_rate(torch, dl, layers, ys, stream, steps, warmup)
    out = {"ms_per_step": round(ms, 5), "step": _dist_us(each),
           "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
           "frac_measured": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "layers": {}}
    # `repeats` copies of the layer set, in decoder order, distinct seeds
    big, big_ys = [], []
    for r in range(repeats):
        for i, (dt, M, N, K, bias, name, act) in enumerate(specs):
            Lr = inputs.make_layer(dt, M, N, K, bias=bias, config_id=cfg, layer_idx=100 + 4 * r + i,
                                   device=dev)
            Lr.act = act
            big.append((name, Lr))
            big_ys.append(out_buffer(Lr, dev))
    ms_big, _, _ = stream_rate(torch, dl, big, big_ys, stream, steps // 2, warmup)
    ws = dl.Workspace.for_shapes([(L.M, L.N, L.K, dl.BF16 if L.dtype == "bf16" else dl.FP8_B128)
                                  for _, L in layers], dev)
    for j, (name, L) in enumerate(layers):
        b = out_bytes(L)
        keep = [q for q in range(len(big)) if big[q][0] != name]
        ms_rest, _, _ = stream_rate(torch, dl, [big[q] for q in keep], [big_ys[q] for q in keep],
                                    stream, steps // 2, warmup)
        d = (ms_big - ms_rest) / repeats
        rest = [layers[i] for i in range(len(layers)) if i != j]
        ms_rest4, _, _ = stream_rate(torch, dl, rest, [ys[i] for i in range(len(layers)) if i != j],
                                     stream, steps, warmup)
        d4 = ms - ms_rest4
        # single calls rotate over the copies (at least ceil(3 L2 / bytes) of them)
        copies = [q for q in range(len(big)) if big[q][0] == name]
        assert len(copies) >= cold_copies(L, l2)
        calls = [layer_call(dl, big[q][1], big_ys[q], ws, stream) for q in copies]
        call = single_call_times(torch, dl, calls, stream, 30)[5:]
        med = statistics.median(call)
        out["layers"][name] = {
            "bytes": b,
            "in_stream_us": round(d * 1e3, 3),
            "in_stream_frac": round(b / (d * 1e-3) / 1e9 / peak, 4) if d > 0 else None,
            "in_stream_4_layer_graph_us": round(d4 * 1e3, 3),
            "in_stream_4_layer_graph_frac": round(b / (d4 * 1e-3) / 1e9 / peak, 4) if d4 > 0 else None,
            "single_call": {**_dist_us(call), "copies": len(calls)},
            "single_call_frac": round(b / (med * 1e-3) / 1e9 / peak, 4)}
    out["in_stream_method"] = (f"in_stream_us = (time of a stream of {repeats} copies of the 4 layers, "
                               f"distinct weights, one graph - the same stream without every copy of "
                               f"the layer) / {repeats}; in_stream_4_layer_graph_us = the 4-layer "
                               f"graph minus the graph without the layer")
    del layers, ys, big, big_ys
    return out


def run_ours(args, rank, world, dist):
    import torch
    import weight_streaming_skinny_gb300 as dl
    from weight_streaming_skinny_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dl.load()
    dl.set_override({"auto": 0, "simt": 1, "mma": 2, "tc": 3}[args.kernel], 0, 0)
    workload = args.workload
    is_model = workload == "qwen72b_model_fp8_m1"
    layers = build_layers(workload, dev)
    ys = [out_buffer(L, dev) for _, L in layers]
    for j in range(1, len(layers)):
        if layers[j][1].x is None:
            layers[j][1].x = ys[j - 1]
    stream = torch.cuda.Stream(dev)
    # algorithmic bytes (a SwiGLU layer writes M x N/2 outputs, an argmax layer M indices)
    nbytes = [out_bytes(L) for _, L in layers]
    step_bytes = sum(nbytes)
    dl_layers = make_dl_layers(dl, layers, ys)
    # the stream's workspace: room for the up-front FP8 activation copies
    ws = dl.Workspace.for_stream(dl_layers)
    # kernels per step: calls mode one per layer plus a prep per FP8 layer; else
    # the library's own count for the stream (prep launches included)
    launches_per_step = (sum(1 if L.dtype == "bf16" else 2 for _, L in layers) if args.mode == "calls"
                         else dl.decode_stream_launches(dl_layers, ws))
    linear_launches = len(layers)
    use_graph = args.mode == "graph"
    torch.cuda.synchronize(dev)

    def step():
        if args.mode == "calls":
            for j, (_, L) in enumerate(layers):
                launch(dl, L, ys[j], ws, stream)
        else:
            dl.decode_stream(dl_layers, ws, use_graph=use_graph, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()

    # ---- timed region: exactly K steps, CUDA events on the launching stream
    # (an event after every step, for the per-step distribution)
    K = args.steps
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.05)
    total_ms_local, per_step = time_steps(torch, step, stream, K)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    # keep the same load running (untimed) until the clock record has samples
    extra_steps = 0
    deadline = time.time() + 3.0
    while len(sampler.lines) < 5 and time.time() < deadline:
        with torch.cuda.stream(stream):
            for _ in range(10):
                step()
        stream.synchronize()
        extra_steps += 10
    sampler.stop()
    total_s, value = replica_rate(total_ms_local * 1e-3, step_bytes * K, dist, world)
    ms_per_step = total_s * 1e3 / K
    # the same K steps once more, untimed by the contract: the two runs must
    # agree within 0.5 % to be accepted
    rep_ms, _ = time_steps(torch, step, stream, K, per_step=False)
    repeat = {"ms_per_step": round(rep_ms / K, 5),
              "rel_diff": round(abs(rep_ms / K - total_ms_local / K) / (total_ms_local / K), 5)}
    repeat["agree_within_0.5pct"] = repeat["rel_diff"] <= 0.005

    peak, peak_kind = measured_peak()

    # ---- isolated single calls (events around each call; untimed).  Layer
    # workloads: every layer; the model: its five shapes, each cycled through
    # distinct decoder layers so that no call finds its weights in L2.
    per_layer = {}
    if not args.skip_extras:
        R = 40
        if is_model:
            shapes = {}
            for j, (name, L) in enumerate(layers):
                shapes.setdefault(name.split(".")[0], []).append(j)
            for name, idxs in shapes.items():
                calls = [layer_call(dl, layers[j][1], ys[j], ws, stream) for j in idxs[:R]]
                t = single_call_times(torch, dl, calls, stream, R + 5)[5:]
                b = nbytes[idxs[0]]
                med = statistics.median(t)
                per_layer[name] = {"bytes": b, "count_per_token": len(idxs), **_dist_us(t),
                                   "GB/s": round(b / (med * 1e-3) / 1e9, 1),
                                   "frac_measured": round(b / (med * 1e-3) / 1e9 / peak, 4)}
        else:
            for j, (name, L) in enumerate(layers):
                t = single_call_times(torch, dl, [layer_call(dl, L, ys[j], ws, stream)], stream, R + 5)[5:]
                med = statistics.median(t)
                b = nbytes[j]
                per_layer[name] = {"bytes": b, **_dist_us(t), "GB/s": round(b / (med * 1e-3) / 1e9, 1),
                                   "frac_measured": round(b / (med * 1e-3) / 1e9 / peak, 4)}

    # ---- end to end through the public API with host buffers: every step
    # copies the step's inputs host -> device (the layers' x that no earlier
    # layer produces) and its results device -> host (the y that no later layer
    # reads), each side staged in one pinned host buffer and one device buffer
    # so that a step issues one copy each way.
    e2e = None
    if not args.skip_e2e:
        chained_in = [j > 0 and layers[j][1].x is ys[j - 1] for j in range(len(layers))]
        chained_out = [j + 1 < len(layers) and chained_in[j + 1] for j in range(len(layers))]

        def staged(tensors):
            offs, n = [], 0
            for t in tensors:
                offs.append(n)
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            return offs, max(n, 256)

        xin = [(j, L.x) for j, (_, L) in enumerate(layers) if not chained_in[j]]
        yout = [(j, ys[j]) for j in range(len(layers)) if not chained_out[j]]
        xo, xn = staged([t for _, t in xin])
        yo, yn = staged([t for _, t in yout])
        dx = torch.empty(xn, dtype=torch.uint8, device=dev)
        dy = torch.empty(yn, dtype=torch.uint8, device=dev)
        hx = torch.zeros(xn, dtype=torch.uint8).pin_memory()
        hy = torch.empty(yn, dtype=torch.uint8).pin_memory()

        def view(buf, off, like):
            nb = like.numel() * like.element_size()
            return buf[off:off + nb].view(like.dtype).view(like.shape)

        xs_e2e, ys_e2e = {}, {}
        for (j, t), o in zip(xin, xo):
            view(hx, o, t).copy_(t.cpu())
            xs_e2e[j] = view(dx, o, t)
        for (j, t), o in zip(yout, yo):
            ys_e2e[j] = view(dy, o, t)
        y_of = [ys_e2e.get(j, ys[j]) for j in range(len(layers))]
        x_of = [xs_e2e[j] if j in xs_e2e else y_of[j - 1] for j in range(len(layers))]
        e2e_layers = [dl.Layer(Ld.dtype, x_of[j], Ld.w, y_of[j], Ld.scales, Ld.bias, act=Ld.act)
                      for j, Ld in enumerate(dl_layers)]
        ws_e2e = dl.Workspace.for_stream(e2e_layers)
        h2d = sum(t.numel() * t.element_size() for _, t in xin)
        d2h = sum(t.numel() * t.element_size() for _, t in yout)
        E = max(3, min(K, 50))

        def e2e_body(graphed_layers):
            dx.copy_(hx, non_blocking=True)
            if args.mode == "calls":
                for j, (_, L) in enumerate(layers):
                    Lj = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, x_of[j], L.w, L.scales, L.bias)
                    Lj.act = L.act
                    launch(dl, Lj, y_of[j], ws_e2e, stream)
            else:
                dl.decode_stream(e2e_layers, ws_e2e, use_graph=graphed_layers, stream=stream)
            hy.copy_(dy, non_blocking=True)

        # graph mode: the whole step -- input copy, the layers, result copy --
        # is captured once as one CUDA graph (the library's launches recorded
        # into it) and replayed each step, as a decode loop would run it.
        step_graph = None

        def e2e_step():
            if step_graph is not None:
                step_graph.replay()
            else:
                e2e_body(use_graph)
            stream.synchronize()

        with torch.cuda.stream(stream):
            for _ in range(2):
                e2e_step()
            if use_graph:
                step_graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(step_graph, stream=stream, capture_error_mode="thread_local"):
                    e2e_body(False)
                for _ in range(2):
                    e2e_step()
            if dist is not None:
                dist.barrier()
            a = time.perf_counter()
            for _ in range(E):
                e2e_step()
            el = time.perf_counter() - a
        el, e2e_gbs = replica_rate(el, step_bytes * E, dist, world)
        e2e = {"value": round(e2e_gbs, 2), "unit": "GB/s",
               "ms_per_step": round(el / E * 1e3, 4), "steps": E,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "each step: the inputs copied host->device and the results device->host "
                       "(one staged copy each way, pinned host memory), weights resident in HBM, "
                       "a host synchronisation after every step" +
                       ("; the copies and the layers replayed as one captured CUDA graph"
                        if use_graph else "")}
        if is_model:
            e2e["ms_per_token"] = e2e["ms_per_step"]
        del step_graph

    # ---- roofline of the dominant kernel, linear_kernel (one launch per
    # layer; the FP8 activation-copy launches hold ~3 % of the serialised
    # kernel time).  Under programmatic dependent launch consecutive launches
    # overlap, so a launch's duration inside the step is taken as the step
    # time divided by the linear launches per step; the isolated duration (an
    # event pair around each call) is given beside it.
    kname = "linear_kernel"
    step_avg_ms = ms_per_step / linear_launches
    bytes_per_launch = step_bytes / linear_launches
    achieved = bytes_per_launch / (step_avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": recorded_traffic(workload, kname),
                "kernel": kname, "bytes_per_launch_avg": int(bytes_per_launch),
                "launches_per_step": linear_launches,
                "step_avg_launch_us_under_pdl": round(step_avg_ms * 1e3, 3),
                "duration": "step time / linear_kernel launches per step (CUDA events over the "
                            "timed region; launches overlap under programmatic dependent launch)"}
    if per_layer:
        if is_model:
            iso_us = sum(v["median_us"] * v["count_per_token"] for v in per_layer.values())
            iso_launch_us = iso_us / linear_launches
        else:
            iso_launch_us = sum(v["median_us"] for v in per_layer.values()) / linear_launches
        iso = bytes_per_launch / (iso_launch_us * 1e-6) / 1e9
        roofline["isolated"] = {"avg_launch_us": round(iso_launch_us, 3), "achieved": round(iso, 1),
                                "frac": round(iso / peak, 4),
                                "note": "median single-call times (an event pair around each call, "
                                        "FP8 calls include their activation-copy launch), weighted "
                                        "by launches per step"}
    res = {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 5), "e2e": e2e,
        "step_distribution": _dist_us(per_step), "repeat": repeat,
        "roofline": roofline, "per_layer": per_layer, "clocks": sampler.summary(),
        "ceiling_ms_at_measured_peak": round(step_bytes / (peak * 1e9) * 1e3, 4),
        "clock_window": f"timed region + {extra_steps} untimed steps of the same workload",
        "gpu_launches": launches_per_step * K, "step_bytes": step_bytes,
    }
    if is_model:
        res["ms_per_token"] = round(ms_per_step, 4)

    # ---- the whole token without graph capture: the same layer list enqueued
    # launch by launch from the host on every step (programmatic dependent
    # launch kept), after the timed region
    if is_model and not args.skip_extras and use_graph:
        ng_step = lambda: dl.decode_stream(dl_layers, ws, use_graph=False, stream=stream)  # noqa: E731
        with torch.cuda.stream(stream):
            for _ in range(3):
                ng_step()
        stream.synchronize()
        ng_ms, ng_each = time_steps(torch, ng_step, stream, 20)
        res["no_graph"] = {"ms_per_token": round(ng_ms / 20, 4), "step": _dist_us(ng_each),
                           "GB/s": round(step_bytes / (ng_ms / 20 * 1e-3) / 1e9, 1),
                           "note": "dl_decode_stream without graph capture: every step enqueues "
                                   "its launches from the host"}

    # ---- the other single-GPU configurations, after the timed region
    if is_model and not args.skip_extras:
        del dl_layers, ws
        extra = {}
        for wl in ("qwen72b_layer_bf16_m1", "qwen72b_layer_fp8_m6"):
            extra[wl] = layer_config_summary(torch, dl, wl, dev, stream, peak)
        # the 1024 x 1024 bf16 GEMV with bias, a latency configuration:
        # microseconds per isolated call, warm (its 2.1 MB stay in L2 from one
        # call to the next) and cold (calls rotated over ceil(3 L2 / 2.1 MB)
        # distinct copies of the layer, so that each call's bytes were evicted)
        L0 = inputs.make_layer(inputs.DTYPE_BF16, 1, 1024, 1024, bias=True, config_id=0, device=dev)
        L0.act = 0
        y0 = out_buffer(L0, dev)
        ws0 = dl.Workspace(dl.workspace_bytes(1, 1024, 1024, dl.BF16), dev)
        t = single_call_times(torch, dl, [layer_call(dl, L0, y0, ws0, stream)], stream, 220)[20:]
        n_cold = cold_copies(L0, torch.cuda.get_device_properties(dev).L2_cache_size)
        cold = []
        for i in range(n_cold):
            Li = inputs.make_layer(inputs.DTYPE_BF16, 1, 1024, 1024, bias=True, config_id=0,
                                   layer_idx=i + 1, device=dev)
            Li.act = 0
            cold.append(layer_call(dl, Li, out_buffer(Li, dev), ws0, stream))
        tc = single_call_times(torch, dl, cold, stream, 2 * n_cold + 20)[20:]
        extra["gemv_bf16_1024_m1"] = {**_dist_us(t), "bytes": L0.algorithmic_bytes,
                                      "note": "latency configuration: 2.1 MB, L2-resident after "
                                              "the first call",
                                      "cold_l2": {**_dist_us(tc), "copies": n_cold,
                                                  "note": "calls rotated over distinct copies "
                                                          "(3 x L2 bytes in all)"}}
        del cold
        res["configs"] = extra
    return res, layers

def _host_copy(L):
    """LayerInputs on the host, keeping the `act` attribute."""
    H = L.to("cpu")
    H.act = getattr(L, "act", 0)
    return H


def cpu_oracle_gbs(layers_host, budget_s: float, row_frac: float = 1.0, threads=None):
    """Oracle GB/s over a bounded sample: row_frac of every layer's rows, repeated
    passes until budget_s of CPU time (at least one pass); all host cores
    unless `threads` is given."""
    import numpy as np
    import oracle
    from weight_streaming_skinny_gb300 import inputs
    prepared = []
    for name, L in layers_host:
        act = getattr(L, "act", 0)
        ncols = L.N // 2 if act == 1 else L.N
        n = max(1, int(ncols * row_frac))                 # outputs (or logits) computed
        cols = np.linspace(0, ncols - 1, n).astype(np.int64)
        nw = 2 * n if act == 1 else n                     # weight rows read
        xb = inputs.bf16_bits(L.x)
        bb = None if L.bias is None else inputs.bf16_bits(L.bias)
        if L.dtype == "bf16":
            args = (oracle.BF16, xb, inputs.bf16_bits(L.w), None, bb)
            wbytes = 2 * nw * L.K
        else:
            args = (oracle.FP8_B128, xb, inputs.u8_codes(L.w), L.scales.cpu().numpy(), bb)
            wbytes = nw * L.K + 4 * ((nw + 127) // 128) * (L.K // 128)
        ybytes = 4 * L.M if act == 2 else 2 * L.M * n
        prepared.append((args, cols, act,
                         wbytes + 2 * L.M * L.K + ybytes + (2 * nw if bb is not None else 0)))
    threads = threads or oracle.default_threads()
    passes, t_total, b_total = 0, 0.0, 0
    while passes == 0 or t_total < budget_s:
        for args, cols, act, b in prepared:
            a = time.perf_counter()
            if act == 1:
                oracle.swiglu(*args[:3], scales=args[3], bias_bits=args[4], outputs=cols,
                              threads=threads)
            else:
                y = oracle.linear(*args[:3], scales=args[3], bias_bits=args[4], rows=cols,
                                  with_abs=False, threads=threads)
                if act == 2:
                    oracle.argmax_lowest(y)
            t_total += time.perf_counter() - a
            b_total += b
        passes += 1
    return b_total / t_total / 1e9, threads, passes, t_total


def dtype_label(workload, specs) -> str:
    """The arithmetic the workload's path computes in."""
    if workload == "qwen72b_model_fp8_m1":
        return ("fp8_e4m3 weights x bf16 activations (80 layers), bf16 lm_head; fp32 accumulate")
    if {s_[0] for s_ in specs} == {"bf16"}:
        return "bf16"
    return "fp8_e4m3 weights x bf16 activations; fp32 accumulate"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen72b_model_fp8_m1", choices=WORKLOADS)
    ap.add_argument("--mode", choices=["graph", "stream", "calls"], default="graph",
                    help="graph: one dl_decode_stream CUDA-graph replay per step (default); "
                         "stream: dl_decode_stream without a graph; calls: one API call per layer")
    ap.add_argument("--kernel", choices=["auto", "simt", "mma", "tc"], default="auto",
                    help="force a kernel family (default: the library's automatic choice)")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the end-to-end leg")
    ap.add_argument("--skip-extras", action="store_true",
                    help="omit the single-call and other-configuration measurements")
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
              "l2": ("L2-resident: a latency case, its 2.1 MB are L2 hits after the first "
                     "step (cold-L2 calls: the model line's configs.gemv_bf16_1024_m1.cold_l2)"
                     if args.workload == "gemv_bf16_1024_m1" else
                     "inputs larger than L2: every step streams every weight matrix of the "
                     "workload (each step >= 0.7 GB) through a 129 MB L2"),
              "parallelism": f"replicas x{world}", "kernel_family": args.kernel,
              "mode": args.mode}
    if len(specs) > 8:
        config["layers"] = {"count": len(specs), "decoder_layers": len(specs) // 4,
                            "per_layer": [s[5].split(".")[0] + ("+swiglu" if s[6] else "")
                                          for s in specs[:4]],
                            "dtype": specs[0][0], "M": specs[0][1],
                            "lm_head": "bf16 152064x8192 with the fused argmax (token ids, no logits)",
                            "chaining": "down -> next qkv, o -> gate_up, gate_up (SwiGLU) -> down, "
                                        "last down -> lm_head"}

    if args.impl == "reference":
        if rank != 0:
            return
        import torch
        if args.workload in ("qwen72b_model_fp8_m1", "qwen72b_decoder_fp8_m1"):
            # bounded sample: decoder layer 0 (and the lm_head), each layer
            # with its own seeded x (not 72 GB of host weights)
            from weight_streaming_skinny_gb300 import inputs
            specs_all, cfg = layer_specs(args.workload)
            layers = []
            for i in sorted({0, 1, 2, 3, len(specs_all) - 1}):
                dt, M, N, K, bias, name, act = specs_all[i]
                Lh = inputs.make_layer(dt, M, N, K, bias=bias, config_id=cfg, layer_idx=i, device="cpu")
                Lh.act = act
                layers.append((name, Lh))
            which = "decoder layer 0's four linears and the lm_head"
        else:
            layers = build_layers(args.workload, "cpu")
            which = "the workload's linears"
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
                "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(args.workload, specs),
                "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                                 "kind": "oracle",
                                 "sample": f"{int(sample_frac * 100)}% of the output rows of each "
                                           f"of {which} (all K), one pass per step"},
                "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    res, layers = run_ours(args, rank, world, dist)
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        if len(layers) > 8:
            pick = [0, 1, 2, 3, len(layers) - 1]
            host_layers = [(layers[i][0], _host_copy(layers[i][1])) for i in pick]
            what = ("decoder layer 0 (QKV, O, gate_up, down) and the lm_head, all rows; GB/s "
                    "applies to the whole 80-layer stream by extrapolation")
        else:
            host_layers = [(n, _host_copy(L)) for n, L in layers]
            what = "the whole step (all rows of the four linears)"
        v, threads, passes, t = cpu_oracle_gbs(host_layers, args.cpu_budget_s, 1.0)
        cpu = {"value": round(v, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{what}, {passes} pass(es), {t:.1f} s of oracle time"}
        # the same oracle on one host core, over a quarter of the rows
        v1, th1, p1, t1 = cpu_oracle_gbs(host_layers, args.cpu_budget_s / 3, 0.25, threads=1)
        cpu["one_core"] = {"value": round(v1, 3), "unit": "GB/s", "cores": th1,
                           "sample": f"25% of the output rows of the same layers, {p1} pass(es), "
                                     f"{t1:.1f} s of oracle time"}
    if rank == 0:
        is_model = args.workload == "qwen72b_model_fp8_m1"
        line = {"metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": dtype_label(args.workload, specs),
                "data": "synthetic (seeded; no trained weights)",
                "config": config, "roofline": res["roofline"], "cpu_baseline": cpu,
                "e2e": res["e2e"], "clocks": res["clocks"], "clock_window": res["clock_window"],
                "gpu_launches": res["gpu_launches"],
                "step_distribution": res["step_distribution"], "repeat": res["repeat"],
                "per_layer": res["per_layer"],
                "ceiling_ms_at_measured_peak": res["ceiling_ms_at_measured_peak"],
                "step_bytes": res["step_bytes"], "kernel_hash": kernel_hash()}
        if is_model:
            line["ms_per_token"] = res["ms_per_token"]
            line["ceiling_ratio"] = round(res["ceiling_ms_at_measured_peak"] / res["ms_per_token"], 4)
        for k in ("no_graph", "configs"):
            if k in res:
                line[k] = res[k]
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

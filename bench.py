"""Benchmark of the FP4 MoE decode layer on GB300.

Metric: microseconds per MoE layer (and the weight-stream GB/s it implies, as a
fraction of the measured HBM bandwidth) on the NVFP4 MTP decode workload:
T=4 token rows, E=256 experts, top-8, hidden 2048, intermediate 512, SwiGLU.

A step is one decode step of a 40-layer model: 40 calls of
qmoe_fp4_moe_forward (one kernel each for routing -> FC1 GEMV + SwiGLU -> FC2 GEMV ->
weighted un-permute, on a primed workspace: no per-call counter reset, each kernel launched
with programmatic dependent launch behind the previous one), each on its own layer's weights
(17 GB in total, far larger than the 129 MB L2), replayed as one CUDA graph.  Inputs are seeded
synthetic data with the workload's shapes and distributions.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the plain CPU oracle (the reference arm of this
project) on a bounded sample of the same workload, on the host's cores.
Multi-GPU runs are independent replicas (the layer has no cross-GPU step
here): one process per GPU under torchrun, max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "nvfp4_mtp_decode"
# DRAM bytes (read + write) of one moe_layer_kernel launch on this workload,
# from one ncu capture of the current kernel; None whenever the kernel changes
# and has not been captured again.
LAYER_TRAFFIC_BYTES = 55054336 + 395264
LAYER_TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one moe_layer_kernel launch of the "
                        "current build (python bench.py --profile-case nvfp4_mtp_decode --layers 3; first layer)")
LAYERS = 40
METRIC = "us per MoE layer (NVFP4 MTP decode, T=4 E=256 top-8 H=2048 I=512)"
UNIT = "us/layer"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_seconds: float, layers_per_rank: int, world: int) -> dict:
    """Replica aggregation: the job's time is the slowest rank's; the job
    processed layers_per_rank * world layers in it."""
    t = reduce_max(per_rank_seconds, world)
    total_layers = layers_per_rank * world
    return dict(seconds=t, total_layers=total_layers, us_per_layer=t * 1e6 / total_layers)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) with host
    timestamps, so the ones inside the timed region can be picked."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 6:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._t is not None:
            self._t.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "inside timed region"
        if not inside and self.samples:
            nearest = min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))
            inside, note = [nearest[1]], "nearest sample (timed region shorter than the 50 ms period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[2 + i].lower() == "active"})
        sm = [float(p[0]) for p in inside if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in inside if p[1].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------- workload

def make_layers(n_layers: int, seed: int, device, workload: str = WORKLOAD):
    """Seeded synthetic layers of a decode workload, generated on the GPU
    (weights, with the workload's distributions) and with the shared host
    generator (activations, logits)."""
    import numpy as np
    import torch
    import synthetic as syn
    wl = syn.WORKLOADS[workload]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    layers = []
    E, H, I = wl.E, wl.H, wl.I
    bs = 16 if wl.fmt == 0 else 32

    def scales(shape):
        if wl.fmt == 0:  # E4M3 codes with value in [0.25, 4): exponent field 5..8, any mantissa
            idx = torch.randint(0, 32, shape, generator=gen, device=device, dtype=torch.int32)
            return (((idx // 8) + 5) << 3 | (idx % 8)).to(torch.uint8)
        return torch.randint(120, 135, shape, generator=gen, device=device, dtype=torch.int32).to(torch.uint8)

    def gscale():
        if wl.fmt != 0:
            return None
        u = torch.randint(0, 5, (E,), generator=gen, device=device, dtype=torch.int32)
        return torch.ldexp(torch.ones(E, device=device), -u.float()).float()

    for li in range(n_layers):
        rng = syn.rng_for(seed, 100 + li)
        x = torch.from_numpy(syn.activations(rng, wl.T, H).view(np.int16)).to(device).view(torch.bfloat16)
        lg = torch.from_numpy(syn.logits(rng, wl.T, E, wl.logit_std, wl.ties, wl.k)).to(device)
        w1 = torch.randint(0, 256, (E, H, I), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
        w2 = torch.randint(0, 256, (E, I, H // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
        layers.append(dict(x=x, logits=lg, w1=w1, s1=scales((E, 2 * I, H // bs)), g1=gscale(),
                           w2=w2, s2=scales((E, H, I // bs)), g2=gscale()))
    return wl, layers


def per_expert_bytes(wl):
    bs = 16 if wl.fmt == 0 else 32
    fc1 = wl.H * wl.I + 2 * wl.I * (wl.H // bs)
    fc2 = wl.I * (wl.H // 2) + wl.H * (wl.I // bs)
    return fc1, fc2


def run_gpu(args):
    import torch
    import block_scaled_fp4_gb300 as q
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    q.build()
    q.load()
    global LAYERS
    LAYERS = args.layers
    wl, layers = make_layers(LAYERS, seed=1234 + rank, device=device)
    fmt = wl.fmt
    if args.scales == "kmajor":
        # weight-load-time preparation, outside every timed region: the block
        # scales of both FCs in the k-major layout
        for L in layers:
            L["s1"] = q.scales_kmajor(L["s1"], wl.fmt)
            L["s2"] = q.scales_kmajor(L["s2"], wl.fmt)
        fmt = wl.fmt | q.SCALES_KMAJOR
        torch.cuda.synchronize()
    if not args.no_primed:
        fmt |= q.WORKSPACE_PRIMED  # the header is zeroed here, once; the kernels keep it zero
    ws_bytes = q.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, fmt)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device) for _ in layers]
    ids = [torch.empty((wl.T, wl.k), dtype=torch.int32, device=device) for _ in layers]
    stream = torch.cuda.Stream(device=device)
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())

    def step(lst=layers):
        for i, L in enumerate(lst):
            q.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                          fmt, wl.k, wl.normalize, out=outs[i], topk_ids=ids[i], workspace=ws)

    # --- graph capture of one step (40 layers)
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    fc1_b, fc2_b = per_expert_bytes(wl)
    act = [len(set(i.cpu().numpy().reshape(-1).tolist())) for i in ids]
    alg_bytes_layer = [a * (fc1_b + fc2_b) + wl.T * wl.H * 2 * 2 + wl.T * wl.E * 4 for a in act]
    mean_alg = sum(alg_bytes_layer) / len(alg_bytes_layer)

    clocks = ClockSampler(device.index or 0)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(world)
    sec = ev0.elapsed_time(ev1) / 1e3
    clocks.stop()
    agg = aggregate(sec, args.steps * LAYERS, world)
    us_layer = agg["us_per_layer"]

    # --- eager (no graph) timing of the same steps, for reference
    with torch.cuda.stream(stream):
        step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n_eager = max(1, min(args.steps, 50))
        for _ in range(n_eager):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    eager_us = e0.elapsed_time(e1) * 1e3 / (n_eager * LAYERS)

    # --- per-kernel durations (stage events around each kernel, eager)
    n_inst = max(1, min(args.steps, 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_inst * LAYERS)]
    with torch.cuda.stream(stream):
        for j, L in enumerate(layers * n_inst):
            for e in evs[j]:
                e.record(stream)  # create the event objects
            q.set_stage_events(evs[j])
            q.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                          fmt, wl.k, wl.normalize, out=outs[j % LAYERS], workspace=ws)
        q.set_stage_events(None)
    torch.cuda.synchronize()
    names = ["layer"]  # one kernel per call (routing inside); without --no-primed no memset before it
    dur = {n: [] for n in names}
    for j in range(len(evs)):
        e = evs[j]
        for i, n in enumerate(names):
            dur[n].append(e[i].elapsed_time(e[i + 1]) * 1e3)
    kern_us = {k: statistics.mean(v) for k, v in dur.items()}
    # the fused layer kernel: active experts' FC1 + FC2 codes and scales, x in, out
    layer_bytes = [a * (fc1_b + fc2_b) + 2 * wl.T * wl.H * 2 for a in act]
    layer_alg = sum(layer_bytes) / len(layer_bytes)
    peak, peak_src = _peaks()
    # achieved: the kernel's average duration over the timed region, where it
    # is the only kernel (one launch per layer)
    layer_gbs = layer_alg / (us_layer * 1e-6) / 1e9

    # --- end to end: host buffers, H2D of each layer's inputs, D2H of each output
    hx = [L["x"].cpu().pin_memory() for L in layers]
    hl = [L["logits"].cpu().pin_memory() for L in layers]
    ho = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in layers]
    dx = [torch.empty_like(L["x"]) for L in layers]
    dl = [torch.empty_like(L["logits"]) for L in layers]
    n_e2e = max(1, min(args.steps, 50))

    def e2e_step():
        for i, L in enumerate(layers):
            dx[i].copy_(hx[i], non_blocking=True)
            dl[i].copy_(hl[i], non_blocking=True)
            q.moe_forward(dx[i], dl[i], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], fmt,
                          wl.k, wl.normalize, out=outs[i], workspace=ws)
            ho[i].copy_(outs[i], non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        x1.record(stream)
    torch.cuda.synchronize()
    e2e_agg = aggregate(x0.elapsed_time(x1) / 1e3, n_e2e * LAYERS, world)
    h2d = LAYERS * (wl.T * wl.H * 2 + wl.T * wl.E * 4)
    d2h = LAYERS * wl.T * wl.H * 2

    res = None
    if rank == 0:
        cpu = cpu_baseline(args) if (world == 1 and not args.no_cpu_baseline) else None
        stream_gbs = mean_alg / (us_layer * 1e-6) / 1e9 * world
        res = {
            "metric": METRIC, "value": round(us_layer, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(agg["seconds"] * 1e3 / args.steps, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "e2m1 x bf16 -> fp32 accumulate (bf16 out)", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: T=4 E=256 k=8 H=2048 I=512 NVFP4 SwiGLU",
                       "layers_per_step": LAYERS, "global_batch_tokens": wl.T * world,
                       "l2": "inputs larger than L2: 40 distinct layers, 17.3 GB of weights per step",
                       "graph": True, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "scale_layout": ("k-major [E, K/16, N], converted once at weight load"
                                        if args.scales == "kmajor" else "[E, N, K/16] as stored"),
                       "workspace": ("primed: zeroed once, no per-call reset, programmatic dependent launch"
                                     if not args.no_primed else "header reset by a memset before every call")},
            "weight_stream": {"alg_bytes_per_layer": int(mean_alg),
                              "mean_active_experts": statistics.mean(act),
                              "gbs": round(stream_gbs, 1), "frac_of_hbm": round(stream_gbs / (peak * world), 4),
                              "peak_gbs": peak, "peak_source": peak_src},
            "eager_us_per_layer": round(eager_us, 3),
            "kernel_us": {k: round(v, 3) for k, v in kern_us.items()},
            "roofline": {"kernel": "moe_layer_kernel (routing + FC1 + SwiGLU + FC2 + un-permute, E2M1 decode)",
                         "bound": "hbm", "achieved": round(layer_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(layer_gbs / peak, 4), "traffic": LAYER_TRAFFIC_BYTES,
                         "traffic_source": LAYER_TRAFFIC_SOURCE,
                         "alg_bytes_per_launch": int(layer_alg), "peak_source": peak_src},
            "gpu_launches": args.steps * LAYERS,
            "e2e": {"value": round(e2e_agg["us_per_layer"], 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks.summary(t_host0, t_host1),
            "cpu_baseline": cpu,
            "dequant": bench_dequant(device, peak) if not args.no_dequant else None,
            "dequant_fc2": (bench_dequant(device, peak, K=1536, N=2048, what="prefill FC2 weights")
                            if not args.no_dequant else None),
            "prefill": bench_prefill(device, peak) if not args.no_prefill else None,
            "routing": bench_routing(device) if not args.no_configs else None,
            "configs": bench_configs(args, device, peak) if not args.no_configs else None,
        }
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return res


# ---------------------------------------------------------------- other decode configs

# Which decode kernel each workload runs on with k-major scales (the library
# picks by the length of one SM's FC1 stream: short streams run the
# one-row-per-pass kernel, longer ones the multi-row kernel).
DECODE_KERNEL = {
    "tiny_nvfp4_decode": "moe_layer_kernel (one row per pass)",
    "nvfp4_mtp_decode": "moe_layer_kernel (one row per pass)",
    "mxfp4_decode": "moe_decode_kernel (multi-row)",
    "nvfp4_verify_edge": "moe_decode_kernel (multi-row)",
}
# DRAM bytes (read + write) of one launch of each workload's kernel, from ncu
# captures of the current kernels (per launch; the captured layer's active
# experts differ from the bench's mean, so compare with that layer's bytes);
# None where no capture of the current kernel exists.
DECODE_TRAFFIC = {
    "nvfp4_mtp_decode": {"bytes": 55054336 + 395264, "source": "ncu, first layer of --profile-case, --layers 3"},
    "nvfp4_verify_edge": {"bytes": 750515200 + 10542336, "source": "ncu, first layer of --profile-case, --layers 3"},
    "mxfp4_decode": {"bytes": 276891648 + 9066496, "source": "ncu, first layer of --profile-case, --layers 3"},
}

DECODE_CONFIGS = {
    # workload: (distinct layers per replay, why that many)
    "tiny_nvfp4_decode": (40, "0.44 MB of weights per layer: L2-resident whatever the rotation (launch-bound)"),
    "mxfp4_decode": (8, "8 distinct layers, 3.4 GB of weights per replay (> L2)"),
    "nvfp4_verify_edge": (4, "4 distinct layers, 13.8 GB of weights per replay (> L2)"),
}


def bench_decode(device, workload: str, n_layers: int, steps: int, peak: float, kmajor: bool = True,
                 cpu_tokens=None) -> dict:
    """One decode workload: n_layers distinct layers replayed as one CUDA graph
    (primed workspace), microseconds per layer, the algorithmic bytes of the
    experts the seeded routing activates, and the fraction of the measured HBM
    bandwidth; plus the oracle's host-core time on a bounded sample."""
    import torch
    import block_scaled_fp4_gb300 as q
    wl, layers = make_layers(n_layers, seed=4321, device=device, workload=workload)
    fmt = wl.fmt
    if kmajor:
        for L in layers:
            L["s1"] = q.scales_kmajor(L["s1"], wl.fmt)
            L["s2"] = q.scales_kmajor(L["s2"], wl.fmt)
        fmt |= q.SCALES_KMAJOR
    fmt |= q.WORKSPACE_PRIMED
    ws = torch.zeros(q.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, fmt), dtype=torch.uint8,
                     device=device)
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device) for _ in layers]
    ids = [torch.empty((wl.T, wl.k), dtype=torch.int32, device=device) for _ in layers]
    stream = torch.cuda.Stream(device=device)
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())

    def step():
        for i, L in enumerate(layers):
            q.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], fmt, wl.k,
                          wl.normalize, wl.alpha, wl.beta, wl.limit, out=outs[i], topk_ids=ids[i], workspace=ws)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    q.check_device_error(ws)
    us = e0.elapsed_time(e1) * 1e3 / (steps * len(layers))
    fc1_b, fc2_b = per_expert_bytes(wl)
    act = [len(set(i.cpu().numpy().reshape(-1).tolist())) for i in ids]
    alg = sum(a * (fc1_b + fc2_b) + 2 * wl.T * wl.H * 2 for a in act) / len(act)
    gbs = alg / (us * 1e-6) / 1e9
    res = {"workload": f"{workload}: T={wl.T} E={wl.E} k={wl.k} H={wl.H} I={wl.I} "
                       f"{'NVFP4' if wl.fmt == 0 else 'MXFP4'} SwiGLU",
           "kernel": DECODE_KERNEL[workload] if kmajor else "moe_layer_kernel (scales as stored)",
           "traffic": DECODE_TRAFFIC.get(workload) if kmajor else None,
           "us_per_layer": round(us, 3), "alg_bytes_per_layer": int(alg),
           "mean_active_experts": sum(act) / len(act), "achieved_gbs": round(gbs, 1), "peak": peak,
           "frac": round(gbs / peak, 4), "layers_per_replay": len(layers), "replays": steps,
           "scale_layout": "k-major" if kmajor else "[E, N, K/bs] as stored"}
    del layers, ws, graph
    torch.cuda.empty_cache()
    if cpu_tokens is not None:
        res["cpu_oracle"] = cpu_oracle_sample(workload, cpu_tokens)
    return res


def cpu_oracle_sample(workload: str, tokens) -> dict:
    """The fp64 oracle on the host cores for `tokens` of one layer, scaled to
    microseconds per whole layer (time x T / tokens)."""
    import numpy as np
    import oracle
    import synthetic as syn
    wl = syn.WORKLOADS[workload]
    oracle.build()
    cores = os.cpu_count() or 1
    L = syn.layer(wl, seed=0)
    tok = np.asarray(tokens, np.int32)
    t0 = time.perf_counter()
    oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], wl.fmt, wl.k,
                       wl.normalize, wl.alpha, wl.beta, wl.limit, tokens=tok, nthreads=cores)
    sec = time.perf_counter() - t0
    return {"value": round(sec * 1e6 * wl.T / len(tok), 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(tok)} of {wl.T} tokens of one layer, scaled to the whole layer"}


def bench_routing(device, reps: int = 200) -> dict:
    """qmoe_route_topk alone on the MTP decode shape (4 tokens, 256 experts,
    top-8): 40 calls on distinct logits replayed as one CUDA graph."""
    import torch
    import block_scaled_fp4_gb300 as q
    import synthetic as syn
    wl = syn.WORKLOADS[WORKLOAD]
    lg = [torch.from_numpy(syn.logits(syn.rng_for(7, i), wl.T, wl.E, wl.logit_std)).to(device) for i in range(40)]
    stream = torch.cuda.Stream(device=device)
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for x in lg:
            q.route_topk(x, wl.k, wl.normalize, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for x in lg:
            q.route_topk(x, wl.k, wl.normalize, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = max(1, reps // 40)
        for _ in range(n):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (n * len(lg))
    return {"kernel": "route_maps_fused_kernel (top-k softmax + permute maps, one launch)",
            "workload": f"T={wl.T} E={wl.E} k={wl.k}", "us_per_call": round(us, 3), "bound": "latency",
            "calls": n * len(lg)}


def bench_configs(args, device, peak: float) -> dict:
    """Every other decode workload, and the MTP decode workload with its block
    scales in the stored [E, N, K/bs] layout."""
    out = {}
    cpu = not args.no_cpu_baseline
    samples = {"tiny_nvfp4_decode": [0], "mxfp4_decode": [0], "nvfp4_verify_edge": [0]}
    for name, (n_layers, why) in DECODE_CONFIGS.items():
        r = bench_decode(device, name, n_layers, max(5, args.steps // 4), peak,
                         cpu_tokens=samples[name] if cpu else None)
        r["l2"] = why
        out[name] = r
    r = bench_decode(device, WORKLOAD, LAYERS, max(5, args.steps // 4), peak, kmajor=False)
    r["l2"] = "40 distinct layers, 17.3 GB of weights per replay (> L2)"
    out[WORKLOAD + " (page-layout scales)"] = r
    return out


# ---------------------------------------------------------------- prefill dequant

def bench_dequant(device, peak: float, reps: int = 10, E: int = 128, K: int = 2048, N: int = 3072,
                  what: str = "prefill FC1 weights") -> dict:
    """The prefill FP4 -> bf16 dequantisation on one FC of the NVFP4 prefill
    shape (FC1: E=128, K=2048, N=3072, 384 MiB codes + 48 MiB scales read,
    1.5 GiB bf16 written; FC2: K=1536, N=2048), far above L2 per launch.
    Event-timed on the launching stream, after warm-up."""
    import torch
    import block_scaled_fp4_gb300 as q
    gen = torch.Generator(device=device)
    gen.manual_seed(77)
    packed = torch.randint(0, 256, (E, K, N // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    idx = torch.randint(0, 32, (E, N, K // 16), generator=gen, device=device, dtype=torch.int32)
    scales = (((idx // 8) + 5) << 3 | (idx % 8)).to(torch.uint8)
    g = torch.ldexp(torch.ones(E, device=device),
                    -torch.randint(0, 5, (E,), generator=gen, device=device).float()).float()
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device=device)
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(3):
            q.dequant(packed, scales, g, q.NVFP4, out=out, stream=stream)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record(stream)
        for i in range(reps):
            q.dequant(packed, scales, g, q.NVFP4, out=out, stream=stream)
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    us = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(reps))
    med = us[len(us) // 2]
    alg = E * K * (N // 2) + E * N * (K // 16) + E * N * K * 2 + E * 4
    gbs = alg / (med * 1e-6) / 1e9
    del packed, scales, out
    return {"kernel": "dequant_kernel<NVFP4> (FP4 -> bf16, [E,K,N/2] -> [E,N,K])",
            "workload": f"E={E} K={K} N={N} NVFP4 ({what})", "us": round(med, 2),
            "us_p10_p90": [round(us[max(0, len(us) // 10)], 2), round(us[min(len(us) - 1, 9 * len(us) // 10)], 2)],
            "bound": "hbm", "alg_bytes": alg, "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "launches": reps}


# ---------------------------------------------------------------- prefill

def bench_prefill(device, hbm_peak: float, reps: int = 5) -> dict:
    """The prefill path on the NVFP4 prefill workload (2048 tokens, 128
    experts, top-8, H=2048, I=1536): the whole forward call with k-major block
    scales (routing, fused W4A16 GEMM for FC1 with SwiGLU, fused W4A16 GEMM for
    FC2, un-permute), the same with scales as stored (two scale rewrites
    more), and with bf16 dequantised weights given (the bf16 grouped GEMMs).
    Per-stage times from events recorded between the call's kernels.
    Event-timed on the launching stream after warm-up."""
    import numpy as np
    import torch
    import block_scaled_fp4_gb300 as q
    import synthetic as syn
    wl = syn.WORKLOADS["nvfp4_prefill"]
    T, E, k, H, I = wl.T, wl.E, wl.k, wl.H, wl.I
    gen = torch.Generator(device=device)
    gen.manual_seed(99)

    def codes(shape):
        return torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.int32).to(torch.uint8)

    def e4m3(shape):
        idx = torch.randint(0, 32, shape, generator=gen, device=device, dtype=torch.int32)
        return (((idx // 8) + 5) << 3 | (idx % 8)).to(torch.uint8)

    def gscale():
        return torch.ldexp(torch.ones(E, device=device),
                           -torch.randint(0, 5, (E,), generator=gen, device=device).float()).float()

    rng = syn.rng_for(1234, 7)
    x = torch.from_numpy(syn.activations(rng, T, H).view(np.int16)).to(device).view(torch.bfloat16)
    lg = torch.from_numpy(syn.logits(rng, T, E, wl.logit_std)).to(device)
    w1, s1, g1 = codes((E, H, I)), e4m3((E, 2 * I, H // 16)), gscale()
    w2, s2, g2 = codes((E, I, H // 2)), e4m3((E, H, I // 16)), gscale()
    s1k, s2k = q.scales_kmajor(s1, q.NVFP4), q.scales_kmajor(s2, q.NVFP4)
    w1d, w2d = q.dequant(w1, s1, g1, q.NVFP4), q.dequant(w2, s2, g2, q.NVFP4)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device=device)
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())
    KM = q.NVFP4 | q.SCALES_KMAJOR
    ws_page = torch.empty(q.forward_workspace_bytes(T, H, I, E, k, q.NVFP4), dtype=torch.uint8, device=device)
    ws_km = torch.empty(q.forward_workspace_bytes(T, H, I, E, k, KM), dtype=torch.uint8, device=device)
    ws_gemm = torch.empty(q.forward_workspace_bytes(T, H, I, E, k, q.NVFP4, True), dtype=torch.uint8, device=device)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
            ev[0].record(stream)
            for i in range(reps):
                fn()
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        us = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(reps))
        return us[len(us) // 2]

    def stages(fn):
        """median per-stage times (us) of `fn` with the six prefill stage events"""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(reps)]
        with torch.cuda.stream(stream):
            fn()
            for e6 in evs:
                for e in e6:
                    e.record(stream)
                q.set_stage_events(e6)
                fn()
            q.set_stage_events(None)
        torch.cuda.synchronize()
        names = ["route", "scale_rewrite", "fc1_gemm", "fc2_gemm", "unpermute"]
        res = {}
        for i, n in enumerate(names):
            v = sorted(e6[i].elapsed_time(e6[i + 1]) * 1e3 for e6 in evs)
            res[n] = round(v[len(v) // 2], 1)
        return res

    f_km = lambda: q.moe_forward(x, lg, w1, s1k, g1, w2, s2k, g2, KM, k, out=out, workspace=ws_km, stream=stream)
    f_page = lambda: q.moe_forward(x, lg, w1, s1, g1, w2, s2, g2, q.NVFP4, k, out=out, workspace=ws_page,
                                   stream=stream)
    f_bf16 = lambda: q.moe_forward(x, lg, w1, s1, g1, w2, s2, g2, q.NVFP4, k, w1_dequant=w1d, w2_dequant=w2d,
                                   out=out, workspace=ws_gemm, stream=stream)
    km = timed(f_km)
    page = timed(f_page)
    gemm = timed(f_bf16)
    st_km = stages(f_km)
    st_bf16 = stages(f_bf16)
    R = T * k
    flops1, flops2 = 2.0 * R * H * 2 * I, 2.0 * R * I * H
    flops = flops1 + flops2
    pbytes1 = E * (H * I + 2 * I * H // 16)   # FC1 packed codes + E4M3 scales
    pbytes2 = E * (I * H // 2 + H * I // 16)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    fc1_tf = flops1 / (st_km["fc1_gemm"] * 1e-6) / 1e12
    fc2_tf = flops2 / (st_km["fc2_gemm"] * 1e-6) / 1e12
    gemm_tf = flops / ((st_km["fc1_gemm"] + st_km["fc2_gemm"]) * 1e-6) / 1e12
    del w1d, w2d, ws_page, ws_km, ws_gemm
    return {"workload": f"nvfp4_prefill: T={T} E={E} k={k} H={H} I={I} NVFP4 SwiGLU",
            "us_forward_kmajor": round(km, 1), "us_forward": round(page, 1),
            "us_forward_predequantised": round(gemm, 1),
            "stages_us_kmajor": st_km, "stages_us_predequantised": st_bf16,
            "gemm_flops": int(flops), "tflops_fused_gemms": round(gemm_tf, 1),
            "tflops_fc1": round(fc1_tf, 1), "tflops_fc2": round(fc2_tf, 1),
            "tensor_peak_tflops": tc_peak, "tensor_frac_fc1": round(fc1_tf / tc_peak, 4),
            "tensor_frac_fused_gemms": round(gemm_tf / tc_peak, 4),
            "packed_weight_bytes": int(pbytes1 + pbytes2),
            "packed_weight_gbs_fc1": round(pbytes1 / (st_km["fc1_gemm"] * 1e-6) / 1e9, 1),
            "kernels": "route_topk + maps, gather_rows, fp4_grouped_gemm_kernel x2 (tcgen05.mma bf16 with the FP4 "
                       "weights decoded in shared memory, TMEM accumulators, clusters of 2 sharing activation rows "
                       "by multicast tensor copies), unpermute; scales as stored add transpose_bytes x2; the "
                       "predequantised call runs grouped_gemm_tc_kernel x2 instead of the fused GEMMs"}


# ---------------------------------------------------------------- CPU (oracle)

def cpu_baseline(args, budget_s: float | None = None) -> dict:
    """The CPU oracle, as it stands, on a bounded sample of the workload: whole
    layers (all 4 tokens), repeated until ~budget seconds of CPU work."""
    import oracle
    import synthetic as syn
    wl = syn.WORKLOADS[WORKLOAD]
    oracle.build()
    budget = budget_s if budget_s is not None else args.cpu_seconds
    cores = os.cpu_count() or 1
    L = syn.layer(wl, seed=0)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                           wl.fmt, wl.k, wl.normalize, nthreads=cores)
        n += 1
        if time.perf_counter() - t0 >= budget:
            break
    sec = time.perf_counter() - t0
    return {"value": round(sec * 1e6 / n, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} full layer(s) of {WORKLOAD} (4 tokens, 32 expert rows), fp64 oracle, "
                      f"OpenMP over (token, expert) pairs"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import synthetic as syn
    wl = syn.WORKLOADS[WORKLOAD]
    oracle.build()
    cores = os.cpu_count() or 1
    L = syn.layer(wl, seed=0)

    def one():
        oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                           wl.fmt, wl.k, wl.normalize, nthreads=cores)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    sec = time.perf_counter() - t0
    us = sec * 1e6 / args.steps
    sample = f"each step = 1 layer of {WORKLOAD} (a bounded sample of the 40-layer step)"
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp64 (oracle)", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: T=4 E=256 k=8 H=2048 I=512 NVFP4 SwiGLU",
                       "layers_per_step": 1},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(workload: str, n_layers: int) -> None:
    """A small case for ncu captures: n_layers distinct layers of one decode
    workload (k-major scales, primed workspace), or of the prefill workload
    (k-major scales), each run twice, eagerly."""
    import torch
    import block_scaled_fp4_gb300 as q
    device = torch.device("cuda", torch.cuda.current_device())
    q.build()
    q.load()
    wl, layers = make_layers(n_layers, seed=4321, device=device, workload=workload)
    for L in layers:
        L["s1"] = q.scales_kmajor(L["s1"], wl.fmt)
        L["s2"] = q.scales_kmajor(L["s2"], wl.fmt)
    fmt = wl.fmt | q.SCALES_KMAJOR | (q.WORKSPACE_PRIMED if workload in DECODE_KERNEL else 0)
    ws = torch.zeros(q.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, fmt), dtype=torch.uint8,
                     device=device)
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device) for _ in layers]
    for _ in range(2):
        for i, L in enumerate(layers):
            q.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], fmt, wl.k,
                          wl.normalize, wl.alpha, wl.beta, wl.limit, out=outs[i], workspace=ws)
    torch.cuda.synchronize()
    q.check_device_error(ws)
    print(f"profile case {workload}: {n_layers} layers x 2, ok")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="distinct layers per step (default 40; fewer only for small profiler runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-primed", action="store_true",
                    help="reset the workspace header before every call (no programmatic dependent launch)")
    ap.add_argument("--no-dequant", action="store_true", help="skip the prefill dequant measurement")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill forward measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other decode workloads, the page-layout line and the routing line")
    ap.add_argument("--scales", default="kmajor", choices=["kmajor", "page"],
                    help="block-scale layout the layer reads (default: k-major, prepared once at load)")
    ap.add_argument("--profile-case", default=None, choices=sorted(DECODE_KERNEL) + ["nvfp4_prefill"],
                    help="profiler helper: run --layers layers of one decode workload (or the prefill workload) "
                         "twice, eagerly, and exit (no timing, no JSON line)")
    args = ap.parse_args(argv)
    if args.profile_case:
        profile_case(args.profile_case, args.layers)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Throughput of the IQ4_NL MoE layer (libmoe) on GB300.

A step is one pass of the whole hot path over one batch: for every layer of
the workload, the router (moe_route_topk) and the layer (moe_iq4nl_decode, or
moe_iq4nl_prefill_grouped for the prefill workload). The default workload is
the Xing4.0-29B-A4B-shaped decode: 1 token through 38 MoE layers (hidden 3584,
64 experts top-4 + 1 shared, expert_ffn 1024, IQ4_NL), synthetic seeded data.

Prints one JSON line (rank 0). Metric: MoE-layer tokens/s (a token = one pass
through all layers of the workload), with the achieved HBM GB/s on distinct
expert bytes and its fraction of the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

Multi-GPU: replicas only (one independent copy of the workload per rank; no
collective on the data path), launched with torch.distributed.run.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer tokens/s and achieved HBM GB/s (% of roofline) at 1 GB300"
UNIT = "tokens/s"
N_SETS = 8
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1,
                    help="workload: 1 Xing decode (default), 2 Qwen3-Next paired decode, "
                         "3 DeepSeek-like wide decode, 4 Xing prefill chunk")
    ap.add_argument("--tokens", type=int, default=None, help="decode batch (config 3: 1/4/16)")
    ap.add_argument("--impl", default="libmoe", choices=["libmoe", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (small profiling cases)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 0.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


def workload(cfg: int, tokens, layers=None):
    import copy
    import synth
    s = synth.SHAPES[cfg]
    if layers is not None and layers < s.L:
        s = copy.copy(s)
        s.L = int(layers)
        s.name = f"{s.name} (first {s.L} layers)"
    T = s.T if tokens is None else int(tokens)
    if cfg != 4 and T > 16:
        T = 16
    return s, T


# ---------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle timing

def oracle_sample(cfg: int, T: int, budget_s: float = 20.0, threads=None, max_tokens: int = 16):
    """Time the oracle on the host cores: route + layer for T tokens of the
    workload, layer by layer, until the layers are done or the budget is spent.
    Returns (tokens/s through the whole layer stack, cores, description)."""
    import oracle
    import synth
    s = synth.SHAPES[cfg]
    seed = synth.seed_of(cfg)
    threads = threads or (os.cpu_count() or 1)
    T_full = T
    T = min(T, max_tokens)                       # a bounded sample of the chunk's tokens
    pairs = T * (s.k + s.n_shared)
    cores = max(1, min(threads, pairs))
    spent, layers = 0.0, 0
    for l in range(s.L):
        Wr, b = synth.router(s, seed, l)
        x = synth.x_rows(seed, l, s.H, T)
        t0 = time.perf_counter()
        ids, w, _, _ = oracle.route(Wr, b, x, s.k)
        spent += time.perf_counter() - t0
        experts = {int(e): synth.expert_mats(s, seed, l, int(e)) for e in np.unique(ids)}
        sh = synth.shared_mats(s, seed, l) if s.n_shared else None
        t0 = time.perf_counter()
        oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, s.n_shared, experts, sh, x, ids, w,
                         mode=oracle.EXACT, threads=threads)
        spent += time.perf_counter() - t0
        layers += 1
        if spent > budget_s:
            break
    # tokens/s through all L layers, scaled from the layers done
    tps = T * layers / s.L / spent
    desc = (f"{T} of {T_full} token(s) through {layers} of {s.L} layers (route + layer, exact "
            f"fp64), {spent:.1f} s, scaled to the full stack")
    return tps, cores, desc


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    s, T = workload(args.config, args.tokens)
    threads = os.cpu_count() or 1
    per = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        tps, cores, desc = oracle_sample(args.config, T, budget_s=6.0, threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            per.append((tps, dt))
    value = float(np.mean([p[0] for p in per]))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * float(np.mean([p[1] for p in per])),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": s.name, "tokens_per_step": T, "layers": s.L},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_libmoe(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import quantized_routed_expert_gb300 as moe
    import synth
    from synth.layers import Layer, x_sets

    s, T = workload(args.config, args.tokens, args.layers)
    seed = synth.seed_of(args.config)
    prefill = args.config == 4
    shape = moe.make_shape(s.H, s.F, s.E, s.k, s.Fs, s.n_shared)
    layers = [Layer(s, seed, l, device=dev) for l in range(s.L)]
    wts = [moe.ExpertWeights(L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down)
           for L in layers]
    xs = x_sets(s, seed, N_SETS, T, device=dev)                   # [S, L, T, H] bf16
    ids = torch.zeros((s.L, T, s.k), dtype=torch.int32, device=dev)
    w = torch.zeros((s.L, T, s.k), dtype=torch.float32, device=dev)
    y = torch.zeros((s.L, T, s.H), dtype=torch.float32, device=dev)
    mode = moe.PREFILL if prefill else moe.DECODE
    ws = moe.workspace(shape, T, mode, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    layer_fn = moe.iq4nl_prefill_grouped if prefill else moe.iq4nl_decode

    def step(xin):
        for l in range(s.L):
            if prefill:
                moe.route_topk(shape, layers[l].router_w, layers[l].bias, xin[l], ids[l], w[l])
                layer_fn(shape, wts[l], xin[l], ids[l], w[l], ws, y=y[l], status=status)
            else:
                moe.iq4nl_decode_routed(shape, layers[l].router_w, layers[l].bias, wts[l], xin[l],
                                        ws, ids=ids[l], weights=w[l], y=y[l], status=status)

    if prefill:
        launches_per_layer = (moe.launches_per_call(shape, T, moe.CALL_ROUTE) +
                              moe.launches_per_call(shape, T, moe.CALL_PREFILL))
    else:
        launches_per_layer = moe.launches_per_call(shape, T, moe.CALL_DECODE_ROUTED)

    # capture one graph per input set
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for i in range(N_SETS):
            step(xs[i])                                            # eager warm-up of each set
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graphs = []
    for i in range(N_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(xs[i])
        graphs.append(g)
    torch.cuda.synchronize()

    # distinct expert bytes per set (from the routes each set produces)
    ids_by_set = []
    for i in range(N_SETS):
        graphs[i].replay()
        torch.cuda.synchronize()
        ids_by_set.append(ids.cpu().numpy().copy())
    eb = s.expert_bytes()
    router_bytes = s.E * s.H * 2
    # algorithmic FLOPs per layer: 3 matrices x 2 x H x F per (token, expert)
    valid_pairs = [(a[l] >= 0).sum() for a in ids_by_set for l in range(s.L)]
    flops_layer = 2.0 * 3.0 * s.H * (float(np.mean(valid_pairs)) * s.F +
                                     (T * s.Fs if s.n_shared else 0))
    bytes_set = []
    for a in ids_by_set:
        tot = 0
        for l in range(s.L):
            u = len(np.unique(a[l]))
            tot += u * eb + (s.expert_bytes(s.Fs) if s.n_shared else 0) + router_bytes
        bytes_set.append(tot)
    bytes_per_step = float(np.mean(bytes_set))

    def barrier():
        if dist is not None:
            dist.barrier()

    for i in range(args.warmup):
        graphs[i % N_SETS].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for i in range(args.steps):
        graphs[i % N_SETS].replay()
    e1.record(cur)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    t_max = torch.tensor([ms], device=dev)
    if dist is not None:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    ms = float(t_max.item())
    st = int(status.item())

    # ---- per-call durations: one graph per kind of call over all layers (the
    # routes of input set 0 in place), replayed on the same stream
    def graph_ms(fn, reps=5):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(s.L):
                fn(l)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(reps):
            g.replay()
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * s.L)

    xin0 = xs[0]
    graphs[0].replay()
    torch.cuda.synchronize()
    layer_ms = graph_ms(lambda l: layer_fn(shape, wts[l], xin0[l], ids[l], w[l], ws, y=y[l],
                                           status=status))
    route_ms = graph_ms(lambda l: moe.route_topk(shape, layers[l].router_w, layers[l].bias,
                                                 xin0[l], ids[l], w[l]))
    layer_bytes = (bytes_set[0] - s.L * router_bytes) / s.L

    hbm, bf16, peak_kind = peaks()
    tokens = T * world
    value = tokens * 1000.0 / ms
    step_gbs = bytes_per_step / (ms * 1e-3) / 1e9
    achieved = layer_bytes / (layer_ms * 1e-3) / 1e9
    tflops = flops_layer / (layer_ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        xin = torch.empty_like(xs[0])
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            step(xin)
        host_x = [xs[i].cpu().pin_memory() for i in range(N_SETS)]
        host_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        for i in range(args.warmup):
            xin.copy_(host_x[i % N_SETS], non_blocking=True)
            g2.replay()
            host_y.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for i in range(args.steps):
            xin.copy_(host_x[i % N_SETS], non_blocking=True)
            g2.replay()
            host_y.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / args.steps
        tmx = torch.tensor([dt], device=dev)
        if dist is not None:
            dist.all_reduce(tmx, op=dist.ReduceOp.MAX)
        dt = float(tmx.item())
        e2e = {"value": tokens / dt, "unit": UNIT,
               "h2d_bytes_per_step": int(xin.numel() * xin.element_size()),
               "d2h_bytes_per_step": int(y.numel() * y.element_size())}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, desc = oracle_sample(args.config, T)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    traffic = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("iq4_nl weights x int16 activations, exact int dot, f32 accumulate"
                      if not prefill else "fp16 x fp16 -> f32 (tcgen05 kind::f16)"),
            "data": "synthetic (seeded; shapes of the pages' models)",
            "config": {"workload": s.name, "tokens_per_step": T, "layers": s.L,
                       "input_sets": N_SETS, "graph": "one CUDA graph per step, PDL between "
                       "kernels",
                       "l2": f"inputs larger than L2: {bytes_per_step / 1e9:.3f} GB of distinct "
                             "expert bytes per step vs 129 MB L2",
                       "parallelism": f"replicas x{world}"},
            "hbm_gbs": step_gbs, "hbm_frac_of_measured": step_gbs / hbm,
            "bytes_per_step": bytes_per_step,
            "roofline": ({"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                          "frac": achieved / hbm, "traffic": traffic,
                          "kernel": "moe_iq4nl_decode (the layer without routing), per call",
                          "peak_kind": peak_kind, "avg_call_ms": layer_ms,
                          "algorithmic_bytes_per_call": layer_bytes}
                         if not prefill else
                         {"bound": "tensor", "achieved": tflops, "peak": bf16, "unit": "TFLOP/s",
                          "frac": tflops / bf16, "traffic": traffic,
                          "kernel": "moe_iq4nl_prefill_grouped (bucket, gather, tcgen05 gate/up "
                                    "and down GEMMs, combine), per call",
                          "peak_kind": peak_kind + " (cuBLAS bf16 dense; kind::f16 fp16 has the "
                                       "same rate)",
                          "avg_call_ms": layer_ms, "algorithmic_flops_per_call": flops_layer}),
            "route_call_ms": route_ms,
            "step_call": "moe_iq4nl_prefill_grouped after moe_route_topk" if prefill else
                         "moe_iq4nl_decode_routed (route + layer in one call)",
            "launches_per_layer": launches_per_layer,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": args.steps * s.L * launches_per_layer,
            "status_word": st,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_libmoe(args)


if __name__ == "__main__":
    sys.exit(main())

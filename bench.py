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
    ap.add_argument("--config", type=int, default=None,
                    help="workload: 1 Xing decode (default), 2 Qwen3-Next paired decode, "
                         "3 DeepSeek-like wide decode, 4 Xing prefill chunk")
    ap.add_argument("--tokens", type=int, default=None, help="decode batch (config 3: 1/4/16)")
    ap.add_argument("--same-tokens", action="store_true",
                    help="every token of a batch is token 0 (decode: the forced-overlap "
                         "variant, each expert of the union read once for all of them)")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the other configurations' block (measured after the headline "
                         "when no --config is given)")
    ap.add_argument("--step", default="layers", choices=["routed", "layers", "chained"],
                    help="decode step: routed = one moe_iq4nl_decode_routed call per layer; "
                         "layers = one moe_iq4nl_decode_layers call for all layers (each its "
                         "own input); chained = the same with layer l+1's input bf16(y_l)")
    ap.add_argument("--impl", default="libmoe", choices=["libmoe", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="prefill workload: E4M3 operands (moe_iq4nl_prefill_grouped_fp8)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (small profiling cases)")
    ap.add_argument("--experts", type=int, default=None,
                    help="keep only N routed experts per layer, same sizes otherwise (small "
                         "profiling cases)")
    a = ap.parse_args()
    # the other configurations are measured only on a default (headline) run
    a.workloads = a.workloads and a.config is None and a.layers is None and a.experts is None \
        and a.tokens is None and not a.same_tokens and not a.fp8
    if a.config is None:
        a.config = 1
    return a


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 0.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


def workload(cfg: int, tokens, layers=None, experts=None):
    import copy
    import synth
    s = synth.SHAPES[cfg]
    if layers is not None and layers < s.L:
        s = copy.copy(s)
        s.L = int(layers)
        s.name = f"{s.name} (first {s.L} layers)"
    if experts is not None and s.k <= experts < s.E:
        s = copy.copy(s)
        s.name = f"{s.name} ({int(experts)} of its {s.E} experts)"
        s.E = int(experts)
    T = s.T if tokens is None else int(tokens)
    if cfg != 4 and T > 16:
        T = 16
    return s, T


# ---------------------------------------------------------------- replicas

def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of every rank's value (the step time of the slowest
    replica); the value itself on one process."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank (replicas:
    every rank runs its own copy of the workload)."""
    return units_per_rank * world / seconds


# ---------------------------------------------------------------- ncu traffic

# ncu figures of a kernel, kept machine-readable next to their summaries:
# profiles/<name>.json with "sources_digest", "tokens", "layers" and
# "dram_bytes_per_launch" (read + write DRAM bytes of one launch).
PROFILE_DECODE_FUSED = "decode_fused_xing_decode.json"
PROFILE_DECODE_LAYERS = "decode_layers_xing_decode.json"

_DECODE_COMMON = (
    "quantized_routed_expert_gb300/csrc/decode_common.cuh",
    "quantized_routed_expert_gb300/csrc/decode.cuh",
    "quantized_routed_expert_gb300/csrc/common.cuh",
    "quantized_routed_expert_gb300/csrc/decode.cu",
    "quantized_routed_expert_gb300/csrc/moe_api.cu",
    "quantized_routed_expert_gb300/csrc/route.cuh",
    "quantized_routed_expert_gb300/csrc/prefill.cuh",
    "quantized_routed_expert_gb300/csrc/util_kernels.cuh",
    "include/moe.h",
    "quantized_routed_expert_gb300/build.py",
)
# What each decode kernel is built and launched from: its translation unit (the
# .cu and every header it includes), the host code that chooses and launches it,
# and the compiler flags. Changing any of these voids its counters.
FUSED_DECODE_SOURCES = ("quantized_routed_expert_gb300/csrc/decode_fused.cu",) + _DECODE_COMMON
LAYERS_DECODE_SOURCES = ("quantized_routed_expert_gb300/csrc/decode_layers.cu",) + _DECODE_COMMON


def code_only(text: str) -> str:
    """C, C++ or CUDA source without its comments, whitespace runs collapsed to
    one space (string and character literals are kept as written)."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def sources_digest(files=FUSED_DECODE_SOURCES) -> str:
    """Digest of the sources a kernel is built and launched from; a profile's
    counters apply only to the sources they were taken on. C/CUDA files enter
    as their code (comments and layout do not change what is compiled); the
    build script enters whole."""
    import hashlib
    h = hashlib.sha256()
    for rel in files:
        h.update(rel.encode())
        with open(os.path.join(ROOT, rel), "rb") as f:
            data = f.read()
        if rel.endswith((".cu", ".cuh", ".h", ".cpp")):
            data = code_only(data.decode("utf-8")).encode("utf-8")
        h.update(data)
    return h.hexdigest()[:16]


def profiled_traffic(name: str, T: int, files=FUSED_DECODE_SOURCES, layers=None):
    """DRAM bytes per launch recorded in profiles/<name>, if they were taken on
    these kernel sources, this token count (and layer count, when given)."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("sources_digest") != sources_digest(files) or int(d.get("tokens", -1)) != T:
            return None
        if layers is not None and int(d.get("layers", -1)) != layers:
            return None
        return {"dram_bytes_per_launch": float(d["dram_bytes_per_launch"]),
                "source": f"profiles/{name}"}
    except (OSError, KeyError, ValueError, TypeError):
        return None


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

class OracleRun:
    """The oracle (exact fp64) on the host cores over the bench workload: the
    same seeds, layers and input sets as the GPU arm, route + layer for each
    layer. Expert blocks are generated once and kept (up to ``cache_bytes``)
    so that generation stays outside the timed calls and repeated passes."""

    def __init__(self, cfg: int, T: int, layers=None, max_tokens: int = 16, threads=None,
                 cache_bytes: float = 3e9, experts=None, fp8: bool = False):
        import oracle
        import synth
        self.mode = oracle.MMA8 if fp8 else oracle.EXACT
        self.s, _ = workload(cfg, None, layers, experts)
        self.seed = synth.seed_of(cfg)
        self.T_full = T
        self.T = min(T, max_tokens)              # a bounded sample of a prefill chunk
        self.threads = threads or (os.cpu_count() or 1)
        s = self.s
        self.cores = max(1, min(self.threads, self.T * (s.k + s.n_shared)))
        self.cache, self.cached, self.cap = {}, 0, cache_bytes
        self.routers = [synth.router(s, self.seed, l) for l in range(s.L)]
        self.shared = [synth.shared_mats(s, self.seed, l) if s.n_shared else None
                       for l in range(s.L)]

    def _expert(self, l: int, e: int):
        import synth
        k = (l, e)
        m = self.cache.get(k)
        if m is None:
            m = synth.expert_mats(self.s, self.seed, l, e)
            nb = sum(a.nbytes for a in m)
            if self.cached + nb <= self.cap:
                self.cache[k] = m
                self.cached += nb
        return m

    def one_pass(self, input_set: int, budget_s: float = float("inf")):
        """Route + layer through the layers for the sample's tokens of one input
        set; stops after the layer that crosses the budget. Returns (tokens/s
        through the whole stack, oracle seconds, layers done)."""
        import oracle
        import synth
        s = self.s
        spent, done = 0.0, 0
        for l in range(s.L):
            Wr, b = self.routers[l]
            x = synth.x_rows(self.seed, l, s.H, self.T, input_set=input_set)
            t0 = time.perf_counter()
            ids, w, _, _ = oracle.route(Wr, b, x, s.k)
            spent += time.perf_counter() - t0
            experts = {int(e): self._expert(l, int(e)) for e in np.unique(ids)}
            t0 = time.perf_counter()
            oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, s.n_shared, experts, self.shared[l], x,
                             ids, w, mode=self.mode, threads=self.threads)
            spent += time.perf_counter() - t0
            done += 1
            if spent > budget_s:
                break
        return self.T * done / s.L / spent, spent, done

    def describe(self, passes: int, layers: int, spent: float) -> str:
        import oracle
        kind = "E4M3-operand (mma8) fp64 oracle" if self.mode == oracle.MMA8 else \
            "exact fp64 oracle"
        return (f"{self.T} of {self.T_full} token(s) of the workload, {passes} pass(es) over "
                f"input sets, {layers} layer calls in all (a full pass is {self.s.L}; route + "
                f"layer, {kind}), {spent:.1f} s of oracle time; tokens/s scaled to "
                f"the full {self.s.L}-layer stack")


def oracle_baseline(cfg: int, T: int, layers=None, budget_s: float = 10.0,
                    wall_s: float = 120.0, experts=None, fp8: bool = False):
    """cpu_baseline: passes over the input sets until about budget_s seconds of
    oracle time (or wall_s of wall time, weight generation included)."""
    run = OracleRun(cfg, T, layers, experts=experts, fp8=fp8)
    t_wall = time.perf_counter()
    toks, spent, passes, calls = 0.0, 0.0, 0, 0
    while spent < budget_s and time.perf_counter() - t_wall < wall_s:
        tps, dt, done = run.one_pass(passes % N_SETS, budget_s - spent)
        toks += tps * dt
        spent += dt
        calls += done
        passes += 1
    return toks / spent, run.cores, run.describe(passes, calls, spent)


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores. Each step
    is one pass of a bounded sample of the workload (at most 16 tokens, at
    most about 3 s of oracle time) over the next input set."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    s, T = workload(args.config, args.tokens, args.layers, args.experts)
    fp8 = getattr(args, "fp8", False) and args.config == 4
    run = OracleRun(args.config, T, args.layers, experts=args.experts, fp8=fp8)
    per = []
    for i in range(args.warmup + args.steps):
        tps, dt, done = run.one_pass(i % N_SETS, budget_s=3.0)
        if i >= args.warmup:
            per.append((tps, dt, done))
    spent = float(sum(p[1] for p in per))
    value = float(sum(p[0] * p[1] for p in per) / spent)
    desc = run.describe(len(per), int(sum(p[2] for p in per)), spent)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * spent / len(per),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' models)",
        "config": {"workload": s.name, "tokens_per_step": T, "layers": s.L,
                   "sample_tokens": run.T, "input_sets": N_SETS,
                   **({"operands": "e4m3"} if fp8 else {})},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": run.cores, "kind": "oracle",
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
    ctx = (world, rank, local, dist, dev)
    line = measure(args, ctx)
    if line is not None and world == 1 and args.workloads:
        line["workloads"] = other_workloads(args, ctx)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# The other configurations, measured in the same process after the headline,
# with the same timing code (no e2e and no CPU baseline for these).
# The Qwen3-Next-shaped layer at one token and at two identical tokens is the
# Red Lite page's reuse check (section 4: a second token on the same experts
# costs about 1.06x one token when each block is decoded once for both).
OTHER_WORKLOADS = (
    {"config": 2, "tokens": None, "step": "layers", "steps": 10, "warmup": 3},
    {"config": 2, "tokens": None, "step": "chained", "steps": 10, "warmup": 3},
    {"config": 2, "tokens": 1, "step": "layers", "steps": 10, "warmup": 3},
    {"config": 2, "tokens": 2, "step": "layers", "steps": 10, "warmup": 3, "same_tokens": True},
    {"config": 3, "tokens": 1, "step": "layers", "steps": 10, "warmup": 3},
    {"config": 3, "tokens": 4, "step": "routed", "steps": 10, "warmup": 3},
    {"config": 3, "tokens": 16, "step": "routed", "steps": 10, "warmup": 3},
    {"config": 4, "tokens": None, "step": "routed", "steps": 10, "warmup": 3},
    {"config": 4, "tokens": None, "step": "routed", "steps": 10, "warmup": 3, "fp8": True},
)


def other_workloads(args, ctx):
    import copy
    import torch
    out = []
    for w in OTHER_WORKLOADS:
        a = copy.copy(args)
        a.config, a.tokens, a.step = w["config"], w["tokens"], w["step"]
        a.steps, a.warmup = w["steps"], w["warmup"]
        a.no_e2e, a.no_cpu_baseline = True, True
        a.same_tokens = bool(w.get("same_tokens", False))
        a.fp8 = bool(w.get("fp8", False))
        a.layers, a.experts = None, None
        r = measure(a, ctx)
        torch.cuda.empty_cache()
        rf = r["roofline"]
        out.append({"workload": r["config"]["workload"], "tokens_per_step": r["config"]["tokens_per_step"],
                    "same_tokens": a.same_tokens,
                    "layers": r["config"]["layers"], "step_call": r["step_call"],
                    "dtype": r["dtype"],
                    "steps": a.steps, "warmup": a.warmup,
                    "ms_per_step": r["ms_per_step"], "step_ms": r["step_ms"],
                    "value": r["value"], "unit": UNIT,
                    "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                    "kernel")},
                    "clocks": r["clocks"], "gpu_launches": r["gpu_launches"],
                    "status_word": r["status_word"]})
    # the reuse check: a step of two identical tokens against a step of one
    one = [o for o in out if "qwen3" in o["workload"] and o["tokens_per_step"] == 1]
    two = [o for o in out if "qwen3" in o["workload"] and o["same_tokens"]]
    if one and two:
        out.append({"reuse_check": "Qwen3-Next-shaped layer, 48 layers: ms per step of two "
                                   "identical tokens / ms per step of one token",
                    "ratio": two[0]["ms_per_step"] / one[0]["ms_per_step"]})
    return out


def measure(args, ctx):
    """One workload: build it, time it, return the bench line (rank 0) or None."""
    import torch
    world, rank, local, dist, dev = ctx

    import quantized_routed_expert_gb300 as moe
    import synth
    from synth.layers import Layer, x_sets

    s, T = workload(args.config, args.tokens, args.layers, args.experts)
    seed = synth.seed_of(args.config)
    prefill = args.config == 4
    fp8 = prefill and getattr(args, "fp8", False)
    shape = moe.make_shape(s.H, s.F, s.E, s.k, s.Fs, s.n_shared)
    layers = [Layer(s, seed, l, device=dev) for l in range(s.L)]
    wts = [moe.ExpertWeights(L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down)
           for L in layers]
    xs = x_sets(s, seed, N_SETS, T, device=dev)                   # [S, L, T, H] bf16
    if args.same_tokens:
        xs[:, :, 1:, :] = xs[:, :, :1, :]
    ids = torch.zeros((s.L, T, s.k), dtype=torch.int32, device=dev)
    w = torch.zeros((s.L, T, s.k), dtype=torch.float32, device=dev)
    y = torch.zeros((s.L, T, s.H), dtype=torch.float32, device=dev)
    mode = (moe.PREFILL_FP8 if fp8 else moe.PREFILL) if prefill else moe.DECODE
    ws = moe.workspace(shape, T, mode, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    layer_fn = moe.iq4nl_prefill_grouped if prefill else moe.iq4nl_decode
    if fp8:
        # each layer's row-exponent table, made once with the weights (not timed)
        rexp = {id(wts[l]): moe.fp8_row_exponents(shape, wts[l]) for l in range(s.L)}

        def layer_fn(shape_, w_, x_, ids_, wt_, ws_, y=None, status=None):
            return moe.iq4nl_prefill_grouped_fp8(shape_, w_, rexp[id(w_)], x_, ids_, wt_, ws_,
                                                 y=y, status=status)

    multi = (not prefill) and args.step in ("layers", "chained")
    chained = args.step == "chained"
    spec = [(wts[l], layers[l].router_w, layers[l].bias) for l in range(s.L)]

    def step(xin):
        if multi:
            moe.iq4nl_decode_layers(shape, spec, xin[0] if chained else xin, ws,
                                    chained=chained, ids=ids, weights=w, y=y, status=status)
            return
        for l in range(s.L):
            if prefill:
                moe.route_topk(shape, layers[l].router_w, layers[l].bias, xin[l], ids[l], w[l])
                layer_fn(shape, wts[l], xin[l], ids[l], w[l], ws, y=y[l], status=status)
            else:
                moe.iq4nl_decode_routed(shape, layers[l].router_w, layers[l].bias, wts[l], xin[l],
                                        ws, ids=ids[l], weights=w[l], y=y[l], status=status)

    if prefill:
        launches_per_layer = (moe.launches_per_call(shape, T, moe.CALL_ROUTE) +
                              moe.launches_per_call(shape, T, moe.CALL_PREFILL_FP8 if fp8
                                                    else moe.CALL_PREFILL))
    elif multi:
        launches_per_layer = moe.launches_per_call(
            shape, T, moe.call_decode_layers(s.L, chained)) / s.L
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
    # keep the GPU under the same load for about half a second before the timed
    # region (untimed replays), so the clock samples show the clocks under load
    t_load = time.perf_counter()
    i_load = 0
    while time.perf_counter() - t_load < 0.5:
        for _ in range(8):
            graphs[i_load % N_SETS].replay()
            i_load += 1
        torch.cuda.synchronize()
    # one event between consecutive steps: the first and last bracket the
    # timed region, the others give the per-step spread
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    cur = torch.cuda.current_stream()
    torch.cuda.nvtx.range_push("timed")          # lets a profiler keep to this region
    evs[0].record(cur)
    for i in range(args.steps):
        graphs[i % N_SETS].replay()
        evs[i + 1].record(cur)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(evs[0].elapsed_time(evs[-1]) / args.steps, dist, dev)
    per_step = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)])
    step_stats = {"median": float(np.median(per_step)),
                  "p10": float(np.percentile(per_step, 10)),
                  "p90": float(np.percentile(per_step, 90)), "of_rank": rank}
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
    value = whole_job_rate(T, world, ms * 1e-3)
    step_gbs = bytes_per_step / (ms * 1e-3) / 1e9
    achieved = layer_bytes / (layer_ms * 1e-3) / 1e9
    layer_call_ms = layer_ms
    tflops = flops_layer / (layer_ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        xin = torch.empty_like(xs[0])
        xuse = xin[:1] if (multi and chained) else xin     # what a step reads
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            step(xin)
        host_x = [(xs[i][:1] if (multi and chained) else xs[i]).cpu().pin_memory()
                  for i in range(N_SETS)]
        host_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        for i in range(args.warmup):
            xuse.copy_(host_x[i % N_SETS], non_blocking=True)
            g2.replay()
            host_y.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for i in range(args.steps):
            xuse.copy_(host_x[i % N_SETS], non_blocking=True)
            g2.replay()
            host_y.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        dt = max_over_ranks((time.perf_counter() - t0) / args.steps, dist, dev)
        e2e = {"value": whole_job_rate(T, world, dt), "unit": UNIT,
               "h2d_bytes_per_step": int(xuse.numel() * xuse.element_size()),
               "d2h_bytes_per_step": int(y.numel() * y.element_size())}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, desc = oracle_baseline(args.config, T, args.layers, experts=args.experts,
                                           fp8=fp8)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    # the dominant kernel: for the fused decode every launch of the step is the
    # one persistent layer kernel (route + experts + combine), so its average
    # launch duration is the timed step over its L launches; otherwise the
    # layer call timed on its own
    fused = (not prefill) and launches_per_layer == 1
    if multi and launches_per_layer * s.L == 1:
        kernel = ("decode_layers_kernel (route + experts + combine of all "
                  f"{s.L} layers, one launch per step{', chained' if chained else ''})")
        launch_ms = ms
        unit_bytes = bytes_per_step
        achieved = unit_bytes / (launch_ms * 1e-3) / 1e9
        prof = (profiled_traffic(PROFILE_DECODE_LAYERS, T, LAYERS_DECODE_SOURCES, s.L)
                if not chained else None)
    elif fused:
        kernel = "decode_fused_kernel (route + experts + combine, one launch per layer)"
        launch_ms = ms / s.L
        unit_bytes = bytes_per_step / s.L
        achieved = unit_bytes / (launch_ms * 1e-3) / 1e9
        prof = profiled_traffic(PROFILE_DECODE_FUSED, T)
    else:
        kernel = ("moe_iq4nl_prefill_grouped_fp8 (bucket, E4M3 gather, tcgen05 kind::f8f6f4 "
                  "gate/up GEMM, h to E4M3, down GEMM, combine), per call"
                  if fp8 else
                  "moe_iq4nl_prefill_grouped (bucket, gather, tcgen05 gate/up and down GEMMs, "
                  "combine), per call" if prefill else
                  "moe_iq4nl_decode (the layer without routing), per call")
        launch_ms = layer_ms
        unit_bytes = layer_bytes
        prof = None
    traffic = prof["dram_bytes_per_launch"] if prof else None
    # the 8-bit contraction's peak: the measured bf16 rate x the nominal fp8/bf16
    # ratio (4.5 / 2.25 PFLOP/s dense)
    tc_peak = 2.0 * bf16 if fp8 else bf16
    tc_kind = (peak_kind + " (cuBLAS bf16 dense x 2, the nominal E4M3/bf16 ratio)" if fp8 else
               peak_kind + " (cuBLAS bf16 dense; kind::f16 fp16 has the same rate)")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "step_ms": step_stats,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("iq4_nl weights x int16 activations, exact int dot, f32 accumulate"
                      if not prefill else
                      "e4m3 x e4m3 -> f32 (tcgen05 kind::f8f6f4)" if fp8 else
                      "fp16 x fp16 -> f32 (tcgen05 kind::f16)"),
            "data": "synthetic (seeded; shapes of the pages' models)",
            "config": {"workload": s.name, "tokens_per_step": T, "layers": s.L,
                       "input_sets": N_SETS, "graph": "one CUDA graph per step, PDL between "
                       "kernels",
                       "l2": f"inputs larger than L2: {bytes_per_step / 1e9:.3f} GB of distinct "
                             "expert bytes per step vs 129 MB L2",
                       "parallelism": f"replicas x{world}",
                       **({"same_tokens": True} if args.same_tokens else {}),
                       **({"operands": "e4m3"} if fp8 else {})},
            "hbm_gbs": step_gbs, "hbm_frac_of_measured": step_gbs / hbm,
            "bytes_per_step": bytes_per_step,
            "roofline": ({"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                          "frac": achieved / hbm, "traffic": traffic, "kernel": kernel,
                          "peak_kind": peak_kind, "avg_launch_ms": launch_ms,
                          "algorithmic_bytes_per_launch": unit_bytes,
                          "traffic_source": prof["source"] if prof else None}
                         if not prefill else
                         {"bound": "tensor", "achieved": tflops, "peak": tc_peak,
                          "unit": "TFLOP/s", "frac": tflops / tc_peak, "traffic": traffic,
                          "kernel": kernel, "peak_kind": tc_kind,
                          "avg_call_ms": layer_ms, "algorithmic_flops_per_call": flops_layer}),
            "layer_call_ms": layer_call_ms, "route_call_ms": route_ms,
            "step_call": ("moe_iq4nl_prefill_grouped_fp8 after moe_route_topk" if fp8 else
                          "moe_iq4nl_prefill_grouped after moe_route_topk") if prefill else
                         (f"moe_iq4nl_decode_layers ({'chained' if chained else 'own inputs'},"
                          " all layers in one call)" if multi else
                          "moe_iq4nl_decode_routed (route + layer in one call)"),
            "launches_per_layer": launches_per_layer,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": int(round(args.steps * s.L * launches_per_layer)),
            "status_word": st,
        }
        return line
    return None


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_libmoe(args)


if __name__ == "__main__":
    sys.exit(main())

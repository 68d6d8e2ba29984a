#!/usr/bin/env python
"""Decode benchmark of the contextually sparse decoder (Deja Vu hot path).

Workload (default): the 40-layer OPT-13B-shaped random-init stack in fp16,
d = 5120, 40 heads of 128, FFN 20480, batch 1, a 1024-position synthetic
prompt, decode positions 1024..1151 (cycled), 20 % of heads (8) and 5 % of
neurons (1024) per layer chosen by rank-1024 look-ahead predictors on a side
stream, KV repair for skipped heads.  One step = one decoded token through
all 40 layers (predict, sparse attention with append + repair, sparse MLP),
replayed as one CUDA graph.  Inputs are larger than L2: each token streams
several GB of distinct weights, so no L2 flush is needed between steps.

Prints one JSON line.  ``--impl reference`` times the float64 CPU oracle on
a bounded sample of the same workload instead.

Multi-GPU: the decode step does not shard (one sequence, one GPU); under
torchrun every rank runs an independent replica and ``value`` sums them.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("sparse decode µs/layer & tokens/s at batch 1; HBM GB/s on selected bytes "
          "vs ~8 TB/s")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="opt13b_stack_fp16")
    p.add_argument("--layers", type=int, default=None,
                   help="run only the first L layers of the workload (small profiling cases)")
    p.add_argument("--cpu-layers", type=int, default=2,
                   help="layers of the workload in the oracle's timed sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ----------------------------------------------------------------- distributed

def _dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as tdist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        tdist.init_process_group(backend=backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as tdist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[2:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def _csrc_sha256():
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "contextual_sparsity_decode_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                   glob.glob(os.path.join(csrc, "*.h")))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic():
    """DRAM bytes per entry-point call from the committed ncu capture, or {}
    when the kernel sources changed since it was taken."""
    try:
        vals = {}
        with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = (x.strip() for x in line.split("=", 1))
                    vals[k] = v
        if vals.get("csrc_sha256") != _csrc_sha256():
            return {}
        return {k: float(v) for k, v in vals.items() if k != "csrc_sha256"}
    except (OSError, ValueError):
        return {}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ----------------------------------------------------------------- workload

def _workload(name, layers=None):
    from synth import WORKLOADS
    w = WORKLOADS[name]
    if layers is not None:
        w = w.with_(layers=max(1, min(layers, w.layers)))
    return w


def _config(w):
    return {
        "workload": (f"{w.name}: {w.layers}-layer OPT-shaped random-init stack, d={w.d}, h={w.h}, "
                     f"d_h={w.d_h}, FFN {w.N}, {w.dtype}, batch 1, prompt {w.n_prompt}, decode "
                     f"positions {w.n_prompt}..{w.n_max - 1} cycled, heads {w.head_pct}% "
                     f"({w.k_heads}) / neurons {w.neuron_pct}% ({w.k_neurons}) via rank-{w.r} "
                     f"look-ahead predictors on a side stream, KV repair"),
        "batch": 1, "layers": w.layers, "d": w.d, "heads": w.h, "d_h": w.d_h, "ffn": w.N,
        "predictor_rank": w.r, "k_heads": w.k_heads, "k_neurons": w.k_neurons,
        "kv_positions": f"{w.n_prompt}..{w.n_max - 1}",
        "l2": "no flush; inputs larger than L2 (each token streams GBs of distinct weights)",
        "parallelism": "replicas (the decode step does not shard)",
    }


def _bytes_per_step(w, mean_n):
    """Algorithmic HBM bytes of one token (weights and KV actually selected,
    plus the predictors, which read all their weights)."""
    s = 2 if w.dtype in ("f16", "bf16") else 4
    d, dh, kA, kM, r = w.d, w.d_h, w.k_heads, w.k_neurons, w.r
    mlp = 2 * kM * d * s + d * s + 8 * d
    attn = kA * 4 * dh * d * s + kA * 2 * (mean_n + 1) * dh * s + 2 * kA * dh * s + d * s + 8 * d
    pred = (d * r + r * w.N + d * r + r * w.h) * s
    return {"mlp": mlp, "attn": attn, "predict": pred}


# ----------------------------------------------------------------- GPU arm

def run_ours(args, rank, world, local):
    import torch
    from contextual_sparsity_decode_gb300 import binding as dv
    from contextual_sparsity_decode_gb300.stack import SparseDecoder
    from synth import embeddings, layer_weights, residual_input

    w = _workload(args.workload, args.layers)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dv.lib()
    layers = [layer_weights(w, l, device=dev) for l in range(w.layers)]
    scale = 1.0 / math.sqrt(w.d_h)
    dec = SparseDecoder(layers, 1, w.n_max, w.k_heads, w.k_neurons, scale)
    dec.prefill([embeddings(w, w.n_prompt, f"X{l}", device=dev)[None] for l in range(w.layers)],
                w.n_prompt)
    r0 = residual_input(w, 1, "r0", device=dev)
    dec.r_stream.copy_(r0)
    dec.capture(advance=(w.n_prompt, w.n_max))
    for _ in range(max(3, args.warmup)):
        dec.replay()
    torch.cuda.synchronize()
    dec.check()

    # ---- timed region: K graph replays on the replay stream
    clocks = Clocks(dev.index)
    clocks.start()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        dec.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    t_ms = _max_over_ranks(e0.elapsed_time(e1), world)
    dec.check()
    ms_step = t_ms / args.steps
    tokens = args.steps * 1 * world
    value = tokens / (t_ms / 1e3)
    mean_n = w.n_prompt + (w.n_gen - 1) / 2.0
    per = _bytes_per_step(w, mean_n)
    step_bytes = w.layers * (per["mlp"] + per["attn"]) + (w.layers + 1 - 1) * per["predict"]

    # ---- per-kernel-family timing (events inside a graph, one family at a time)
    fam = {}
    n_rep = max(5, min(20, args.steps))
    for kind in ("mlp", "attn", "predict"):
        dec.timed = kind
        dec.t_ev = []
        dec.capture(advance=(w.n_prompt, w.n_max))
        n_ev = len(dec.t_ev)
        tot, cnt = 0.0, 0
        for _ in range(n_rep):
            dec.replay()
            torch.cuda.synchronize()
            for i in range(0, n_ev, 2):
                tot += dec.t_ev[i].elapsed_time(dec.t_ev[i + 1])
                cnt += 1
        dec.timed = None
        us = 1e3 * tot / max(cnt, 1)
        fam[kind] = {"us_per_launch": us, "bytes_per_launch": per[kind],
                     "gbs": per[kind] / (us * 1e-6) / 1e9 if us > 0 else None,
                     "launches_per_step": cnt / n_rep}
    dec.capture(advance=(w.n_prompt, w.n_max))
    peak, peak_kind = _peaks()
    dom = max(fam, key=lambda k: fam[k]["us_per_launch"] * fam[k]["launches_per_step"])
    kernel_names = {"mlp": "dv_sparse_mlp: mlp_fused_kernel (up-projection and combine in one launch)",
                    "attn": "dv_sparse_attn: attn_qkv_kernel + attn_decode_kernel + rows_combine_kernel",
                    "predict": "dv_predict: rows_dot x2 + select_kernel"}
    traffic = _traffic().get({"mlp": "dv_sparse_mlp", "attn": "dv_sparse_attn", "predict": "dv_predict"}[dom])
    roof = {"bound": "hbm", "kernel": kernel_names[dom], "achieved": fam[dom]["gbs"],
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "frac": (fam[dom]["gbs"] / peak) if fam[dom]["gbs"] else None, "traffic": traffic,
            "bytes_per_launch": fam[dom]["bytes_per_launch"]}

    # ---- end to end through the public API with host buffers
    h_in = torch.empty((1, w.d), dtype=torch.float32, pin_memory=True)
    h_out = torch.empty((1, w.d), dtype=torch.float32, pin_memory=True)
    h_in.copy_(dec.r_stream.cpu())
    torch.cuda.synchronize()
    _barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.r_stream.copy_(h_in, non_blocking=True)
        dec.replay()
        h_out.copy_(dec.r_stream, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        h_in.copy_(h_out)
    t_e2e = _max_over_ranks(time.perf_counter() - t0, world)
    dec.check()
    e2e = {"value": tokens / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": 4 * w.d,
           "d2h_bytes_per_step": 4 * w.d}

    # per layer: 2 layernorms, 3 attention kernels, 1 MLP kernel (batch 1),
    # 3 predictor kernels (layer 0 on the main stream, the look-ahead ones on
    # the side stream); one position update per token
    launches_per_step = w.layers * (2 + 3 + 1 + 3) + 1
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "accumulate": "f32", "data": "synthetic",
        "config": _config(w),
        "us_per_layer": 1e3 * ms_step / w.layers,
        "selected_bytes_per_step": step_bytes,
        "hbm_gbs_selected": step_bytes / (ms_step * 1e-3) / 1e9,
        "hbm_frac_selected": step_bytes / (ms_step * 1e-3) / 1e9 / peak,
        "kernels": fam, "roofline": roof, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_sample(args, w, layers=[{k: v for k, v in L.items()} for L in
                                                          layers[: args.cpu_layers]])
    return out


# ----------------------------------------------------------------- CPU oracle

def _oracle_setup(w, layers_dev=None, n_layers=2):
    """Float64 copies of the first n_layers of the workload plus caches with
    the prompt stored (untimed)."""
    import numpy as np
    import oracle
    from synth import embeddings, layer_weights, residual_input
    if layers_dev is None:
        layers_src = [layer_weights(w, l) for l in range(n_layers)]
    else:
        layers_src = layers_dev[:n_layers]
    layers64 = [{k: v.detach().cpu().double().numpy() for k, v in L.items()} for L in layers_src]
    caches = []
    for l in range(n_layers):
        c = oracle.KVCache.empty(w.h, w.n_max, w.d_h, w.d, w.dtype)
        c.X[: w.n_prompt] = embeddings(w, w.n_prompt, f"X{l}").double().numpy()
        oracle.kv_prefill(c, layers64[l]["Wqkv"], w.n_prompt)
        caches.append(c)
    r = residual_input(w, 1, "r0").double().numpy()[0]
    return layers64, caches, r


def cpu_sample(args, w, layers=None):
    """Time the oracle on one decoded token through ``--cpu-layers`` layers of
    the workload and scale to the full stack."""
    import oracle
    nl = max(1, min(args.cpu_layers, w.layers))
    layers64, caches, r = _oracle_setup(w, layers, nl)
    scale = 1.0 / math.sqrt(w.d_h)
    times = []
    n = w.n_prompt
    for t in range(3):
        t0 = time.perf_counter()
        r, _ = oracle.decode_stack(r, layers64, caches, n + t, scale, w.dtype, w.k_heads, w.k_neurons)
        times.append(time.perf_counter() - t0)
    per_token_full = statistics.median(times) * w.layers / nl
    return {"value": 1.0 / per_token_full, "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": (f"float64 numpy oracle, 1 decoded token through {nl} of {w.layers} layers "
                       f"at full width (median of 3 tokens), scaled by {w.layers}/{nl}; BLAS "
                       f"threads = all host cores")}


def run_reference(args, rank, world):
    import oracle
    w = _workload(args.workload, args.layers)
    nl = max(1, min(args.cpu_layers, w.layers))
    layers64, caches, r = _oracle_setup(w, None, nl)
    scale = 1.0 / math.sqrt(w.d_h)
    n = w.n_prompt
    t_total = 0.0
    for i in range(args.warmup + args.steps):
        pos = w.n_prompt + (i % w.n_gen)
        t0 = time.perf_counter()
        r, _ = oracle.decode_stack(r, layers64, caches, pos, scale, w.dtype, w.k_heads, w.k_neurons)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            t_total += dt
    per_token_full = (t_total / args.steps) * w.layers / nl
    value = 1.0 / per_token_full
    sample = (f"float64 numpy oracle, each step 1 decoded token through {nl} of {w.layers} layers "
              f"at full width, scaled by {w.layers}/{nl}")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_token_full,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = _args()
    rank, world, local = _dist()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    out = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Decode benchmark of the contextually sparse decoder (Deja Vu hot path).

Default workload: the 40-layer OPT-13B-shaped random-init stack in fp16,
d = 5120, 40 heads of 128, FFN 20480, batch 1, a 1024-position synthetic
prompt, decode positions 1024..1151 (cycled), 20 % of heads (8) and 5 % of
neurons (1024) per layer chosen by rank-1024 look-ahead predictors on a side
stream, KV repair for skipped heads.  One step = one decoded token through
all 40 layers (predict, sparse attention with append + repair, sparse MLP),
replayed as one CUDA graph.  Inputs are larger than L2: each token streams
several GB of distinct weights, so no L2 flush is needed between steps.

Prints one JSON line.  ``--workload``, ``--batch`` and ``--keep`` select
another configuration (the OPT-1.3B layer, the OPT-30B batch / sparsity
sweep, the OPT-175B slice, the fp32 MLP block); ``--sweep`` runs all of
them, one JSON line each.  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload instead.

Multi-GPU: the decode step does not shard (one sequence, one GPU); with
``--gpus N`` every rank runs an independent replica and ``value`` sums them
(started through torch.distributed.run when not already under it).
"""

from __future__ import annotations

import argparse
import ctypes
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

# Layers timed for the stacks whose full depth would only repeat the same
# per-layer work (every layer has its own weights, larger than L2).
SWEEP_LAYERS = {"opt1.3b_layer_fp16": 8, "opt30b_stack_bf16": 4}
SWEEP = ([("mlp_d768_fp32", 1, None), ("opt1.3b_layer_fp16", 1, None)] +
         [("opt30b_stack_bf16", b, k) for b in (1, 4, 16, 32) for k in (50, 25, 10, 5)] +
         [("opt30b_stack_bf16", 1, 20), ("opt175b_slice_fp16", 1, None), ("opt175b_slice_fp16", 8, None),
          ("opt13b_stack_fp16", 1, None)])


def _args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="opt13b_stack_fp16")
    p.add_argument("--batch", type=int, default=1, help="sequences decoded together")
    p.add_argument("--keep", type=int, default=None,
                   help="percent of heads and of neurons kept (default: the workload's)")
    p.add_argument("--layers", type=int, default=None,
                   help="run only the first L layers of the workload (small profiling cases)")
    p.add_argument("--sweep", action="store_true", help="every configuration, one line each")
    p.add_argument("--cpu-layers", type=int, default=2,
                   help="layers of the workload in the oracle's timed sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prefill", choices=("synthetic", "dense"), default="synthetic",
                   help="prompt state: drawn layer inputs with their K/V (fast), or the dense "
                        "causal prompt pass through every layer (timed and reported)")
    return p.parse_args(argv)


# ----------------------------------------------------------------- distributed

def _spawn_replicas(args) -> int:
    """--gpus N outside torch.distributed.run: start N ranks through it."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1", "--master-port=29517",
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


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
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------- workload

def _workload(name, layers=None, keep=None):
    from synth import WORKLOADS
    w = WORKLOADS[name]
    if layers is not None:
        w = w.with_(layers=max(1, min(layers, w.layers)))
    if keep is not None:
        w = w.with_(head_pct=keep, neuron_pct=keep)
    return w


def _config(w, B, full_layers):
    desc = (f"{w.name}: {w.layers}-layer OPT-shaped random-init stack, d={w.d}, h={w.h}, "
            f"d_h={w.d_h}, FFN {w.N}, {w.dtype}, batch {B}, prompt {w.n_prompt}, decode "
            f"positions {w.n_prompt}..{w.n_max - 1} cycled, heads {w.head_pct}% "
            f"({w.k_heads}) / neurons {w.neuron_pct}% ({w.k_neurons}) via rank-{w.r} "
            f"look-ahead predictors on a side stream, KV repair")
    if w.layers != full_layers:
        desc += f"; {w.layers} of the {full_layers} layers timed (per-layer figures are unaffected)"
    return {
        "workload": desc, "batch": B, "layers": w.layers, "d": w.d, "heads": w.h, "d_h": w.d_h,
        "ffn": w.N, "predictor_rank": w.r, "k_heads": w.k_heads, "k_neurons": w.k_neurons,
        "kv_positions": f"{w.n_prompt}..{w.n_max - 1}",
        "l2": "no flush; inputs larger than L2 (each step streams distinct weights well above L2)",
        "parallelism": "replicas (the decode step does not shard)",
    }


def _esize(dtype):
    return 2 if dtype in ("f16", "bf16") else 4


def _block_bytes(w, B, mean_n, uA, uM, sumA):
    """Algorithmic HBM bytes of one call of each entry point: the selected
    weights (the batch union uA heads / uM neurons, read once), the selected
    heads' KV rows (sumA = sum over rows of their head counts), the inputs
    and the fp32 output read and written; the predictor reads all its
    weights."""
    s = _esize(w.dtype)
    d, dh, r = w.d, w.d_h, w.r
    mlp = 2 * uM * d * s + B * d * s + B * 8 * d
    attn = (uA * 4 * dh * d * s + sumA * 2 * (mean_n + 1) * dh * s + 2 * sumA * dh * s
            + B * d * s + B * 8 * d)
    pred = (d * r + r * w.N + d * r + r * w.h) * s
    return {"mlp": mlp, "attn": attn, "predict": pred, "ln": B * (4 * d + s * d)}


# ----------------------------------------------------------------- GPU arm

KNAMES = {"mlp": "dv_sparse_mlp", "attn": "dv_sparse_attn", "predict": "dv_predict",
          "ln": "dv_layernorm"}
KERNELS = {"mlp": "mlp_fused_kernel (batch 1; else union + up + combine, or union + tcgen05 up/down)",
           "attn": "batch 1: qkv1_tc_kernel (16-bit, d_h 128; else attn_qkv_kernel) + attn_decode_kernel + "
                   "rows_combine_kernel or rows_stream_kernel; 2+ rows: repair plan + tcgen05 q/K/V + decode + "
                   "tcgen05 output projection",
           "predict": "rows_dot x2 + select_kernel (2+ rows: pred_tc_kernel x2 + select_kernel)",
           "ln": "layernorm_kernel"}


def _union_sizes(dec):
    """Mean batch-union sizes of the heads and neurons selected in the last
    step (host read, outside the timed region)."""
    import torch
    uA = uM = sumA = 0.0
    for l in range(dec.L):
        ha = [set(dec.head_idx[l][b, : int(dec.head_cnt[l][b])].tolist()) for b in range(dec.B)]
        hm = [set(dec.neur_idx[l][b, : int(dec.neur_cnt[l][b])].tolist()) for b in range(dec.B)]
        uA += len(set().union(*ha))
        uM += len(set().union(*hm))
        sumA += sum(len(x) for x in ha)
    torch.cuda.synchronize()
    return uA / dec.L, uM / dec.L, sumA / dec.L


def _families(dec, kinds, n_rep, advance, stream=None):
    """Mean isolated time of one call of each entry point: a second capture
    with timing events around every such call (the events keep the calls
    from overlapping their neighbours, so these are isolated-call times)."""
    import torch
    fam = {}
    for kind in kinds:
        dec.timed = kind
        dec.t_ev = []
        dec.capture(advance=advance)
        n_ev = len(dec.t_ev)
        tot, cnt = 0.0, 0
        for _ in range(n_rep):
            dec.replay()
            torch.cuda.synchronize()
            for i in range(0, n_ev, 2):
                tot += dec.t_ev[i].elapsed_time(dec.t_ev[i + 1])
                cnt += 1
        dec.timed = None
        fam[kind] = {"us_per_call": 1e3 * tot / max(cnt, 1), "calls_per_step": cnt / n_rep}
    dec.capture(advance=advance)
    return fam


def run_stack(args, w, B, rank, world, local, full_layers, with_e2e=True):
    import torch
    from contextual_sparsity_decode_gb300 import binding as dv
    from contextual_sparsity_decode_gb300.stack import SparseDecoder
    from synth import embeddings, layer_weights, residual_input

    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dv.lib()
    layers = [layer_weights(w, l, device=dev) for l in range(w.layers)]
    scale = 1.0 / math.sqrt(w.d_h)
    n_cache = (w.n_max + 15) // 16 * 16  # the cache holds a multiple of 16 positions
    dec = SparseDecoder(layers, B, n_cache, w.k_heads, w.k_neurons, scale)
    prefill = None
    if getattr(args, "prefill", "synthetic") == "dense":
        # the prompt through every layer with all heads and neurons, position
        # by position (the decode kernels with S = all)
        E = torch.stack([embeddings(w, w.n_prompt, f"E/{b}", device=dev).float() for b in range(B)])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dec.prefill_dense(E, w.n_prompt)
        torch.cuda.synchronize()
        dt_s = time.perf_counter() - t0
        prefill = {"kind": "dense causal prompt pass, S = all heads and neurons, one graph per position",
                   "positions": w.n_prompt, "layers": w.layers, "rows": B, "s": dt_s,
                   "positions_per_s": w.n_prompt * B / dt_s}
        del E
    else:
        dec.prefill([torch.stack([embeddings(w, w.n_prompt, f"X{l}" if B == 1 else f"X{l}/{b}", device=dev)
                                  for b in range(B)]) for l in range(w.layers)], w.n_prompt)
    dec.r_stream.copy_(residual_input(w, B, "r0", device=dev))
    out = _time_stack(args, dec, w, B, full_layers, world)
    if prefill is not None:
        out["prefill"] = prefill
    if with_e2e:
        # ---- end to end through the public API with host buffers
        h_in = torch.empty((B, w.d), dtype=torch.float32, pin_memory=True)
        h_out = torch.empty((B, w.d), dtype=torch.float32, pin_memory=True)
        h_in.copy_(dec.r_stream.cpu())
        # one graph per token: copy in, the step, copy out (SparseDecoder.capture)
        dec.capture(advance=(w.n_prompt, w.n_max), host_io=(h_in, h_out))
        for _ in range(max(3, args.warmup)):
            dec.replay()
            torch.cuda.current_stream().synchronize()
            h_in.copy_(h_out)
        torch.cuda.synchronize()
        _barrier(world)
        # at least 100 host round trips: one late wake-up of the host thread
        # then moves the mean by well under 1 %
        n_e2e = max(args.steps, 100)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            dec.replay()
            torch.cuda.current_stream().synchronize()
            h_in.copy_(h_out)
        t_e2e = _max_over_ranks(time.perf_counter() - t0, world)
        dec.check()
        dec.capture(advance=(w.n_prompt, w.n_max))
        out["e2e"] = {"value": n_e2e * B * world / t_e2e, "unit": "tokens/s", "tokens_timed": n_e2e * B * world,
                      "h2d_bytes_per_step": 4 * w.d * B, "d2h_bytes_per_step": 4 * w.d * B}
    return out, dec, layers


def run_mlp_block(args, w):
    """The fp32 MLP block (d = 768, 4d = 3072): a step is the rank-128
    neuron predictor plus the sparse MLP on the 5 % of neurons with the
    largest true pre-activation y . W^1[:, j] (chosen outside the timed
    region).  R weight replicas rotate so that the weights read per graph
    replay (R x 19 MB) are several times L2."""
    import torch
    from contextual_sparsity_decode_gb300 import binding as dv
    from synth import draw
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dv.lib()
    R, d, N, r, k = 32, w.d, w.N, w.r, w.k_neurons
    reps = []
    for i in range(R):
        W1 = draw((N, d), 0.02, w.wid, f"rep{i}/W1", w.dtype, dev)
        W2 = draw((N, d), 0.02, w.wid, f"rep{i}/W2", w.dtype, dev)
        P1 = draw((r, d), d ** -0.5, w.wid, f"rep{i}/PM1", w.dtype, dev)
        P2 = draw((N, r), r ** -0.5, w.wid, f"rep{i}/PM2", w.dtype, dev)
        y = draw((1, d), 1.0, w.wid, f"rep{i}/y", w.dtype, dev)
        S = torch.sort(torch.topk((W1 @ y[0]).double(), k).indices).values.to(torch.int32)[None]
        reps.append(dict(W1=W1, W2=W2, P1=P1, P2=P2, y=y, S=S.contiguous(),
                         cnt=torch.tensor([k], dtype=torch.int32, device=dev),
                         pidx=torch.zeros(1, k, dtype=torch.int32, device=dev),
                         pcnt=torch.zeros(1, dtype=torch.int32, device=dev),
                         out=torch.zeros(1, d, device=dev)))
    ws_p = dv.workspace(dv.dv_predict_workspace_size(1, 1, r, N))
    ws_m = dv.workspace(dv.dv_sparse_mlp_workspace_size(1, d, N, k))
    t_ev = []

    def ops(kind=None):
        for x in reps:
            if kind == "predict":
                t_ev.append(torch.cuda.Event(enable_timing=True, external=True))
                t_ev[-1].record()
            dv.dv_predict(x["y"], [dv.Predictor(x["P1"], x["P2"], x["pidx"], x["pcnt"], dv.DV_TOPK, k)], ws_p)
            if kind == "predict":
                t_ev.append(torch.cuda.Event(enable_timing=True, external=True))
                t_ev[-1].record()
            if kind == "mlp":
                t_ev.append(torch.cuda.Event(enable_timing=True, external=True))
                t_ev[-1].record()
            dv.dv_sparse_mlp(x["y"], x["W1"], x["W2"], x["S"], x["cnt"], x["out"], ws_m)
            if kind == "mlp":
                t_ev.append(torch.cuda.Event(enable_timing=True, external=True))
                t_ev[-1].record()

    def capture(kind=None):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                ops(kind)
        torch.cuda.current_stream().wait_stream(s)
        return g

    k0 = dv.dv_kernel_launches()
    g = capture()
    launches_per_graph = dv.dv_kernel_launches() - k0
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    clocks = Clocks(0)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    for ws in (ws_p, ws_m):
        assert dv.dv_check(ws)[0] == 0
    ms_step = e0.elapsed_time(e1) / (args.steps * R)
    hbm, _, peak_kind = _peaks()
    s = _esize(w.dtype)
    per = {"mlp": 2 * k * d * s + d * s + 4 * d, "predict": (d * r + r * N) * s}
    blocks = {}
    for kind in ("mlp", "predict"):
        t_ev.clear()
        gk = capture(kind)
        tot = 0.0
        for _ in range(5):
            gk.replay()
            torch.cuda.synchronize()
            tot += sum(t_ev[i].elapsed_time(t_ev[i + 1]) for i in range(0, len(t_ev), 2))
        us = 1e3 * tot / (5 * R)
        blocks[kind] = {"entry_point": KNAMES[kind], "bytes_per_call": per[kind], "calls_per_step": 1,
                        "us_per_call_isolated": us, "gbs_isolated": per[kind] / (us * 1e-6) / 1e9,
                        "frac_isolated": per[kind] / (us * 1e-6) / 1e9 / hbm}
    roof = {"bound": "hbm", "kernel": f"dv_sparse_mlp: {KERNELS['mlp']}",
            "achieved": blocks["mlp"]["gbs_isolated"], "peak": hbm, "peak_source": peak_kind, "unit": "GB/s",
            "frac": blocks["mlp"]["frac_isolated"], "traffic": None, "bytes_per_launch": per["mlp"]}
    return {
        "metric": METRIC, "value": 1e3 / ms_step, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "accumulate": "f32", "data": "synthetic",
        "config": {"workload": (f"{w.name}: one sparse MLP block, fp32, d={d}, 4d={N}, ReLU, batch 1, "
                                f"S_M = top {w.neuron_pct}% ({k}) neurons by the true pre-activation, "
                                f"plus the rank-{r} neuron predictor; {R} weight replicas rotate "
                                f"({R * 2 * N * d * s / 1e6:.0f} MB per pass, above L2)"),
                   "batch": 1, "d": d, "ffn": N, "predictor_rank": r, "k_neurons": k,
                   "l2": f"{R} weight replicas rotate (inputs larger than L2)"},
        "us_per_layer": 1e3 * ms_step, "blocks": blocks, "roofline": roof,
        "gpu_launches": launches_per_graph // R * args.steps, "clocks": clk,
    }


def run_ours(args, rank, world, local, workload=None, B=None, keep=None, layers=None):
    from synth import WORKLOADS
    name = workload or args.workload
    B = B or args.batch
    full = WORKLOADS[name].layers
    w = _workload(name, layers if layers is not None else args.layers, keep if keep is not None else args.keep)
    if name == "mlp_d768_fp32":
        return run_mlp_block(args, w), None, None
    return run_stack(args, w, B, rank, world, local, full, with_e2e=(B == 1))


def run_sweep(args):
    import gc

    import torch
    lines = []
    cur = None  # reuse one decoder (weights, prefilled caches) across keep values
    for name, B, keep in SWEEP:
        layers = SWEEP_LAYERS.get(name)
        if name == "opt30b_stack_bf16" and cur is not None and cur[0] == (name, B):
            out = _rekeep(args, cur, keep)
        else:
            cur = None
            gc.collect()
            torch.cuda.empty_cache()
            out, dec, lw = run_ours(args, 0, 1, 0, workload=name, B=B, keep=keep, layers=layers)
            if name == "opt30b_stack_bf16":
                cur = ((name, B), dec, lw, keep)
        print(json.dumps(out), flush=True)
        lines.append(out)
    return lines


def _rekeep(args, cur, keep):
    """The next OPT-30B sparsity point on the decoder of the previous one
    (same weights and prompt caches, new keep counts)."""
    from synth import WORKLOADS
    (name, B), dec, layers, _ = cur
    w = _workload(name, SWEEP_LAYERS[name], keep)
    dec.set_keep(w.k_heads, w.k_neurons)
    return _time_stack(args, dec, w, B, WORKLOADS[name].layers)


def _time_stack(args, dec, w, B, full_layers, world=1):
    """Capture one token of `dec` as a CUDA graph, time K replays, then the
    isolated calls of each entry point; returns the JSON line (no e2e)."""
    import torch

    from contextual_sparsity_decode_gb300 import binding as dv
    advance = (w.n_prompt, w.n_max)
    k0 = dv.dv_kernel_launches()
    dec.capture(advance=advance)
    launches_per_step = dv.dv_kernel_launches() - k0
    for _ in range(max(3, args.warmup)):
        dec.replay()
    torch.cuda.synchronize()
    dec.check()

    # ---- timed region: K graph replays on the replay stream
    clocks = Clocks(torch.cuda.current_device())
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
    value = args.steps * B * world / (t_ms / 1e3)
    uA, uM, sumA = _union_sizes(dec)
    per = _block_bytes(w, B, w.n_prompt + (w.n_gen - 1) / 2.0, uA, uM, sumA)
    step_bytes = w.layers * (per["mlp"] + per["attn"] + 2 * per["ln"] + per["predict"])

    # ---- per entry point: isolated-call times, then their share of the step
    fam = _families(dec, ("mlp", "attn", "predict", "ln"), max(5, min(20, args.steps)), advance)
    hbm, bf16, peak_kind = _peaks()
    chain = sum(fam[k]["us_per_call"] * fam[k]["calls_per_step"] for k in ("attn", "mlp", "ln"))
    blocks = {}
    for k in ("attn", "mlp", "predict", "ln"):
        iso = fam[k]["us_per_call"]
        e = {"entry_point": KNAMES[k], "kernels": KERNELS[k], "bytes_per_call": per[k],
             "calls_per_step": fam[k]["calls_per_step"], "us_per_call_isolated": iso,
             "gbs_isolated": per[k] / (iso * 1e-6) / 1e9 if iso > 0 else None}
        e["frac_isolated"] = e["gbs_isolated"] / hbm if e["gbs_isolated"] else None
        if k != "predict" and chain > 0:
            # the main chain (layernorms, attention, MLP) fills the step; each
            # call gets the step's time in proportion to its isolated time
            ins = iso * (1e3 * ms_step) / chain
            e["us_per_call_in_step"] = ins
            e["gbs_in_step"] = per[k] / (ins * 1e-6) / 1e9
            e["frac_in_step"] = e["gbs_in_step"] / hbm
        blocks[k] = e
    if B >= 2 and w.dtype != "f32":
        # tensor-core MLP: the union contraction's flops (both products)
        fl = 4.0 * uM * w.d * B
        t = blocks["mlp"]["us_per_call_isolated"] * 1e-6
        blocks["mlp"]["tensor_tflops_isolated"] = fl / t / 1e12
        blocks["mlp"]["tensor_frac_isolated"] = fl / t / 1e12 / bf16
    dom = max(("attn", "mlp"), key=lambda k: blocks[k]["us_per_call_isolated"] * blocks[k]["calls_per_step"])
    traffic = _traffic().get(KNAMES[dom]) if B == 1 and w.name == "opt13b_stack_fp16" else None
    roof = {"bound": "hbm", "kernel": f"{KNAMES[dom]}: {KERNELS[dom]}",
            "achieved": blocks[dom]["gbs_isolated"], "peak": hbm, "peak_source": peak_kind, "unit": "GB/s",
            "frac": blocks[dom]["frac_isolated"], "traffic": traffic,
            "bytes_per_launch": blocks[dom]["bytes_per_call"],
            "timing": "CUDA events around every call of the entry point inside the captured step "
                      "(isolated calls); in-step shares are in blocks"}
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "accumulate": "f32", "data": "synthetic",
        "config": _config(w, B, full_layers),
        "us_per_layer": 1e3 * ms_step / w.layers,
        "selected_bytes_per_step": step_bytes,
        "hbm_gbs_selected": step_bytes / (ms_step * 1e-3) / 1e9,
        "hbm_frac_selected": step_bytes / (ms_step * 1e-3) / 1e9 / hbm,
        "union": {"heads": uA, "neurons": uM, "heads_per_row_sum": sumA},
        "blocks": blocks, "roofline": roof, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }


# ----------------------------------------------------------------- CPU oracle

def _blas_threads(n):
    """Set the BLAS thread count of numpy's bundled OpenBLAS (returns the
    previous count, or None when the library offers no such call)."""
    names = [("scipy_openblas_set_num_threads64_", "scipy_openblas_get_num_threads64_"),
             ("scipy_openblas_set_num_threads", "scipy_openblas_get_num_threads"),
             ("openblas_set_num_threads64_", "openblas_get_num_threads64_"),
             ("openblas_set_num_threads", "openblas_get_num_threads")]
    try:
        paths = {line.split()[-1] for line in open("/proc/self/maps") if "openblas" in line.lower()}
    except OSError:
        return None
    for p in paths:
        try:
            L = ctypes.CDLL(p)
        except OSError:
            continue
        for set_name, get_name in names:
            if hasattr(L, set_name) and hasattr(L, get_name):
                prev = int(getattr(L, get_name)())
                getattr(L, set_name)(int(n))
                return prev
    return None


def _oracle_setup(w, layers_dev=None, n_layers=2):
    """Float64 copies of the first n_layers of the workload plus caches with
    the prompt stored (untimed)."""
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


def _oracle_tokens(w, layers64, caches, r, n_tok, start=0):
    import oracle
    scale = 1.0 / math.sqrt(w.d_h)
    times = []
    for t in range(n_tok):
        pos = w.n_prompt + ((start + t) % w.n_gen)
        t0 = time.perf_counter()
        r, _ = oracle.decode_stack(r, layers64, caches, pos, scale, w.dtype, w.k_heads, w.k_neurons)
        times.append(time.perf_counter() - t0)
    return times, r


def cpu_sample(args, w, layers=None):
    """The oracle on decoded tokens through ``--cpu-layers`` layers of the
    workload, scaled to the full stack: with every host core, then with one
    BLAS thread."""
    nl = max(1, min(args.cpu_layers, w.layers))
    layers64, caches, r = _oracle_setup(w, layers, nl)
    times, r = _oracle_tokens(w, layers64, caches, r, 3)
    per_token_full = statistics.median(times) * w.layers / nl
    out = {"value": 1.0 / per_token_full, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": (f"float64 numpy oracle, 1 decoded token through {nl} of {w.layers} layers "
                      f"at full width (median of 3 tokens), scaled by {w.layers}/{nl}; BLAS "
                      f"threads = all host cores")}
    prev = _blas_threads(1)
    if prev is not None:
        try:
            t1, r = _oracle_tokens(w, layers64, caches, r, 2, start=3)
        finally:
            _blas_threads(prev)
        out["single_thread"] = {"value": 1.0 / (statistics.median(t1) * w.layers / nl), "unit": "tokens/s",
                                "cores": 1, "sample": "the same, median of 2 tokens, one BLAS thread"}
    return out


def run_reference(args, rank, world):
    w = _workload(args.workload, args.layers, args.keep)
    nl = max(1, min(args.cpu_layers, w.layers))
    layers64, caches, r = _oracle_setup(w, None, nl)
    times, r = _oracle_tokens(w, layers64, caches, r, args.warmup + args.steps)
    t_sample = sum(times[args.warmup:]) / args.steps
    scale_to = w.layers / nl
    value = 1.0 / (t_sample * scale_to)
    sample = (f"float64 numpy oracle, each step 1 decoded token through {nl} of {w.layers} layers "
              f"at full width (ms_per_step is that measured sample); tokens/s = 1 / (sample time "
              f"x {w.layers}/{nl})")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_sample,
            "sample_layers": nl, "scaled_to_layers": w.layers, "scale_factor": scale_to,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, 1, w.layers),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = _args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(_spawn_replicas(args))
    rank, world, local = _dist()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    out, _, layers = run_ours(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "opt13b_stack_fp16":
        w = _workload(args.workload, args.layers, args.keep)
        out["cpu_baseline"] = cpu_sample(args, w, layers=[dict(L) for L in layers[: args.cpu_layers]])
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()

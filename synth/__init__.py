"""Seeded synthetic inputs for the contextually sparse decode step.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds shapes, seeds and random draws only -- none of the
method's arithmetic -- so that both sides are fed the very same bytes.

Workloads are OPT-shaped (OPT-1.3B / 13B / 30B / 175B layer widths) with
random-initialised weights; no trained checkpoint or dataset is involved.

Distributions (one per tensor family):
  * model weights W (Wqkv, Wo, W1, W2) ~ N(0, 0.02^2)
  * token embeddings y and prompt embeddings X ~ N(0, 1)
  * predictor layers P ~ N(0, 1/fan_in), which keeps the predictor's logits
    near N(0, 0.5) so that the sigmoid is far from saturation.

Every tensor is drawn in float32 from a torch generator seeded with
(base seed + workload id, tensor tag) and then rounded once (round to nearest
even) to its storage type, so the stored bytes are exactly representable in
that type.  Large tensors can be drawn directly on a CUDA device; callers that
need the same values on both sides draw once and copy.
"""

from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, Optional

import torch

BASE_SEED = 20231017

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def keep_count(percent: int, total: int) -> int:
    """Number of units kept when ``percent`` % of ``total`` are selected,
    rounded up (integer arithmetic: 5 % of 8192 -> 410, 20 % of 32 -> 7)."""
    return -((-percent * total) // 100)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload (a model width plus decode settings)."""

    name: str
    wid: int                 # workload id, added to BASE_SEED
    d: int                   # model dimension
    h: int                   # attention heads
    d_h: int                 # head dimension
    N: int                   # MLP neurons (4d)
    r: int                   # predictor rank
    dtype: str               # storage type of weights, embeddings and KV cache
    layers: int = 1
    n_prompt: int = 0        # positions already in the KV cache before decoding
    n_gen: int = 1           # decoded tokens
    batch: int = 1
    head_pct: int = 20       # percent of heads kept
    neuron_pct: int = 5      # percent of neurons kept

    @property
    def k_heads(self) -> int:
        return keep_count(self.head_pct, self.h)

    @property
    def k_neurons(self) -> int:
        return keep_count(self.neuron_pct, self.N)

    @property
    def n_max(self) -> int:
        return self.n_prompt + self.n_gen

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # single sparse MLP block, fp32, neurons = top 5 % of the true pre-activation
    "mlp_d768_fp32": Workload("mlp_d768_fp32", 1, d=768, h=12, d_h=64, N=3072,
                              r=128, dtype="f32", n_prompt=0, n_gen=1),
    # one OPT-1.3B-shaped decoder layer, KV cache of 512 prompt positions
    "opt1.3b_layer_fp16": Workload("opt1.3b_layer_fp16", 2, d=2048, h=32, d_h=64,
                                   N=8192, r=1024, dtype="f16", n_prompt=512,
                                   n_gen=1),
    # 40-layer OPT-13B-shaped stack: prompt 1024, 128 decoded tokens
    "opt13b_stack_fp16": Workload("opt13b_stack_fp16", 3, d=5120, h=40, d_h=128,
                                  N=20480, r=1024, dtype="f16", layers=40,
                                  n_prompt=1024, n_gen=128),
    # 48-layer OPT-30B-shaped stack, KV length 2048, batch / sparsity sweeps
    "opt30b_stack_bf16": Workload("opt30b_stack_bf16", 4, d=7168, h=56, d_h=128,
                                  N=28672, r=1024, dtype="bf16", layers=48,
                                  n_prompt=2047, n_gen=1),
    # OPT-175B-shaped 4-layer slice, KV length 2048, batch 1 and 8
    "opt175b_slice_fp16": Workload("opt175b_slice_fp16", 5, d=12288, h=96, d_h=128,
                                   N=49152, r=1024, dtype="f16", layers=4,
                                   n_prompt=2047, n_gen=1),
}


def _seed(wid: int, tag: str) -> int:
    return (BASE_SEED + wid) * 1_000_003 + zlib.crc32(tag.encode())


def draw(shape, std: float, wid: int, tag: str, dtype: str = "f32",
         device="cpu") -> torch.Tensor:
    """N(0, std^2) tensor of ``shape`` rounded to ``dtype``; deterministic in
    (wid, tag, device type)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(_seed(wid, tag))
    x = torch.randn(tuple(shape), generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(TORCH_DTYPES[dtype])


def layer_weights(w: Workload, layer: int = 0, device="cpu",
                  dtype: Optional[str] = None) -> Dict[str, torch.Tensor]:
    """Weights of one decoder layer in the storage layouts of the library:

    Wqkv [h][3][d_h][d]  row t of block (i, m) = column t of W_i^m (m = Q, K, V)
    Wo   [h][d_h][d]     W_i^O
    W1n  [N][d]          row j = column j of W^1 (neuron j's input weights)
    W2n  [N][d]          row j = column j of W^2 (neuron j's output weights)
    PA1t [r][d], PA2t [h][r]   head predictor, rows = columns of P1 / P2
    PM1t [r][d], PM2t [N][r]   neuron predictor
    """
    dt = dtype or w.dtype
    t = f"L{layer}/"
    s = 0.02
    return {
        "Wqkv": draw((w.h, 3, w.d_h, w.d), s, w.wid, t + "Wqkv", dt, device),
        "Wo": draw((w.h, w.d_h, w.d), s, w.wid, t + "Wo", dt, device),
        "W1n": draw((w.N, w.d), s, w.wid, t + "W1", dt, device),
        "W2n": draw((w.N, w.d), s, w.wid, t + "W2", dt, device),
        "PA1t": draw((w.r, w.d), w.d ** -0.5, w.wid, t + "PA1", dt, device),
        "PA2t": draw((w.h, w.r), w.r ** -0.5, w.wid, t + "PA2", dt, device),
        "PM1t": draw((w.r, w.d), w.d ** -0.5, w.wid, t + "PM1", dt, device),
        "PM2t": draw((w.N, w.r), w.r ** -0.5, w.wid, t + "PM2", dt, device),
    }


def embeddings(w: Workload, rows: int, tag: str, device="cpu",
               dtype: Optional[str] = None) -> torch.Tensor:
    """[rows][d] token embeddings ~ N(0, 1) in the storage type."""
    return draw((rows, w.d), 1.0, w.wid, "emb/" + tag, dtype or w.dtype, device)


def residual_input(w: Workload, batch: int, tag: str, device="cpu") -> torch.Tensor:
    """[batch][d] float32 residual-stream input of the first layer ~ N(0, 1)."""
    return draw((batch, w.d), 1.0, w.wid, "resid/" + tag, "f32", device)

"""GPU parity of the true-sparsity labeller (dv_label_neurons, dv_label_heads)
and of dv_select_scores with the float64 oracle ("用Deja Vu来提高 LLM 的推理速度"
§1 Contextual Sparsity: the heads and neurons whose outputs over the input
sequence have the largest L2 norm; §2: a threshold on that norm gives the
predictor's labels).

Norms: every element within 1e-4 relative (plus 1e-5 of the largest norm)
of the oracle's, whose K/V are rounded to the storage type as the kernels'
are; fp32 accumulation of d-term products and of T squared terms keeps the
GPU's relative error near 1e-6.  Label sets (top-k of the GPU's norms):
exact, except units whose oracle norm is within 1e-5 (relative) of the k-th
largest."""

import math

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from dvtest import check_selection, f64
from synth import draw

pytestmark = pytest.mark.gpu


def _close(got, ref, what):
    tol = 1e-4 * np.abs(ref) + 1e-5 * np.abs(ref).max()
    bad = np.flatnonzero(np.abs(got - ref) > tol)
    assert bad.size == 0, f"{what}: {bad[:5]} got {got[bad[:5]]} ref {ref[bad[:5]]}"


def _labels(norms_gpu, ref, k, what):
    dev = "cuda"
    idx = torch.zeros((1, k), dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = dv.workspace(256)
    dv.dv_select_scores(norms_gpu[None], dv.DV_TOPK, k, 0.0, idx, cnt, ws)
    assert dv.dv_check(ws) == (0, 0)
    got = idx[0, : int(cnt[0])].cpu().numpy()
    kth = np.sort(ref)[::-1][k - 1]
    check_selection(got, oracle.label(ref, "topk", k), ref, "topk", k, window=1e-5 * kth)


NEURON_CASES = [
    # name            T     d     N      dtype   k
    ("tiny_f16",       5,   64,   300,   "f16",  15),
    ("ragged_bf16",    300, 136,  1000,  "bf16", 50),
    ("opt13b_prompt",  1024, 5120, 20480, "f16", 1024),
]


@pytest.mark.parametrize("case", NEURON_CASES, ids=[c[0] for c in NEURON_CASES])
def test_neuron_norms(case):
    name, T, d, N, dtype, k = case
    dev = "cuda"
    X = draw((T, d), 1.0, 351, name + "/X", dtype)
    W1n = draw((N, d), d ** -0.5, 351, name + "/W1", dtype)
    norms = torch.full((N,), -1.0, device=dev)
    ws = dv.workspace(dv.dv_label_workspace_size(T, d, N, 0, 0))
    dv.dv_label_neurons(X.to(dev), W1n.to(dev), norms, ws)
    assert dv.dv_check(ws) == (0, 0)
    ref = oracle.neuron_norms(f64(X), W1n.float().numpy())
    _close(f64(norms), ref, name)
    _labels(norms, ref, k, name)


HEAD_CASES = [
    # name            T     d     h   d_h  dtype   scale  k
    ("tiny_f16",       7,   64,   4,  64,  "f16",  "isq", 2),
    ("ragged_bf16",    300, 512,  4,  128, "bf16", "one", 1),
    ("mid_f16",        200, 1024, 16, 64,  "f16",  "isq", 3),
    ("opt13b_prompt",  1024, 5120, 40, 128, "f16", "isq", 8),
]


@pytest.mark.parametrize("case", HEAD_CASES, ids=[c[0] for c in HEAD_CASES])
def test_head_norms(case):
    name, T, d, h, d_h, dtype, sc, k = case
    dev = "cuda"
    scale = 1.0 / math.sqrt(d_h) if sc == "isq" else 1.0
    X = draw((T, d), 1.0, 352, name + "/X", dtype)
    Wqkv = draw((h, 3, d_h, d), d ** -0.5, 352, name + "/Wqkv", dtype)
    norms = torch.full((h,), -1.0, device=dev)
    ws = dv.workspace(dv.dv_label_workspace_size(T, d, 0, h, d_h))
    dv.dv_label_heads(X.to(dev), Wqkv.to(dev), scale, norms, ws)
    assert dv.dv_check(ws) == (0, 0)
    ref = oracle.head_norms(f64(X), Wqkv.float().numpy(), scale, dtype)
    _close(f64(norms), ref, name)
    _labels(norms, ref, k, name)


@pytest.mark.parametrize("N", [5000, 20000, 20001])
def test_select_scores_topk_threshold_and_ties(N):
    """Rows of non-negative scores with repeated values: top-k (ties to the
    lower index) and threshold lists equal the oracle's exactly.  With few
    distinct values the cut's bin holds hundreds of keys, so the selection
    refines to one key value and takes the lowest indices equal to it."""
    dev = "cuda"
    g = torch.Generator().manual_seed(5)
    S_many = torch.randint(0, 700, (3, N), generator=g).float() / 64.0  # many ties
    S_few = torch.randint(0, 16, (3, N), generator=g).float() / 8.0     # hundreds of keys per value
    ws = dv.workspace(256)
    for S, mode, k, t in ((S_many, dv.DV_TOPK, 400, 0.0), (S_many, dv.DV_TOPK, 1, 0.0),
                          (S_many, dv.DV_TOPK, N - 1, 0.0), (S_many, dv.DV_TOPK, 4000, 0.0),
                          (S_many, dv.DV_THRESHOLD, 0, 9.5), (S_few, dv.DV_TOPK, 777, 0.0),
                          (S_few, dv.DV_TOPK, N // 2, 0.0), (S_few, dv.DV_THRESHOLD, 0, 1.0)):
        cap = N
        idx = torch.full((3, cap), -1, dtype=torch.int32, device=dev)
        cnt = torch.zeros(3, dtype=torch.int32, device=dev)
        dv.dv_select_scores(S.to(dev), mode, k, t, idx, cnt, ws)
        assert dv.dv_check(ws) == (0, 0)
        for b in range(3):
            got = idx[b, : int(cnt[b])].cpu().numpy().tolist()
            s64 = S[b].double().numpy()
            ref = oracle.select_topk(s64, k) if mode == dv.DV_TOPK else oracle.select_threshold(s64, t)
            assert got == ref.tolist(), (mode, b)


def test_label_rejects_fp32_and_bad_shapes():
    dev = "cuda"
    X = torch.zeros((4, 64), dtype=torch.float32, device=dev)
    W = torch.zeros((8, 64), dtype=torch.float32, device=dev)
    norms = torch.zeros(8, device=dev)
    ws = dv.workspace(dv.dv_label_workspace_size(4, 64, 8, 2, 64))
    with pytest.raises(dv.DvError) as e:
        dv.dv_label_neurons(X, W, norms, ws)
    assert e.value.status == 2
    Wq = torch.zeros((2, 3, 96, 64), dtype=torch.float16, device=dev)
    with pytest.raises(dv.DvError) as e:
        dv.dv_label_heads(X.half(), Wq, 1.0, norms, ws)
    assert e.value.status == 7

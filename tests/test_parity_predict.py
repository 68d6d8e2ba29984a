"""GPU parity of dv_predict / dv_lookahead with the float64 oracle.

Scores: within 1e-5 of the oracle's sigmoid.  Index lists: exact except units
whose oracle score is within 1e-5 of the boundary.  The selection step alone
is also checked bit-exactly: the oracle's selection applied to the kernel's
own fp32 scores must reproduce the kernel's list.
"""

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from dvtest import TORCH, ascending_unique, check_selection, f64, topk_list_is_valid
from synth import draw

pytestmark = pytest.mark.gpu

#        name                    B   d      r     N      dtype   mode        k     t
CASES = [
    ("tiny_heads_f16",           1, 64,    32,   40,    "f16",  "topk",     8,    0.5),
    ("ragged_f16",               2, 136,   40,   1000,  "f16",  "topk",     77,   0.5),
    ("mlp768_f32",               1, 768,   128,  3072,  "f32",  "topk",     154,  0.5),
    ("opt1.3b_heads_f16",        1, 2048,  1024, 32,    "f16",  "topk",     7,    0.5),
    ("opt1.3b_neurons_f16",      1, 2048,  1024, 8192,  "f16",  "topk",     410,  0.5),
    ("opt13b_neurons_f16",       1, 5120,  1024, 20480, "f16",  "topk",     1024, 0.5),
    ("opt30b_neurons_bf16",      1, 7168,  1024, 28672, "bf16", "topk",     1434, 0.5),
    ("opt175b_neurons_f16",      1, 12288, 1024, 49152, "f16",  "topk",     2458, 0.5),
    ("threshold_bf16_b3",        3, 512,   256,  4096,  "bf16", "threshold", 0,   0.5),
    ("threshold_t07_f16",        1, 1024,  256,  2000,  "f16",  "threshold", 0,   0.7),
    ("k0_f16",                   1, 256,   64,   500,   "f16",  "topk",     0,    0.5),
    ("kN_f16",                   1, 256,   64,   500,   "f16",  "topk",     500,  0.5),
    ("batch8_f16",               8, 1024,  256,  4096,  "f16",  "topk",     205,  0.5),
    ("batch32_bf16",             32, 1024, 256,  4096,  "bf16", "topk",     205,  0.5),
    # tensor-core predictor (2..32 rows): ragged rows, r and d off the tiles
    ("batch13_ragged_f16",       13, 1032, 200,  3000,  "f16",  "topk",     150,  0.5),
    ("batch16_threshold_bf16",   16, 2048, 1024, 8192,  "bf16", "threshold", 0,   0.5),
    ("opt13b_neurons_b32_f16",   32, 5120, 1024, 20480, "f16",  "topk",     1024, 0.5),
    ("opt30b_neurons_b24_bf16",  24, 7168, 1024, 28672, "bf16", "topk",     1434, 0.5),
]


def _inputs(name, B, d, r, N, dtype, wid=101):
    y = draw((B, d), 1.0, wid, name + "/y", dtype)
    P1t = draw((r, d), d ** -0.5, wid, name + "/P1", dtype)
    P2t = draw((N, r), r ** -0.5, wid, name + "/P2", dtype)
    return y, P1t, P2t


def _run(y, preds_spec, dtype):
    """preds_spec: list of (P1t, P2t, mode, k, t, cap); returns per predictor
    (idx [B][cap], count [B], scores [B][N]) on the host."""
    B = y.shape[0]
    dev = "cuda"
    preds, outs = [], []
    for P1t, P2t, mode, k, t, cap in preds_spec:
        N = P2t.shape[0]
        idx = torch.full((B, cap), -7, dtype=torch.int32, device=dev)
        cnt = torch.full((B,), -1, dtype=torch.int32, device=dev)
        sc = torch.zeros((B, N), dtype=torch.float32, device=dev)
        preds.append(dv.Predictor(P1t.to(dev), P2t.to(dev), idx, cnt,
                                  dv.DV_TOPK if mode == "topk" else dv.DV_THRESHOLD, k, t, sc))
        outs.append((idx, cnt, sc))
    r_max = max(p.P1t.shape[0] for p in preds)
    N_max = max(p.P2t.shape[0] for p in preds)
    ws = dv.workspace(dv.dv_predict_workspace_size(B, len(preds), r_max, N_max))
    dv.dv_predict(y.to(dev), preds, ws)
    st, info = dv.dv_check(ws)
    assert st == 0, (st, info)
    return [(i.cpu().numpy(), c.cpu().numpy(), s.cpu().double().numpy()) for i, c, s in outs]


def _compare(y, P1t, P2t, mode, k, t, got):
    idx, cnt, s_gpu = got
    lists, s_ref, _ = oracle.predict(f64(y), f64(P1t), f64(P2t), mode, k=k, t=t)
    assert np.max(np.abs(s_gpu - s_ref)) <= 1e-5
    flips = 0
    for b in range(y.shape[0]):
        n = int(cnt[b])
        g = idx[b, :n]
        assert ascending_unique(g)
        flips += check_selection(g, lists[b], s_ref[b], mode, k, t)
        # the kernel's decision on its own fp32 scores is exact: a valid top-k
        # (with the index tie rule) or exactly the units above t
        if mode == "topk":
            assert topk_list_is_valid(g, s_gpu[b], k)
        else:
            assert g.tolist() == np.flatnonzero(s_gpu[b] > np.float32(t)).tolist()
    return flips


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_predict_parity(case):
    name, B, d, r, N, dtype, mode, k, t = case
    y, P1t, P2t = _inputs(name, B, d, r, N, dtype)
    cap = N if mode == "threshold" else max(k, 1)
    got = _run(y, [(P1t, P2t, mode, k, t, cap)], dtype)[0]
    _compare(y, P1t, P2t, mode, k, t, got)


def test_predict_two_predictors_fused():
    """Head and neuron predictors of one layer in one call."""
    B, d, r = 2, 2048, 1024
    y = draw((B, d), 1.0, 102, "y", "f16")
    PA1 = draw((r, d), d ** -0.5, 102, "PA1", "f16")
    PA2 = draw((32, r), r ** -0.5, 102, "PA2", "f16")
    PM1 = draw((r, d), d ** -0.5, 102, "PM1", "f16")
    PM2 = draw((8192, r), r ** -0.5, 102, "PM2", "f16")
    got = _run(y, [(PA1, PA2, "topk", 7, 0.5, 7), (PM1, PM2, "topk", 410, 0.5, 410)], "f16")
    _compare(y, PA1, PA2, "topk", 7, 0.5, got[0])
    _compare(y, PM1, PM2, "topk", 410, 0.5, got[1])


def test_predict_two_predictors_fused_batched():
    """Head and neuron predictors of one layer in one call for 20 rows (the
    tensor-core path: one launch per product holds both predictors' tiles)."""
    B, d = 20, 5120
    y = draw((B, d), 1.0, 103, "y", "f16")
    PA1 = draw((512, d), d ** -0.5, 103, "PA1", "f16")
    PA2 = draw((40, 512), 512 ** -0.5, 103, "PA2", "f16")
    PM1 = draw((1024, d), d ** -0.5, 103, "PM1", "f16")
    PM2 = draw((20480, 1024), 1024 ** -0.5, 103, "PM2", "f16")
    got = _run(y, [(PA1, PA2, "topk", 8, 0.5, 8), (PM1, PM2, "threshold", 0, 0.5, 20480)], "f16")
    _compare(y, PA1, PA2, "topk", 8, 0.5, got[0])
    _compare(y, PM1, PM2, "threshold", 0, 0.5, got[1])


def test_threshold_capacity_truncates_and_reports():
    y, P1t, P2t = _inputs("cap", 1, 256, 64, 2000, "f16")
    dev = "cuda"
    idx = torch.zeros((1, 50), dtype=torch.int32, device=dev)
    cnt = torch.zeros((1,), dtype=torch.int32, device=dev)
    sc = torch.zeros((1, 2000), dtype=torch.float32, device=dev)
    p = dv.Predictor(P1t.to(dev), P2t.to(dev), idx, cnt, dv.DV_THRESHOLD, 0, 0.5, sc)
    ws = dv.workspace(dv.dv_predict_workspace_size(1, 1, 64, 2000))
    dv.dv_predict(y.to(dev), [p], ws)
    st, info = dv.dv_check(ws)
    s = sc.cpu().double().numpy()[0]
    full = np.flatnonzero(s > 0.5)
    assert st == 8 and info == len(full)  # DV_ERR_CAPACITY, with the full count
    assert int(cnt.item()) == 50
    assert idx.cpu().numpy()[0].tolist() == full[:50].tolist()
    assert dv.dv_check(ws)[0] == 0  # the error word was cleared


def test_lookahead_on_side_stream_matches_predict():
    B, d, r, N = 1, 1024, 256, 4096
    y, P1t, P2t = _inputs("la", B, d, r, N, "f16")
    dev = "cuda"
    y = y.to(dev)
    ref = _run(y, [(P1t, P2t, "topk", 205, 0.5, 205)], "f16")[0]
    idx = torch.zeros((B, 205), dtype=torch.int32, device=dev)
    cnt = torch.zeros((B,), dtype=torch.int32, device=dev)
    p = dv.Predictor(P1t.to(dev), P2t.to(dev), idx, cnt, dv.DV_TOPK, 205)
    ws = dv.workspace(dv.dv_predict_workspace_size(B, 1, r, N))
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    ready, done = dv.make_event(main), dv.make_event(main)
    y2 = torch.empty_like(y)
    y2.copy_(y)                      # produced on the main stream
    ready.record(main)
    dv.dv_lookahead(y2, [p], ws, ready, side, done)
    main.wait_event(done)
    out = idx.clone()                # consumed on the main stream after the event
    torch.cuda.synchronize()
    assert out.cpu().numpy()[0].tolist() == ref[0][0].tolist()
    assert int(cnt.item()) == 205


#        name          N     distinct  scale  k
TIES = [
    ("dup3",          2100, 700,      1.0,   150),   # ties inside the cut's bin (direct ranking)
    ("dup512",        4096, 8,        1.0,   1000),  # 512 equal keys per value (refinement path)
    ("constant",      1000, 1,        0.0,   300),   # every score exactly 0.5
    ("saturated",     4096, 4096,     300.0, 100),   # hundreds of scores exactly 1.0f
]


@pytest.mark.parametrize("case", TIES, ids=[c[0] for c in TIES])
def test_topk_ties_resolved_by_index(case):
    """Duplicated P2 rows give bit-identical scores (every row is reduced in
    the same order), so the list must take equal scores lowest index first,
    through both the direct ranking of the cut's bin and the refinement."""
    name, N, distinct, scale, k = case
    d, r = 512, 128
    y = draw((1, d), 1.0, 107, name + "/y", "f16")
    P1t = draw((r, d), d ** -0.5, 107, name + "/P1", "f16")
    base = draw((distinct, r), r ** -0.5, 107, name + "/P2", "f32") * scale
    P2t = base.repeat((N + distinct - 1) // distinct, 1)[:N]
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(7))
    P2t = P2t[perm].to(torch.float16)
    idx, cnt, s = _run(y, [(P1t, P2t, "topk", k, 0.5, k)], "f16")[0]
    g = idx[0, : int(cnt[0])]
    assert int(cnt[0]) == k
    assert topk_list_is_valid(g, s[0], k)
    if name == "constant":
        assert g.tolist() == list(range(k))
    if name == "saturated":
        assert int(np.sum(s[0] == 1.0)) > 2 * k   # the cut lies among exact ties

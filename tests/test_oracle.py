"""Pins of the float64 oracle to facts that do not come from the oracle itself:
hand-derived worked examples (tests/golden), closed forms, special cases that
reduce to textbook library routines (torch float64 attention / linear / layer
norm), invariants of the formulas, and brute force on tiny inputs.

The ``check_*`` functions read the oracle through ``oracle.core``'s module
attributes, so the planted-mistake tests at the end can swap one step of the
oracle for a plausible wrong version and show that some pin fails.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.core as core

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _t(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.float64)


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------

def _round_sig_bits(x, bits):
    """Independent RNE to ``bits`` significant bits through scaling by the
    binade: x / 2^(floor(log2|x|) - bits + 1) rounded half-to-even."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    e = np.floor(np.log2(np.abs(x[nz])))
    scale = np.exp2(e - bits + 1)
    out[nz] = np.round(x[nz] / scale) * scale   # np.round: half to even
    return out


def check_round_to():
    xs = RNG(1).standard_normal(20000) * np.exp2(RNG(2).integers(-8, 8, 20000))
    xs = xs[np.abs(xs) >= 2.0 ** -14]            # inside f16's normal range
    assert np.array_equal(core.round_to(xs, "f16"), _round_sig_bits(xs, 11))
    assert np.array_equal(core.round_to(xs, "bf16"), _round_sig_bits(xs, 8))
    # ties to even, at 1: f16 spacing 2^-10, bf16 spacing 2^-7
    assert core.round_to(1 + 2.0 ** -11, "f16") == 1.0
    assert core.round_to(1 + 3 * 2.0 ** -11, "f16") == 1 + 2.0 ** -9
    assert core.round_to(1 + 2.0 ** -8, "bf16") == 1.0
    assert core.round_to(1 + 3 * 2.0 ** -8, "bf16") == 1 + 2.0 ** -6
    # bf16 of float32-representable values agrees with torch's own cast
    x32 = torch.randn(5000, dtype=torch.float32, generator=torch.Generator().manual_seed(3))
    ref = x32.to(torch.bfloat16).double().numpy()
    assert np.array_equal(core.round_to(x32.double().numpy(), "bf16"), ref)


def test_round_to():
    check_round_to()


# ---------------------------------------------------------------------------
# predictor
# ---------------------------------------------------------------------------

def check_predictor_golden():
    g = _golden("predictor_four_units.json")
    y, P1t, P2t = (np.array(g[k], float) for k in ("y", "P1t", "P2t"))
    z = core.predictor_logits(core.predictor_hidden(y, P1t), P2t)[0]
    assert np.array_equal(z, np.array(g["z"], float))
    for c in g["topk"]:
        S, _, _ = core.predict(y, P1t, P2t, "topk", k=c["k"])
        assert S[0].tolist() == c["S"], c
    for c in g["threshold"]:
        S, _, _ = core.predict(y, P1t, P2t, "threshold", t=c["t"])
        assert S[0].tolist() == c["S"], c


def check_predictor_loops():
    """Explicit loops over the two-layer predictor on a tiny shape."""
    rng = RNG(5)
    d, r, N = 5, 4, 6
    y, P1t, P2t = rng.standard_normal(d), rng.standard_normal((r, d)), rng.standard_normal((N, r))
    h = [max(0.0, sum(y[i] * P1t[j, i] for i in range(d))) for j in range(r)]
    z = [sum(h[j] * P2t[k, j] for j in range(r)) for k in range(N)]
    s = [1.0 / (1.0 + math.exp(-zk)) for zk in z]
    _, s_o, z_o = core.predict(y, P1t, P2t, "topk", k=2)
    assert np.allclose(z_o[0], z, rtol=1e-14, atol=1e-14)
    assert np.allclose(s_o[0], s, rtol=1e-14, atol=1e-14)


def check_topk_brute_force():
    """Top-k = the k-subset with the largest total score (distinct scores),
    for every k on tiny inputs; equal scores -> the first k indices."""
    rng = RNG(7)
    for N in (1, 5, 8):
        s = rng.random(N)
        for k in range(N + 1):
            best = max(itertools.combinations(range(N), k), key=lambda c: s[list(c)].sum())
            assert core.select_topk(s, k).tolist() == sorted(best)
    flat = np.full(9, 0.5)
    for k in range(10):
        assert core.select_topk(flat, k).tolist() == list(range(k))


def check_threshold_is_sign_of_logit():
    rng = RNG(8)
    z = rng.standard_normal(4000)
    z = z[np.abs(z) > 1e-9]
    s = core.sigmoid(z)
    assert np.array_equal(core.select_threshold(s, 0.5), np.flatnonzero(z > 0))


def check_predictor_special_cases():
    rng = RNG(9)
    d, r, N = 6, 6, 10
    y = rng.standard_normal(d)
    # P1 = identity -> h = ReLU(y)
    assert np.array_equal(core.predictor_hidden(y, np.eye(r)), np.maximum(0, y)[None])
    P1t = rng.standard_normal((r, d))
    # P2 = 0 -> every score is exactly 1/2: top-k is the first k units and a
    # strict threshold at 1/2 selects nothing
    Sk, s, _ = core.predict(y, P1t, np.zeros((N, r)), "topk", k=4)
    assert np.all(s == 0.5) and Sk[0].tolist() == [0, 1, 2, 3]
    St, _, _ = core.predict(y, P1t, np.zeros((N, r)), "threshold", t=0.5)
    assert St[0].size == 0
    P2t = rng.standard_normal((N, r))
    assert core.predict(y, P1t, P2t, "topk", k=N)[0][0].tolist() == list(range(N))
    assert core.predict(y, P1t, P2t, "topk", k=0)[0][0].size == 0


def test_predictor_golden():
    check_predictor_golden()


def test_predictor_loops():
    check_predictor_loops()


def test_topk_brute_force():
    check_topk_brute_force()


def test_threshold_sign():
    check_threshold_is_sign_of_logit()


def test_predictor_special_cases():
    check_predictor_special_cases()


def test_predict_batched_rows_independent():
    rng = RNG(10)
    Y = rng.standard_normal((3, 8))
    P1t, P2t = rng.standard_normal((5, 8)), rng.standard_normal((12, 5))
    Sb, sb, _ = core.predict(Y, P1t, P2t, "topk", k=4)
    for b in range(3):
        S1, s1, _ = core.predict(Y[b], P1t, P2t, "topk", k=4)
        assert Sb[b].tolist() == S1[0].tolist()
        assert np.allclose(sb[b], s1[0], rtol=1e-13, atol=0)


# ---------------------------------------------------------------------------
# sparsified MLP
# ---------------------------------------------------------------------------

def _mlp_case(seed, d=16, N=40):
    rng = RNG(seed)
    return rng.standard_normal(d), rng.standard_normal((N, d)), rng.standard_normal((N, d))


def check_mlp_golden():
    g = _golden("mlp_three_neurons.json")
    y, W1n, W2n = (np.array(g[k], float) for k in ("y", "W1n", "W2n"))
    for c in g["cases"]:
        assert np.array_equal(core.sparse_mlp(y, W1n, W2n, c["S"]), np.array(c["out"], float)), c


def check_mlp_all_equals_textbook_dense():
    """S_M = all neurons: the textbook dense MLP ReLU(y W1) W2^T (torch)."""
    y, W1n, W2n = _mlp_case(11)
    ref = F.linear(F.relu(F.linear(_t(y), _t(W1n))), _t(W2n).T).numpy()
    out = core.sparse_mlp(y, W1n, W2n, np.arange(W1n.shape[0]))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def check_mlp_equals_zeroed_dense():
    """Sparse over S equals the dense MLP with W^1 (resp. W^2) columns outside S
    set to zero (torch, dense)."""
    y, W1n, W2n = _mlp_case(12)
    S = np.sort(RNG(13).choice(W1n.shape[0], 9, replace=False))
    keep = torch.zeros(W1n.shape[0], dtype=torch.bool)
    keep[torch.as_tensor(S)] = True
    W1z = torch.where(keep[:, None], _t(W1n), 0.0)
    W2z = torch.where(keep[:, None], _t(W2n), 0.0)
    ref1 = F.linear(F.relu(F.linear(_t(y), W1z)), _t(W2n).T).numpy()
    ref2 = F.linear(F.relu(F.linear(_t(y), _t(W1n))), W2z.T).numpy()
    out = core.sparse_mlp(y, W1n, W2n, S)
    assert np.allclose(out, ref1, rtol=1e-12, atol=1e-12)
    assert np.allclose(out, ref2, rtol=1e-12, atol=1e-12)


def check_mlp_additive():
    y, W1n, W2n = _mlp_case(14)
    perm = RNG(15).permutation(W1n.shape[0])
    S1, S2 = np.sort(perm[:11]), np.sort(perm[11:25])
    both = core.sparse_mlp(y, W1n, W2n, np.sort(np.r_[S1, S2]))
    parts = core.sparse_mlp(y, W1n, W2n, S1) + core.sparse_mlp(y, W1n, W2n, S2)
    assert np.allclose(both, parts, rtol=1e-12, atol=1e-12)


def check_mlp_one_hot_closed_form():
    """y = e_i, S = {j}: pre-activation is W^1[i, j], out = ReLU(W^1[i, j]) W^2[:, j]."""
    _, W1n, W2n = _mlp_case(16)
    d = W1n.shape[1]
    for i, j in [(0, 0), (3, 7), (d - 1, 39)]:
        y = np.zeros(d)
        y[i] = 1.0
        ref = max(0.0, W1n[j, i]) * W2n[j]
        assert np.array_equal(core.sparse_mlp(y, W1n, W2n, [j]), ref)


def check_mlp_loops():
    y, W1n, W2n = _mlp_case(17, d=4, N=6)
    S = [1, 4, 5]
    ref = [0.0] * 4
    for j in S:
        u = sum(y[c] * W1n[j, c] for c in range(4))
        a = u if u > 0 else 0.0
        for c in range(4):
            ref[c] += a * W2n[j, c]
    assert np.allclose(core.sparse_mlp(y, W1n, W2n, S), ref, rtol=1e-14, atol=1e-14)


def test_mlp_golden():
    check_mlp_golden()


def test_mlp_all_equals_textbook_dense():
    check_mlp_all_equals_textbook_dense()


def test_mlp_equals_zeroed_dense():
    check_mlp_equals_zeroed_dense()


def test_mlp_additive():
    check_mlp_additive()


def test_mlp_one_hot():
    check_mlp_one_hot_closed_form()


def test_mlp_loops():
    check_mlp_loops()


def test_mlp_empty_and_batched():
    y, W1n, W2n = _mlp_case(18)
    assert np.array_equal(core.sparse_mlp(y, W1n, W2n, []), np.zeros(16))
    Y = RNG(19).standard_normal((3, 16))
    S = [np.array([1, 5]), np.array([], int), np.arange(40)]
    out = core.sparse_mlp_batched(Y, W1n, W2n, S)
    for b in range(3):
        assert np.array_equal(out[b], core.sparse_mlp(Y[b], W1n, W2n, S[b]))


def test_dense_mlp_zeroed_helper():
    y, W1n, W2n = _mlp_case(20)
    S = [0, 3, 9]
    assert np.allclose(core.dense_mlp_zeroed(y, W1n, W2n, S),
                       core.sparse_mlp(y, W1n, W2n, S), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# sparsified attention + KV repair
# ---------------------------------------------------------------------------

def _attn_case(seed, d=12, h=4, d_h=3, n=6, dtype="f64"):
    rng = RNG(seed)
    Wqkv = rng.standard_normal((h, 3, d_h, d)) * 0.4
    Wo = rng.standard_normal((h, d_h, d))
    X = rng.standard_normal((n + 1, d))
    return Wqkv, Wo, X


def _dense_prefill(Wqkv, X, n, dtype):
    """Cache with positions 0..n-1 stored for all heads (a dense prompt)."""
    h, _, d_h, d = Wqkv.shape
    cache = core.KVCache.empty(h, n + 1, d_h, d, dtype)
    for j in range(n):
        core.kv_append(cache, X[j], Wqkv, j, range(h))
    return cache


def _textbook_mha(Wqkv, Wo, X, n, c):
    """Dense MHA of token n over positions 0..n in the concat form:
    concat_i softmax(c q_i K_i^T) V_i, times the stacked W^O (torch SDPA)."""
    h, _, d_h, d = Wqkv.shape
    Xt = _t(X[:n + 1])
    Q = torch.stack([Xt[n:n + 1] @ _t(Wqkv[i, 0]).T for i in range(h)])[None]
    K = torch.stack([Xt @ _t(Wqkv[i, 1]).T for i in range(h)])[None]
    V = torch.stack([Xt @ _t(Wqkv[i, 2]).T for i in range(h)])[None]
    A = F.scaled_dot_product_attention(Q, K, V, scale=c)[0]          # [h][1][d_h]
    return (A.permute(1, 0, 2).reshape(1, h * d_h) @ _t(Wo).reshape(h * d_h, d))[0].numpy()


def check_attn_golden():
    g = _golden("attn_two_heads_repair.json")
    Wqkv, Wo = np.array(g["Wqkv"], float), np.array(g["Wo"], float)
    cache = core.KVCache.empty(g["h"], 2, g["d_h"], g["d"], "f64")
    for st in g["steps"]:
        before = cache.valid.copy()
        out = core.sparse_attn(np.array(st["y"]), Wqkv, Wo, cache, st["pos"], st["S_A"], g["scale"])
        assert np.allclose(out, st["out"], rtol=1e-14, atol=1e-14), (out, st)
        missing = sum(1 for i in st["S_A"] for j in range(st["pos"]) if not before[i, j])
        assert missing == st["repaired"]


def check_attn_all_equals_textbook_dense():
    for c in (1.0, 1 / math.sqrt(3)):
        Wqkv, Wo, X = _attn_case(21)
        n = X.shape[0] - 1
        cache = _dense_prefill(Wqkv, X, n, "f64")
        out = core.sparse_attn(X[n], Wqkv, Wo, cache, n, range(Wqkv.shape[0]), c)
        assert np.allclose(out, _textbook_mha(Wqkv, Wo, X, n, c), rtol=1e-12, atol=1e-12)


def check_attn_equals_zeroed_wo():
    """Sparse over S_A equals the dense MHA with W_i^O = 0 outside S_A."""
    Wqkv, Wo, X = _attn_case(22)
    n = X.shape[0] - 1
    S_A = [0, 2]
    Woz = Wo.copy()
    Woz[[1, 3]] = 0.0
    cache = _dense_prefill(Wqkv, X, n, "f64")
    out = core.sparse_attn(X[n], Wqkv, Wo, cache, n, S_A, 0.5)
    assert np.allclose(out, _textbook_mha(Wqkv, Woz, X, n, 0.5), rtol=1e-12, atol=1e-12)


def check_attn_additive():
    Wqkv, Wo, X = _attn_case(23)
    n = X.shape[0] - 1
    base = _dense_prefill(Wqkv, X, n, "f64")
    a = core.sparse_attn(X[n], Wqkv, Wo, base.copy(), n, [0, 3], 1.0)
    b = core.sparse_attn(X[n], Wqkv, Wo, base.copy(), n, [1], 1.0)
    ab = core.sparse_attn(X[n], Wqkv, Wo, base.copy(), n, [0, 1, 3], 1.0)
    assert np.allclose(ab, a + b, rtol=1e-12, atol=1e-12)


def check_attn_first_position_closed_form():
    """n = 0: the softmax has one term, so H_i = y W_i^V and
    out = sum_i (y W_i^V) W_i^O."""
    Wqkv, Wo, X = _attn_case(24)
    h, _, d_h, d = Wqkv.shape
    cache = core.KVCache.empty(h, 1, d_h, d, "f64")
    S_A = [1, 2]
    out = core.sparse_attn(X[0], Wqkv, Wo, cache, 0, S_A, 1.0)
    ref = sum((Wqkv[i, 2] @ X[0]) @ Wo[i] for i in S_A)
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-13)


def check_attn_uniform_cases():
    """W^Q = 0 (or all positions identical) makes the softmax uniform, so
    H_i is the mean of the value rows."""
    Wqkv, Wo, X = _attn_case(25)
    n = X.shape[0] - 1
    h = Wqkv.shape[0]
    Wq0 = Wqkv.copy()
    Wq0[:, 0] = 0.0
    cache = _dense_prefill(Wq0, X, n, "f64")
    out = core.sparse_attn(X[n], Wq0, Wo, cache, n, range(h), 2.0)
    ref = sum((Wqkv[i, 2] @ X.T).mean(axis=1) @ Wo[i] for i in range(h))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    Xs = np.tile(X[:1], (n + 1, 1))
    cache = _dense_prefill(Wqkv, Xs, n, "f64")
    out = core.sparse_attn(Xs[n], Wqkv, Wo, cache, n, range(h), 1.0)
    ref = sum((Wqkv[i, 2] @ Xs[0]) @ Wo[i] for i in range(h))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def check_attn_history_invariance():
    """Any history of head selections followed by KV repair gives exactly the
    output of a cache in which every head was computed at every step
    (stored rows are the same rounded X W products), in every storage type."""
    for dtype in ("f64", "f16", "bf16"):
        Wqkv, Wo, X = _attn_case(26, n=9)
        h, _, d_h, d = Wqkv.shape
        X = core.round_to(X, dtype)
        rng = RNG(27)
        sparse = core.KVCache.empty(h, 10, d_h, d, dtype)
        dense = core.KVCache.empty(h, 10, d_h, d, dtype)
        for n in range(10):
            S = np.sort(rng.choice(h, rng.integers(1, h + 1), replace=False))
            o_s = core.sparse_attn(X[n], Wqkv, Wo, sparse, n, S, 0.7)
            ref_cache = dense.copy()
            core.kv_append(dense, X[n], Wqkv, n, range(h))
            o_d = core.sparse_attn(X[n], Wqkv, Wo, ref_cache, n, S, 0.7)
            assert np.array_equal(o_s, o_d), (dtype, n)
            assert np.array_equal(sparse.K[:, :n + 1][sparse.valid[:, :n + 1]],
                                  dense.K[:, :n + 1][sparse.valid[:, :n + 1]])


def check_kv_rounding():
    """Stored K/V are the storage-type rounding of X W (and X is stored as is)."""
    Wqkv, Wo, X = _attn_case(28)
    X = core.round_to(X, "f16")
    h, _, d_h, d = Wqkv.shape
    cache = core.KVCache.empty(h, 2, d_h, d, "f16")
    core.sparse_attn(X[0], Wqkv, Wo, cache, 0, [1], 1.0)
    assert np.array_equal(cache.X[0], X[0])
    ref = (Wqkv[1, 1] @ X[0]).astype(np.float16).astype(np.float64)
    assert np.array_equal(cache.K[1, 0], ref)
    assert not cache.valid[0, 0] and cache.valid[1, 0]


def test_attn_golden():
    check_attn_golden()


def test_attn_all_equals_textbook_dense():
    check_attn_all_equals_textbook_dense()


def test_attn_equals_zeroed_wo():
    check_attn_equals_zeroed_wo()


def test_attn_additive():
    check_attn_additive()


def test_attn_first_position():
    check_attn_first_position_closed_form()


def test_attn_uniform_cases():
    check_attn_uniform_cases()


def test_attn_history_invariance():
    check_attn_history_invariance()


def test_kv_rounding():
    check_kv_rounding()


def test_kv_repair_counts():
    Wqkv, Wo, X = _attn_case(29, n=5)
    h, _, d_h, d = Wqkv.shape
    cache = core.KVCache.empty(h, 6, d_h, d, "f64")
    core.sparse_attn(X[0], Wqkv, Wo, cache, 0, [0], 1.0)
    core.sparse_attn(X[1], Wqkv, Wo, cache, 1, [1], 1.0)   # repairs head 1 at 0
    core.sparse_attn(X[2], Wqkv, Wo, cache, 2, [2], 1.0)   # repairs head 2 at 0, 1
    assert cache.valid[:3, :3].tolist() == [[True, False, False],
                                            [True, True, False],
                                            [True, True, True]]
    assert core.kv_repair(cache, Wqkv, 3, [0, 1, 2, 3]) == 2 + 1 + 0 + 3


def test_attn_batched_rows_independent():
    Wqkv, Wo, X = _attn_case(30)
    h, _, d_h, d = Wqkv.shape
    caches = [_dense_prefill(Wqkv, X, 4, "f64") for _ in range(2)]
    refs = [c.copy() for c in caches]
    Y = RNG(31).standard_normal((2, d))
    S = [np.array([0, 1]), np.array([3])]
    out = core.sparse_attn_batched(Y, Wqkv, Wo, caches, [4, 4], S, 1.0)
    for b in range(2):
        assert np.array_equal(out[b], core.sparse_attn(Y[b], Wqkv, Wo, refs[b], 4, S[b], 1.0))


# ---------------------------------------------------------------------------
# layer norm, decoder layer and stack
# ---------------------------------------------------------------------------

def check_layernorm():
    x = RNG(32).standard_normal((3, 64)) * 3 + 1
    ref = F.layer_norm(_t(x), (64,), eps=core.EPS_LN).numpy()
    assert np.allclose(core.layernorm(x), ref, rtol=1e-12, atol=1e-12)
    out = core.layernorm(x)
    var = x.var(axis=1)
    assert np.allclose(out.mean(axis=1), 0, atol=1e-12)
    assert np.allclose(out.var(axis=1) * (var + core.EPS_LN) / var, 1, atol=1e-12)


def test_layernorm():
    check_layernorm()


def _tiny_layers(L, d=16, h=4, d_h=4, N=24, r=8, seed=40):
    rng = RNG(seed)
    return [{"Wqkv": rng.standard_normal((h, 3, d_h, d)) * 0.3,
             "Wo": rng.standard_normal((h, d_h, d)) * 0.3,
             "W1n": rng.standard_normal((N, d)) * 0.3,
             "W2n": rng.standard_normal((N, d)) * 0.3,
             "PA1t": rng.standard_normal((r, d)) / 4, "PA2t": rng.standard_normal((h, r)) / 3,
             "PM1t": rng.standard_normal((r, d)) / 4, "PM2t": rng.standard_normal((N, r)) / 3}
            for _ in range(L)]


def check_layer_dense_equals_textbook():
    """All heads and neurons selected: a textbook pre-LN decoder layer
    (torch layer_norm, SDPA in concat form, linear) in float64."""
    W = _tiny_layers(1)[0]
    h, _, d_h, d = W["Wqkv"].shape
    n = 5
    rng = RNG(41)
    X = rng.standard_normal((n, d))
    r = rng.standard_normal(d)
    cache = _dense_prefill(W["Wqkv"], np.vstack([X, np.zeros(d)]), n, "f64")
    out, y_a = core.decode_layer(r, W, cache, n, range(h), range(W["W1n"].shape[0]), 0.5, "f64")
    ln = lambda v: F.layer_norm(v, (d,), eps=core.EPS_LN)
    ya = ln(_t(r))
    Xall = np.vstack([X, ya.numpy()])
    r1 = _t(r) + _t(_textbook_mha(W["Wqkv"], W["Wo"], Xall, n, 0.5))
    r2 = r1 + F.linear(F.relu(F.linear(ln(r1), _t(W["W1n"]))), _t(W["W2n"]).T)
    assert np.allclose(out, r2.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(y_a, ya.numpy(), rtol=1e-14, atol=1e-14)


def test_layer_dense_equals_textbook():
    check_layer_dense_equals_textbook()


def test_stack_lookahead_composition():
    """Layer 0 predicts from its own attention input; layer l+1's sets are
    predicted from layer l's attention input (checked step by step)."""
    L, kh, kn = 3, 2, 5
    layers = _tiny_layers(L)
    h, _, d_h, d = layers[0]["Wqkv"].shape
    r0 = RNG(42).standard_normal(d)
    caches = [core.KVCache.empty(h, 1, d_h, d, "f16") for _ in range(L)]
    out, sets = core.decode_stack(r0, layers, caches, 0, 0.5, "f16", kh, kn)
    r = r0.copy()
    caches2 = [core.KVCache.empty(h, 1, d_h, d, "f16") for _ in range(L)]
    for l in range(L):
        y_a = core.round_to(core.layernorm(r), "f16")
        src = y_a if l == 0 else prev_y
        S_A = core.predict(src, layers[l]["PA1t"], layers[l]["PA2t"], "topk", kh)[0][0]
        S_M = core.predict(src, layers[l]["PM1t"], layers[l]["PM2t"], "topk", kn)[0][0]
        assert sets[l][0].tolist() == S_A.tolist() and sets[l][1].tolist() == S_M.tolist()
        r, prev_y = core.decode_layer(r, layers[l], caches2[l], 0, S_A, S_M, 0.5, "f16")
    assert np.array_equal(out, r)


def check_prefill_dense_equals_causal_textbook():
    """The dense prompt pass (every head and neuron, positions in order,
    token by token) equals a textbook causal pre-LN stack in matrix form over
    the whole prompt: torch layer_norm, causal scaled-dot-product attention
    (torch SDPA, is_causal), linear layers; every layer's stored inputs and
    K/V rows are the matrix form's."""
    L, T, c = 2, 6, 0.5
    layers = _tiny_layers(L)
    h, _, d_h, d = layers[0]["Wqkv"].shape
    E = RNG(43).standard_normal((T, d))
    caches = [core.KVCache.empty(h, T, d_h, d, "f64") for _ in range(L)]
    out = core.prefill_dense(E, layers, caches, c, "f64")
    ln = lambda v: F.layer_norm(v, (d,), eps=core.EPS_LN)
    R = _t(E)
    for l, W in enumerate(layers):
        Y = ln(R)
        Wq, Wk, Wv = (_t(W["Wqkv"][:, m]) for m in range(3))  # [h][d_h][d]
        Q = torch.einsum("td,hed->hte", Y, Wq)
        K = torch.einsum("td,hed->hte", Y, Wk)
        V = torch.einsum("td,hed->hte", Y, Wv)
        H = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=c)  # [h][T][d_h]
        R = R + torch.einsum("hte,hed->td", H, _t(W["Wo"]))
        R = R + F.linear(F.relu(F.linear(ln(R), _t(W["W1n"]))), _t(W["W2n"]).T)
        assert np.allclose(caches[l].X[:T], Y.numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(caches[l].K[:, :T], K.numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(caches[l].V[:, :T], V.numpy(), rtol=1e-12, atol=1e-12)
        assert caches[l].valid[:, :T].all()
    assert np.allclose(out, R.numpy(), rtol=1e-11, atol=1e-11)


def test_prefill_dense_equals_causal_textbook():
    check_prefill_dense_equals_causal_textbook()


# ---------------------------------------------------------------------------
# planted mistakes: each plausible error in one oracle step fails some pin
# ---------------------------------------------------------------------------

def _relu_dropped_mlp(y, W1n, W2n, S_M):
    S = np.asarray(S_M, dtype=np.int64)
    if S.size == 0:
        return np.zeros(W2n.shape[1])
    return W2n[S].T @ (W1n[S] @ np.asarray(y).reshape(-1))


def _down_with_w1_mlp(y, W1n, W2n, S_M):
    S = np.asarray(S_M, dtype=np.int64)
    if S.size == 0:
        return np.zeros(W2n.shape[1])
    a = np.maximum(0.0, W1n[S] @ np.asarray(y).reshape(-1))
    return W1n[S].T @ a


def _sigmoid_sign_flipped(z):
    return 1.0 / (1.0 + np.exp(z))


def _head_output_no_normalise(q, K, V, c):
    logits = c * (K @ q)
    return np.exp(logits - logits.max()) @ V


def _head_output_drops_current(q, K, V, c):
    K, V = (K[:-1], V[:-1]) if K.shape[0] > 1 else (K, V)
    logits = c * (K @ q)
    w = np.exp(logits - logits.max())
    return (w @ V) / w.sum()


def _topk_ties_high_index(key, k):
    order = np.lexsort((-np.arange(len(key)), -np.asarray(key)))
    return np.sort(order[:k]).astype(np.int32)


def _repair_skipped(cache, Wqkv, n, S_A):
    return 0


def _round_bf16_truncate(x, dtype):
    x = np.asarray(x, dtype=np.float64)
    if dtype != "bf16":
        return _ORIG_ROUND(x, dtype)
    m, e = np.frexp(x)
    return np.ldexp(np.trunc(np.ldexp(m, 8)), e - 8)


_ORIG_ROUND = core.round_to

MUTANTS = [
    ("sparse_mlp", _relu_dropped_mlp, [check_mlp_golden, check_mlp_all_equals_textbook_dense]),
    ("sparse_mlp", _down_with_w1_mlp, [check_mlp_golden, check_mlp_loops,
                                       check_mlp_all_equals_textbook_dense]),
    ("sigmoid", _sigmoid_sign_flipped, [check_predictor_golden, check_predictor_loops]),
    ("head_output", _head_output_no_normalise, [check_attn_golden, check_attn_all_equals_textbook_dense]),
    ("head_output", _head_output_drops_current, [check_attn_golden,
                                                 check_attn_all_equals_textbook_dense,
                                                 check_prefill_dense_equals_causal_textbook]),
    ("select_topk", _topk_ties_high_index, [check_predictor_golden, check_topk_brute_force,
                                            check_predictor_special_cases]),
    ("kv_repair", _repair_skipped, [check_attn_golden, check_attn_history_invariance]),
    ("round_to", _round_bf16_truncate, [check_round_to]),
]


@pytest.mark.parametrize("name,mutant,pins", MUTANTS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant, pins):
    monkeypatch.setattr(core, name, mutant)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()


def test_kv_prefill_matches_append():
    Wqkv, Wo, X = _attn_case(33, n=7)
    h, _, d_h, d = Wqkv.shape
    a = core.KVCache.empty(h, 8, d_h, d, "f64")
    b = core.KVCache.empty(h, 8, d_h, d, "f64")
    for j in range(7):
        core.kv_append(a, X[j], Wqkv, j, range(h))
    b.X[:7] = X[:7]
    core.kv_prefill(b, Wqkv, 7)
    assert np.array_equal(a.valid, b.valid)
    assert np.allclose(a.K, b.K, rtol=1e-13, atol=1e-13) and np.allclose(a.V, b.V, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# true-sparsity labels (the blog page, §1 Contextual Sparsity and §2)
# ---------------------------------------------------------------------------

def _labels_golden():
    with open(os.path.join(GOLDEN, "labels_two_tokens.json")) as f:
        return json.load(f)


def _golden_wqkv(g):
    Wqkv = np.zeros((2, 3, 1, 2))
    for i in range(2):
        Wqkv[i, 0, 0] = g["Wq"][i][0]
        Wqkv[i, 1, 0] = [0.0, g["Wk_second"]]
        Wqkv[i, 2, 0] = g["Wv"][i][0]
    return Wqkv


def check_labels_golden():
    g = _labels_golden()
    n = core.neuron_norms(np.array(g["X_neurons"], float), np.array(g["W1n"], float))
    assert n.shape == (3,) and np.allclose(n, g["neuron_norms"], rtol=0, atol=1e-14)
    Wqkv = _golden_wqkv(g)
    X = np.array(g["X_heads"], float)
    H = core.head_outputs_causal(X, Wqkv, 1.0, "f64")
    assert np.allclose(H, g["head_outputs"], rtol=0, atol=1e-14)
    assert np.allclose(core.head_norms(X, Wqkv, 1.0, "f64"), g["head_norms"], rtol=0, atol=1e-14)
    assert core.label(n, "topk", 1).tolist() == g["top1_neurons"]
    assert core.label(n, "topk", 2).tolist() == g["top2_neurons"]
    assert core.label(n, "threshold", t=1.0).tolist() == g["threshold1_neurons"]
    assert core.label(core.head_norms(X, Wqkv, 1.0, "f64"), "topk", 1).tolist() == g["top1_heads"]


def test_labels_golden():
    check_labels_golden()


def check_neuron_norms_special_cases():
    rng = RNG(71)
    d, N = 12, 9
    W1n = rng.standard_normal((N, d))
    # one token: the norm is the activation itself, ReLU of the pre-activation
    x = rng.standard_normal(d)
    n1 = core.neuron_norms(x[None], W1n)
    assert n1.shape == (N,) and np.allclose(n1, np.maximum(0.0, W1n @ x), rtol=0, atol=1e-13)
    # squared norms add over blocks of tokens
    X1, X2 = rng.standard_normal((4, d)), rng.standard_normal((3, d))
    n12 = core.neuron_norms(np.vstack([X1, X2]), W1n)
    assert np.allclose(n12 ** 2, core.neuron_norms(X1, W1n) ** 2 + core.neuron_norms(X2, W1n) ** 2,
                       rtol=1e-12, atol=1e-12)
    # explicit loops
    X = rng.standard_normal((5, d))
    ref = np.zeros(N)
    for j in range(N):
        s = 0.0
        for t in range(5):
            u = sum(X[t, i] * W1n[j, i] for i in range(d))
            s += max(0.0, u) ** 2
        ref[j] = math.sqrt(s)
    assert np.allclose(core.neuron_norms(X, W1n), ref, rtol=1e-12, atol=1e-12)


def test_neuron_norms_special_cases():
    check_neuron_norms_special_cases()


def check_head_outputs_causal():
    rng = RNG(72)
    h, d_h, d, T = 3, 4, 8, 6
    Wqkv = rng.standard_normal((h, 3, d_h, d)) * 0.5
    X = rng.standard_normal((T, d))
    for dtype in ("f64", "bf16"):
        H = core.head_outputs_causal(X, Wqkv, 0.7, dtype)
        # textbook causal attention (torch float64, boolean causal mask)
        for i in range(h):
            Q = torch.tensor(X @ Wqkv[i, 0].T)
            K = torch.tensor(core.round_to(X @ Wqkv[i, 1].T, dtype))
            V = torch.tensor(core.round_to(X @ Wqkv[i, 2].T, dtype))
            ref = F.scaled_dot_product_attention(Q[None], K[None], V[None], is_causal=True, scale=0.7)[0]
            assert np.allclose(H[i], ref.numpy(), rtol=1e-12, atol=1e-12)
        # a prefix of the sequence has the same outputs (causality)
        Hp = core.head_outputs_causal(X[:3], Wqkv, 0.7, dtype)
        assert np.array_equal(Hp, H[:, :3])
    # one token: the head output is its own value row
    H1 = core.head_outputs_causal(X[:1], Wqkv, 0.7, "f64")
    for i in range(h):
        assert np.allclose(H1[i, 0], Wqkv[i, 2] @ X[0], rtol=0, atol=1e-13)
    # W^Q = 0: uniform weights, running means of the value rows
    Wz = Wqkv.copy()
    Wz[:, 0] = 0.0
    Hz = core.head_outputs_causal(X, Wz, 0.7, "f64")
    for i in range(h):
        Vr = X @ Wz[i, 2].T
        assert np.allclose(Hz[i], np.cumsum(Vr, axis=0) / np.arange(1, T + 1)[:, None], rtol=1e-12,
                           atol=1e-12)
    # the norms are the Frobenius norms of these matrices
    n = core.head_norms(X, Wqkv, 0.7, "f64")
    assert np.allclose(n, [np.linalg.norm(core.head_outputs_causal(X, Wqkv, 0.7, "f64")[i]) for i in range(h)],
                       rtol=1e-13, atol=0)


def test_head_outputs_causal():
    check_head_outputs_causal()


def _neuron_norms_no_relu(X, W1n):
    A = np.atleast_2d(X) @ W1n.T
    return np.sqrt((A * A).sum(axis=0))


def _neuron_norms_per_token(X, W1n):
    A = np.maximum(0.0, np.atleast_2d(X) @ W1n.T)
    return np.sqrt((A * A).sum(axis=1))


def _head_outputs_not_causal(X, Wqkv, c, dtype):
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    T = X.shape[0]
    h, _, d_h, _ = Wqkv.shape
    out = np.zeros((h, T, d_h))
    for i in range(h):
        Q = X @ Wqkv[i, 0].T
        K = core.round_to(X @ Wqkv[i, 1].T, dtype)
        V = core.round_to(X @ Wqkv[i, 2].T, dtype)
        for t in range(T):
            out[i, t] = core.head_output(Q[t], K, V, c)
    return out


LABEL_MUTANTS = [
    ("neuron_norms", _neuron_norms_no_relu, [check_labels_golden, check_neuron_norms_special_cases]),
    ("neuron_norms", _neuron_norms_per_token, [check_labels_golden, check_neuron_norms_special_cases]),
    ("head_outputs_causal", _head_outputs_not_causal, [check_labels_golden, check_head_outputs_causal]),
]


@pytest.mark.parametrize("name,mutant,pins", LABEL_MUTANTS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in LABEL_MUTANTS])
def test_planted_label_mistake_is_caught(monkeypatch, name, mutant, pins):
    monkeypatch.setattr(core, name, mutant)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()

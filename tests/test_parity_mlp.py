"""GPU parity of dv_sparse_mlp with the float64 oracle (given identical
index lists): relative L2 error <= 1e-3 for fp16 / bf16 and <= 1e-5 for fp32,
element by element on every output."""

import zlib

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from dvtest import assert_rel_l2, f64
from synth import draw, keep_count

pytestmark = pytest.mark.gpu

#        name                     B   d      N      dtype   k
CASES = [
    ("tiny_ragged_f16",           1, 64,    100,   "f16",  7),
    ("d136_f16",                  1, 136,   544,   "f16",  33),
    ("opt1.3b_f16",               1, 2048,  8192,  "f16",  410),
    ("opt13b_f16",                1, 5120,  20480, "f16",  1024),
    ("d2560_f16_5chunk",          1, 2560,  10240, "f16",  301),
    ("f32_d1200_5chunk_ragged",   1, 1200,  4800,  "f32",  97),
    ("batch3_f16_d5120",          3, 5120,  20480, "f16",  555),
    ("opt30b_bf16",               1, 7168,  28672, "bf16", 1434),
    ("opt30b_bf16_half",          1, 7168,  28672, "bf16", 14336),
    ("opt175b_f16",               1, 12288, 49152, "f16",  2458),
    ("bf16_small",                1, 512,   2048,  "bf16", 103),
    ("f32_d1024",                 1, 1024,  4096,  "f32",  205),
    ("batch3_f16",                3, 1024,  4096,  "f16",  205),
    ("batch8_f16",                8, 2048,  8192,  "f16",  410),
    ("batch13_bf16",              13, 1024, 4096,  "bf16", 205),
    ("batch16_f16_tc",            16, 2048, 8192,  "f16",  410),
    ("batch32_bf16_opt30b_tc",    32, 7168, 28672, "bf16", 1434),
    ("batch32_f16_ragged_tc",     32, 768,  3000,  "f16",  77),
    ("batch8_f32_cuda_cores",     8, 512,   2048,  "f32",  103),
    ("stream_ragged_f16",         1, 8200,  8400,  "f16",  3100),   # >= 96 MB: streaming pass
    ("stream_f32",                1, 4096,  16384, "f32",  3100),
    ("all_neurons_f16",           1, 256,   1024,  "f16",  1024),
    ("one_neuron_f16",            1, 256,   1024,  "f16",  1),
]


def _weights(name, d, N, dtype, wid=201):
    return (draw((N, d), 0.02, wid, name + "/W1", dtype), draw((N, d), 0.02, wid, name + "/W2", dtype))


def _sets(name, B, N, k):
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    return [torch.sort(torch.randperm(N, generator=g)[:k]).values.to(torch.int32) for _ in range(B)]


def _run(y, W1n, W2n, sets, cap, accumulate=False, base=None, ws=None):
    dev = "cuda"
    B, d = y.shape
    idx = torch.full((B, cap), -1, dtype=torch.int32)
    cnt = torch.zeros(B, dtype=torch.int32)
    for b, s in enumerate(sets):
        idx[b, : len(s)] = s
        cnt[b] = len(s)
    out = (base.clone() if base is not None else torch.full((B, d), 123.0)).to(dev)
    if ws is None:
        ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(B, d, W1n.shape[0], cap))
    dv.dv_sparse_mlp(y.to(dev), W1n.to(dev), W2n.to(dev), idx.to(dev), cnt.to(dev), out, ws,
                     accumulate=accumulate)
    st, info = dv.dv_check(ws)
    return out.cpu().double().numpy(), st, info


def _marks(case):
    # batches of 2+ rows in a 16-bit type run on the tcgen05 path
    return [pytest.mark.tc] if case[1] >= 8 and case[4] != "f32" else []


@pytest.mark.parametrize("case", [pytest.param(c, id=c[0], marks=_marks(c)) for c in CASES])
def test_sparse_mlp_parity(case):
    name, B, d, N, dtype, k = case
    W1n, W2n = _weights(name, d, N, dtype)
    y = draw((B, d), 1.0, 201, name + "/y", dtype)
    sets = _sets(name, B, N, k)
    out, st, info = _run(y, W1n, W2n, sets, k)
    assert st == 0, (st, info)
    ref = oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s.numpy() for s in sets])
    for b in range(B):
        assert_rel_l2(out[b], ref[b], dtype, f"{name} row {b}")


def test_fp32_mlp_block_true_preactivation_top5pct():
    """Single fp32 MLP block, d = 768, 4d = 3072: S_M = the 154 neurons with the
    largest true pre-activation y . W^1[:, j] (computed by the oracle)."""
    d, N = 768, 3072
    k = keep_count(5, N)
    W1n, W2n = _weights("c1", d, N, "f32", wid=1)
    y = draw((1, d), 1.0, 1, "c1/y", "f32")
    pre = f64(W1n) @ f64(y)[0]
    S = oracle.select_topk(pre, k)
    out, st, _ = _run(y, W1n, W2n, [torch.from_numpy(S)], k)
    assert st == 0 and k == 154
    ref = oracle.sparse_mlp(f64(y)[0], f64(W1n), f64(W2n), S)
    assert_rel_l2(out[0], ref, "f32", "fp32 block")


def test_accumulate_adds_to_residual():
    d, N, k = 1024, 4096, 205
    W1n, W2n = _weights("acc", d, N, "f16")
    y = draw((2, d), 1.0, 202, "acc/y", "f16")
    base = draw((2, d), 3.0, 202, "acc/base", "f32")
    sets = _sets("acc", 2, N, k)
    out, st, _ = _run(y, W1n, W2n, sets, k, accumulate=True, base=base)
    assert st == 0
    ref = oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s.numpy() for s in sets])
    for b in range(2):
        assert_rel_l2(out[b] - f64(base)[b], ref[b], "f16", "accumulate")


def test_empty_selection_gives_zero():
    d, N = 512, 2048
    W1n, W2n = _weights("empty", d, N, "f16")
    y = draw((2, d), 1.0, 203, "empty/y", "f16")
    out, st, _ = _run(y, W1n, W2n, [torch.zeros(0, dtype=torch.int32)] * 2, 16)
    assert st == 0 and np.all(out == 0.0)


def test_out_of_range_index_is_skipped_and_reported():
    d, N, k = 512, 2048, 20
    W1n, W2n = _weights("oor", d, N, "f16")
    y = draw((1, d), 1.0, 204, "oor/y", "f16")
    S = _sets("oor", 1, N, k)[0].clone()
    S[-1] = N + 5  # outside [0, N)
    out, st, info = _run(y, W1n, W2n, [S], k)
    assert st == 5 and info == N + 5   # DV_ERR_INDEX_RANGE
    ref = oracle.sparse_mlp(f64(y)[0], f64(W1n), f64(W2n), S[:-1].numpy())
    assert_rel_l2(out[0], ref, "f16", "valid part")


def test_batch_rows_use_their_own_sets():
    """Masked union semantics: each row equals its batch-1 result."""
    d, N, k = 1024, 4096, 205
    W1n, W2n = _weights("mask", d, N, "f16")
    y = draw((4, d), 1.0, 205, "mask/y", "f16")
    sets = _sets("mask", 4, N, k)
    out, st, _ = _run(y, W1n, W2n, sets, k)
    assert st == 0
    for b in range(4):
        one, _, _ = _run(y[b:b + 1], W1n, W2n, [sets[b]], k)
        assert np.allclose(out[b], one[0], rtol=1e-5, atol=1e-6)


def test_batch1_calls_share_one_workspace():
    """At batch 1 both products run in one launch whose arrival counters live
    in the workspace: consecutive calls on one workspace (different sets, an
    empty one, accumulate on and off, an index outside [0, N)) each match
    the oracle, and the counters are back at zero after each call."""
    d, N, cap = 1024, 4096, 300
    W1n, W2n = _weights("reuse", d, N, "f16")
    dev = "cuda"
    W1d, W2d = W1n.to(dev), W2n.to(dev)
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(1, d, N, cap))
    g = torch.Generator().manual_seed(11)
    for step, k in enumerate([205, 0, 300, 1, 150, 40]):
        y = draw((1, d), 1.0, 208, f"reuse/y{step}", "f16")
        S = torch.sort(torch.randperm(N, generator=g)[:k]).values.to(torch.int32)
        bad = step == 5
        if bad:
            S[-1] = N + 3
        idx = torch.full((1, cap), -1, dtype=torch.int32)
        idx[0, :k] = S
        cnt = torch.tensor([k], dtype=torch.int32)
        acc = step % 2 == 1
        base = draw((1, d), 1.0, 208, f"reuse/base{step}", "f32")
        out = base.clone().to(dev) if acc else torch.full((1, d), 55.0, device=dev)
        dv.dv_sparse_mlp(y.to(dev), W1d, W2d, idx.to(dev), cnt.to(dev), out, ws, accumulate=acc)
        st, info = dv.dv_check(ws)
        assert (st, info) == ((5, N + 3) if bad else (0, 0)), (step, st, info)
        got = f64(out)[0] - (f64(base)[0] if acc else 0.0)
        kept = [j for j in S.tolist() if j < N]
        if not kept:
            assert np.all(got == 0.0)
        else:
            ref = oracle.sparse_mlp(f64(y)[0], f64(W1n), f64(W2n), np.array(kept))
            assert_rel_l2(got, ref, "f16", f"call {step}")


def test_streaming_pass_out_of_range_index_and_reuse():
    """The streaming batch-1 pass (selected rows >= 96 MB): an index outside
    [0, N) is skipped and reported; the same workspace then serves a clean
    call, accumulating into a residual."""
    d, N, k = 8192, 16384, 3100
    W1n, W2n = _weights("strm", d, N, "f16")
    y = draw((1, d), 1.0, 209, "strm/y", "f16")
    S = _sets("strm", 1, N, k)[0].clone()
    S[7] = N + 11
    S = torch.sort(S).values
    out, st, info = _run(y, W1n, W2n, [S], k)
    assert st == 5 and info == N + 11
    kept = S[S < N].numpy()
    assert_rel_l2(out[0], oracle.sparse_mlp(f64(y)[0], f64(W1n), f64(W2n), kept), "f16", "valid part")
    base = draw((1, d), 1.0, 209, "strm/base", "f32")
    S2 = _sets("strm2", 1, N, k)[0]
    out2, st2, _ = _run(y, W1n, W2n, [S2], k, accumulate=True, base=base)
    assert st2 == 0
    assert_rel_l2(out2[0] - f64(base)[0], oracle.sparse_mlp(f64(y)[0], f64(W1n), f64(W2n), S2.numpy()),
                  "f16", "accumulate")


def test_large_batch_union_with_out_of_range_index():
    """16 rows x 600 neurons: the union is built in two passes over a grid;
    an index outside [0, N) in one row is skipped and reported, every row
    still matches its own set."""
    B, d, N, k = 16, 1024, 4096, 600
    W1n, W2n = _weights("bigu", d, N, "f16")
    y = draw((B, d), 1.0, 210, "bigu/y", "f16")
    sets = _sets("bigu", B, N, k)
    bad = sets[5].clone()
    bad[-1] = N + 2
    sets[5] = bad
    out, st, info = _run(y, W1n, W2n, sets, k)
    assert st == 5 and info == N + 2
    ref = oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s[s < N].numpy() for s in sets])
    for b in range(B):
        assert_rel_l2(out[b], ref[b], "f16", f"row {b}")


@pytest.mark.tc
def test_device_split_up_projection_partial_tiles():
    """32 rows whose sets overlap heavily: the largest possible union (all
    28672 neurons) has more tiles than half the SMs, so the up-projection's
    K split is chosen on the device from the actual union (16 or ~80 tiles
    of 128: 4 or 3 splits, partial tiles summed with fp32 atomics and
    finished by each tile's last CTA).  Three calls on one workspace, the
    union shrinking and growing between them, each against the oracle (the
    partial tiles and their counts must come back to zero after every call)."""
    B, d, N, k = 32, 7168, 28672, 1434
    name = "dsplit"
    W1n, W2n = _weights(name, d, N, "bf16")
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(B, d, N, k))
    g = torch.Generator().manual_seed(77)
    for call, pool_n in enumerate((2000, 10000, 2000)):
        pool = torch.randperm(N, generator=g)[:pool_n]
        sets = [torch.sort(pool[torch.randperm(pool_n, generator=g)[:k]]).values.to(torch.int32)
                for _ in range(B)]
        y = draw((B, d), 1.0, 212, f"{name}/y{call}", "bf16")
        base = draw((B, d), 1.0, 212, f"{name}/base{call}", "f32")
        out, st, info = _run(y, W1n, W2n, sets, k, accumulate=True, base=base, ws=ws)
        assert (st, info) == (0, 0), (call, st, info)
        ref = oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s.numpy() for s in sets])
        for b in range(B):
            assert_rel_l2(out[b] - f64(base)[b], ref[b], "bf16", f"call {call} row {b}")


@pytest.mark.parametrize("B,cap", [(4, 100), (16, 600)], ids=["one_cta_union", "two_pass_union"])
def test_batch_count_above_capacity_is_clamped_and_reported(B, cap):
    """A row whose count exceeds the list's capacity: the union uses its
    first cap entries and reports DV_ERR_CAPACITY (the single-CTA union
    below 8192 entries and the two-pass union above)."""
    d, N = 1024, 4096
    name = f"capx_{B}"
    W1n, W2n = _weights(name, d, N, "f16")
    y = draw((B, d), 1.0, 213, name + "/y", "f16")
    sets = _sets(name, B, N, cap)
    dev = "cuda"
    idx = torch.stack(sets).to(torch.int32)
    cnt = torch.full((B,), cap, dtype=torch.int32)
    cnt[1] = cap + 5
    out = torch.zeros(B, d, device=dev)
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(B, d, N, cap))
    dv.dv_sparse_mlp(y.to(dev), W1n.to(dev), W2n.to(dev), idx.to(dev), cnt.to(dev), out, ws)
    st, info = dv.dv_check(ws)
    assert (st, info) == (8, cap + 5)  # DV_ERR_CAPACITY
    ref = oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s.numpy() for s in sets])
    got = out.cpu().double().numpy()
    for b in range(B):
        assert_rel_l2(got[b], ref[b], "f16", f"row {b}")

"""GPU parity of dv_kv_repair -- the prompt's KV cache fill and the bulk
repair of skipped heads -- with the float64 oracle (oracle.kv_prefill for a
dense prompt, oracle.kv_repair for scattered missing positions).

For 16-bit storage the product X[j] [W_i^K; W_i^V]^T runs on the tcgen05
tensor cores (one CTA per head and 128 missing positions, X rows gathered
by TMA); fp32 storage uses the CUDA-core GEMM.  Checked:
  * every filled K/V element within one unit in the last place of the
    oracle's rounded product, plus an fp32 summation allowance;
  * K/V rows that were already valid, rows of heads not selected and rows at
    or after the position are left untouched (sentinel values survive);
  * the valid flags: 1 for every j < pos of every selected head, else as
    before.
The Deja Vu reading notes, "Typical LLM procedure" (the prompt phase builds
the KV cache of every layer) and "Sparsity operator for Attention" (skipped
heads recomputed from the stored embeddings)."""

import zlib

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from dvtest import TORCH, f64, within_ulp
from synth import draw

pytestmark = pytest.mark.gpu

SENT = 7.0  # sentinel in rows that must not be written


def _fill(name, B, d, h, d_h, dtype, n_max, pos, heads, valid_p, check_heads=None, wid=331):
    """Run dv_kv_repair on a cache whose valid flags are drawn with
    probability valid_p (1.0 = nothing missing, 0.0 = a dense prompt) and
    compare with the oracle.  heads[b] = selected heads of row b."""
    dev = "cuda"
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    Wqkv = draw((h, 3, d_h, d), d ** -0.5, wid, name + "/Wqkv", dtype)
    X = draw((B, n_max, d), 1.0, wid, name + "/X", dtype)
    valid = (torch.rand((B, h, n_max), generator=g) < valid_p).to(torch.uint8)
    kv = dv.KV.empty(B, h, n_max, d_h, d, TORCH[dtype], dev)
    kv.K.fill_(SENT)
    kv.V.fill_(-SENT)
    kv.X.copy_(X.to(dev))
    kv.valid.copy_(valid.to(dev))
    cap = max(1, max(len(x) for x in heads))
    idx = torch.full((B, cap), -1, dtype=torch.int32)
    cnt = torch.zeros(B, dtype=torch.int32)
    for b, hs in enumerate(heads):
        idx[b, : len(hs)] = torch.tensor(hs, dtype=torch.int32)
        cnt[b] = len(hs)
    pos_t = torch.tensor(pos, dtype=torch.int32)
    ws = dv.workspace(dv.dv_sparse_attn_workspace_size(B, d, h, d_h, cap, n_max))
    dv.dv_kv_repair(kv, Wqkv.to(dev), pos_t.to(dev), idx.to(dev), cnt.to(dev), ws)
    assert dv.dv_check(ws) == (0, 0)
    K, V, vflag = f64(kv.K), f64(kv.V), kv.valid.cpu().numpy().astype(bool)
    W64 = Wqkv.float().numpy()  # exact; products with the float64 X run in float64
    X64 = f64(X)
    for b in range(B):
        n = pos[b]
        sel = set(heads[b])
        c = oracle.KVCache(np.full((h, n_max, d_h), SENT), np.full((h, n_max, d_h), -SENT), X64[b].copy(),
                           valid[b].numpy().astype(bool), dtype)
        if valid_p == 0.0 and len(sel) == h:
            oracle.kv_prefill(c, W64, n, heads=check_heads)
            if check_heads is not None:  # the other heads are checked for their flags only
                c.valid[:, :n] = True
        else:
            oracle.kv_repair(c, W64, n, sorted(sel))
        assert np.array_equal(vflag[b], c.valid), f"{name} row {b}: valid flags"
        for i in (check_heads if check_heads is not None else range(h)):
            for got, ref, what in ((K[b, i], c.K[i], "K"), (V[b, i], c.V[i], "V")):
                filled = ref != (SENT if what == "K" else -SENT)
                # rows never filled keep the sentinel exactly
                assert np.all(got[~filled] == ref[~filled]), f"{name} row {b} head {i} {what}: untouched rows"
                if filled.any():
                    # fp32 accumulation of d products: ~sqrt(d) roundings of the running sum
                    acc = 4.0 * np.sqrt(d) * 2.0 ** -24 * np.abs(ref[filled]).max()
                    assert within_ulp(got[filled], ref[filled], dtype, acc_floor=acc), \
                        f"{name} row {b} head {i} {what}: filled rows"


def test_dense_prompt_opt13b_f16():
    """The OPT-13B-shaped prompt: 1024 positions, all 40 heads, d = 5120."""
    _fill("p13b", 1, 5120, 40, 128, "f16", 1040, [1024], [list(range(40))], 0.0)


def test_dense_prompt_opt175b_f16_sampled_heads():
    """The OPT-175B-shaped prompt: 2047 positions, all 96 heads, d = 12288
    (the tensor-core kernel fills every head; 6 heads are compared element by
    element, the flags of all)."""
    _fill("p175b", 1, 12288, 96, 128, "f16", 2048, [2047], [list(range(96))], 0.0,
          check_heads=[0, 1, 37, 64, 94, 95])


def test_dense_prompt_opt30b_bf16_batch():
    """Two OPT-30B-shaped rows (d = 7168, 56 heads) with ragged prompts."""
    _fill("p30b", 2, 7168, 56, 128, "bf16", 2048, [2047, 777], [list(range(56))] * 2, 0.0,
          check_heads=[0, 13, 55])


@pytest.mark.parametrize("valid_p", [0.5, 0.97])
def test_scattered_repair_f16(valid_p):
    """Random missing positions (more than 128 per head, so several position
    tiles; more than 2048 positions, so several scan rounds), random head
    subsets per row, ragged positions."""
    _fill(f"scat{valid_p}", 3, 1024, 12, 128, "f16", 2560, [2500, 9, 1300],
          [[0, 3, 4, 11], [5], [1, 2, 3, 4, 5, 6, 7, 8]], valid_p)


def test_scattered_repair_bf16_dh64_ragged_d():
    """d_h = 64 and d = 136 (the last 64-element step of d is partly outside
    the row: the copy fills zeros there)."""
    _fill("scat64", 2, 136, 6, 64, "bf16", 304, [300, 157], [[0, 5], [1, 2, 3]], 0.3)


def test_scattered_repair_f32_cuda_cores():
    _fill("scat32", 2, 256, 4, 128, "f32", 208, [200, 31], [[0, 3], [1]], 0.4)


def test_nothing_missing_and_no_heads():
    """All flags set: nothing is written; an empty head list: nothing either."""
    _fill("none", 1, 512, 8, 64, "f16", 64, [50], [[1, 2, 7]], 1.0)
    _fill("empty", 2, 512, 8, 64, "f16", 64, [50, 20], [[], []], 0.2)

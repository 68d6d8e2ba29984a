"""Teacher-forced parity of the decoder stack with the float64 oracle.

The GPU runs the real decode path -- pre-LN layers, layer l+1's heads and
neurons predicted from layer l's attention input on a side stream
(dv_lookahead), the whole token replayed as one CUDA graph -- for several
tokens.  The stack keeps each layer's own inputs: the attention input
y_a[l], the MLP input y_m[l], and the residual stream before layer 0 and
after every block.  The oracle then takes each link of the chain on the
GPU's own inputs ("用Deja Vu来提高 LLM 的推理速度" §3.1 and the Deja Vu reading
notes, "Reducing Overhead with Asynchronous Execution", for the look-ahead;
"Sparsified Attention" / "Sparsified MLP" for the blocks):

* index lists: layer 0's from its own y_a[0], layer l's from y_a[l-1];
  exact except units whose oracle score is within 1e-5 of the k-th score;
* layer norms: y_a[l] = LN(residual before the layer) and y_m[l] = LN(residual
  after the attention), within one unit in the last place of the storage type;
* attention: the residual's change across the block against the oracle's
  MHA_{S_A}(y_a[l]) over its own KV cache (own prefill, own appends and
  repairs), relative L2 <= 1e-3 (fp16 / bf16);
* MLP: the residual's change against MLP_{S_M}(y_m[l]), relative L2 <= 1e-3;
* after the last token, every layer's KV cache: the valid flags exactly and
  the K/V rows within one unit in the last place of the oracle's.

The blocks are checked with the GPU's index lists (identical to the
oracle's outside the 1e-5 window), so every layer of every token is compared:
nothing stops at a near-tie flip.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from contextual_sparsity_decode_gb300.stack import SparseDecoder
from dvtest import assert_rel_l2, check_selection, within_ulp
from synth import WORKLOADS, Workload, embeddings, layer_weights, residual_input

pytestmark = pytest.mark.gpu


def _np(t: torch.Tensor) -> np.ndarray:
    """Host float64 copy (exact for every storage type)."""
    return t.detach().to("cpu", torch.float32).double().numpy()


def _run_gpu(w: Workload, B: int, steps: int):
    """Decode `steps` tokens on the GPU and return the per-token records,
    the prompt embeddings and the decoder (for its weights and caches)."""
    dev = "cuda"
    layers = [layer_weights(w, l, device=dev) for l in range(w.layers)]
    n_max = ((w.n_prompt + steps + 15) // 16) * 16
    scale = 1.0 / math.sqrt(w.d_h)
    dec = SparseDecoder(layers, B, n_max, w.k_heads, w.k_neurons, scale, trace=True)
    Xp = [torch.stack([embeddings(w, w.n_prompt, f"X{l}/{b}", device=dev) for b in range(B)])
          for l in range(w.layers)]
    dec.prefill(Xp, w.n_prompt)
    dec.r_stream.copy_(residual_input(w, B, "r0", device=dev))
    recs = []
    for t in range(steps):
        if t == 1:
            dec.capture(advance=(0, n_max))
        if t >= 1:
            dec.replay()
        else:  # the first token runs eagerly, the others replay the graph
            dec.step_ops()
            dv.dv_positions_advance(dec.pos, 0, n_max)
        dec.check()
        L = w.layers
        recs.append({
            "r_in0": _np(dec.r_in0),
            "r_mid": [_np(dec.r_mid[l]) for l in range(L)],
            "r_out": [_np(dec.r_out[l]) for l in range(L)],
            "y_a": [_np(dec.y_a[l]) for l in range(L)],
            "y_m": [_np(dec.y_m[l]) for l in range(L)],
            "S_A": [[dec.head_idx[l][b, : int(dec.head_cnt[l][b])].cpu().numpy() for b in range(B)]
                    for l in range(L)],
            "S_M": [[dec.neur_idx[l][b, : int(dec.neur_cnt[l][b])].cpu().numpy() for b in range(B)]
                    for l in range(L)],
        })
    return recs, Xp, dec, scale


def _teacher_forced(w: Workload, B: int, steps: int):
    recs, Xp, dec, scale = _run_gpu(w, B, steps)
    dt = w.dtype
    flips = 0
    compared = 0
    for l in range(w.layers):
        # this layer's weights on the host (float32 holds every storage type
        # exactly; each product with a float64 vector runs in float64)
        W = {k: v.detach().to("cpu", torch.float32).numpy() for k, v in dec.layers[l].items()}
        for k in ("PA1t", "PA2t", "PM1t", "PM2t"):
            W[k] = W[k].astype(np.float64)
        caches = []
        for b in range(B):
            c = oracle.KVCache.empty(w.h, dec.n_max, w.d_h, w.d, dt)
            c.X[: w.n_prompt] = _np(Xp[l][b])
            oracle.kv_prefill(c, W["Wqkv"], w.n_prompt)
            caches.append(c)
        for t, rec in enumerate(recs):
            n = w.n_prompt + t
            r_in = rec["r_in0"] if l == 0 else rec["r_out"][l - 1]
            src = rec["y_a"][0] if l == 0 else rec["y_a"][l - 1]
            for b in range(B):
                where = f"layer {l} token {t} row {b}"
                # index lists predicted from the GPU's own predictor input
                S_A, sA, _ = oracle.predict(src[b], W["PA1t"], W["PA2t"], "topk", w.k_heads)
                S_M, sM, _ = oracle.predict(src[b], W["PM1t"], W["PM2t"], "topk", w.k_neurons)
                gA, gM = rec["S_A"][l][b], rec["S_M"][l][b]
                assert np.all(np.diff(gA) > 0) and np.all(np.diff(gM) > 0), where
                flips += check_selection(gA, S_A[0], sA[0], "topk", w.k_heads)
                flips += check_selection(gM, S_M[0], sM[0], "topk", w.k_neurons)
                # pre-LN of each block
                assert within_ulp(rec["y_a"][l][b], oracle.layernorm(r_in[b]), dt), where + " LN_a"
                assert within_ulp(rec["y_m"][l][b], oracle.layernorm(rec["r_mid"][l][b]), dt), \
                    where + " LN_m"
                # the attention block on its own input, with the lists it used
                ref_a = oracle.sparse_attn(rec["y_a"][l][b], W["Wqkv"], W["Wo"], caches[b], n,
                                           gA.tolist(), scale)
                assert_rel_l2(rec["r_mid"][l][b] - r_in[b], ref_a, dt, where + " attention")
                ref_m = oracle.sparse_mlp(rec["y_m"][l][b], W["W1n"], W["W2n"], gM)
                assert_rel_l2(rec["r_out"][l][b] - rec["r_mid"][l][b], ref_m, dt, where + " mlp")
                compared += 1
        # the KV cache after the last token: same valid flags, K/V within 1 ulp
        kv = dec.kv[l]
        for b in range(B):
            valid = kv.valid[b].cpu().numpy().astype(bool)
            assert np.array_equal(valid, caches[b].valid), f"layer {l} row {b} valid flags"
            for name, ref in (("K", caches[b].K), ("V", caches[b].V)):
                got = _np(getattr(kv, name)[b])
                # fp32 accumulation of d products: ~sqrt(d) roundings of the running sum
                acc = 4.0 * np.sqrt(w.d) * 2.0 ** -24 * np.abs(ref).max()
                assert within_ulp(got[valid], ref[valid], dt, acc_floor=acc), f"layer {l} row {b} {name}"
    assert compared == w.layers * steps * B
    return flips


def test_tiny_stack_teacher_forced():
    w = Workload("tiny_stack", 31, d=256, h=8, d_h=64, N=1024, r=64, dtype="f16", layers=3,
                 n_prompt=20, n_gen=6, head_pct=25, neuron_pct=5)
    _teacher_forced(w, B=1, steps=6)


def test_bf16_stack_teacher_forced():
    w = Workload("bf16_stack", 32, d=512, h=8, d_h=128, N=2048, r=128, dtype="bf16", layers=4,
                 n_prompt=33, n_gen=5, head_pct=25, neuron_pct=10)
    _teacher_forced(w, B=1, steps=5)


def test_batched_stack_teacher_forced():
    """Three sequences decoded together: every row has its own lists, cache
    and residual stream (the batch union is read once)."""
    w = Workload("batch_stack", 33, d=512, h=8, d_h=64, N=2048, r=128, dtype="f16", layers=3,
                 n_prompt=40, n_gen=4, head_pct=25, neuron_pct=5)
    _teacher_forced(w, B=3, steps=4)


def test_batch8_stack_teacher_forced():
    """Eight sequences: both sparse blocks take the tensor-core path (the
    batch union as a dense contraction), accumulating into the residual."""
    w = Workload("batch8_stack", 34, d=512, h=8, d_h=64, N=2048, r=128, dtype="f16", layers=2,
                 n_prompt=24, n_gen=4, head_pct=25, neuron_pct=5)
    _teacher_forced(w, B=8, steps=4)


def test_opt13b_stack_all_layers_teacher_forced():
    """All 40 layers of the OPT-13B-shaped stack (d = 5120, 40 heads of 128,
    FFN 20480, rank-1024 predictors, 8 heads / 1024 neurons) after the
    1024-position prompt, for 8 decoded tokens: the benchmark's configuration."""
    w = WORKLOADS["opt13b_stack_fp16"]
    _teacher_forced(w, B=1, steps=8)


def _prefill_teacher_forced(w: Workload, B: int):
    """The dense prompt pass (SparseDecoder.prefill_dense) against the
    oracle, position by position and layer by layer on the GPU's own inputs
    (Deja Vu reading notes, "Typical LLM procedure"): LN outputs within one
    ulp, the attention block with every head over the position's causal
    prefix and the MLP with every neuron within rel-L2 1e-3, and after the
    prompt every layer's stored inputs X, valid flags and K/V rows."""
    dev = "cuda"
    layers = [layer_weights(w, l, device=dev) for l in range(w.layers)]
    n_max = ((w.n_prompt + 15) // 16) * 16
    scale = 1.0 / math.sqrt(w.d_h)
    dec = SparseDecoder(layers, B, n_max, w.k_heads, w.k_neurons, scale, trace=True)
    E = torch.stack([embeddings(w, w.n_prompt, f"E/{b}", device=dev).float() for b in range(B)])
    L = w.layers
    recs = []

    def record(t):
        recs.append({"r_in0": _np(dec.r_in0), "r_mid": [_np(dec.r_mid[l]) for l in range(L)],
                     "r_out": [_np(dec.r_out[l]) for l in range(L)],
                     "y_a": [_np(dec.y_a[l]) for l in range(L)], "y_m": [_np(dec.y_m[l]) for l in range(L)]})

    dec.prefill_dense(E, w.n_prompt, on_position=record)
    assert dec.k_heads == w.k_heads and dec.k_neurons == w.k_neurons
    assert dec.pos.cpu().tolist() == [w.n_prompt] * B
    dt = w.dtype
    E64 = _np(E)
    every_h, every_n = list(range(w.h)), np.arange(w.N)
    for l in range(L):
        W = {k: v.detach().to("cpu", torch.float32).numpy() for k, v in dec.layers[l].items()}
        caches = [oracle.KVCache.empty(w.h, n_max, w.d_h, w.d, dt) for _ in range(B)]
        for t, rec in enumerate(recs):
            r_in = rec["r_in0"] if l == 0 else rec["r_out"][l - 1]
            if l == 0:
                assert np.array_equal(r_in, E64[:, t]), f"position {t}: layer 0 input"
            for b in range(B):
                where = f"layer {l} position {t} row {b}"
                assert within_ulp(rec["y_a"][l][b], oracle.layernorm(r_in[b]), dt), where + " LN_a"
                assert within_ulp(rec["y_m"][l][b], oracle.layernorm(rec["r_mid"][l][b]), dt), \
                    where + " LN_m"
                ref_a = oracle.sparse_attn(rec["y_a"][l][b], W["Wqkv"], W["Wo"], caches[b], t, every_h, scale)
                assert_rel_l2(rec["r_mid"][l][b] - r_in[b], ref_a, dt, where + " attention")
                ref_m = oracle.sparse_mlp(rec["y_m"][l][b], W["W1n"], W["W2n"], every_n)
                assert_rel_l2(rec["r_out"][l][b] - rec["r_mid"][l][b], ref_m, dt, where + " mlp")
        kv = dec.kv[l]
        T = w.n_prompt
        for b in range(B):
            assert np.array_equal(_np(kv.X[b])[:T], caches[b].X[:T]), f"layer {l} row {b} X"
            valid = kv.valid[b].cpu().numpy().astype(bool)
            assert valid[:, :T].all() and not valid[:, T:].any(), f"layer {l} row {b} valid flags"
            for name, ref in (("K", caches[b].K), ("V", caches[b].V)):
                got = _np(getattr(kv, name)[b])[:, :T]
                acc = 4.0 * np.sqrt(w.d) * 2.0 ** -24 * np.abs(ref[:, :T]).max()
                assert within_ulp(got, ref[:, :T], dt, acc_floor=acc), f"layer {l} row {b} {name}"


def test_prefill_dense_two_rows_f16():
    """Two sequences (the batched tensor-core paths with every unit)."""
    w = Workload("prefill_b2", 35, d=256, h=4, d_h=64, N=512, r=64, dtype="f16", layers=2,
                 n_prompt=9, n_gen=1, head_pct=50, neuron_pct=10)
    _prefill_teacher_forced(w, B=2)


def test_prefill_dense_one_row_bf16_dh128():
    """One sequence, d_h = 128 (the batch-1 tensor-core projection with
    every head: 4 tiles x 3 and the KV append at each position)."""
    w = Workload("prefill_b1", 36, d=512, h=4, d_h=128, N=1024, r=64, dtype="bf16", layers=2,
                 n_prompt=12, n_gen=1, head_pct=50, neuron_pct=10)
    _prefill_teacher_forced(w, B=1)


def test_host_io_graph_matches_device_loop():
    """A host-driven token loop on a graph that carries its own copies
    (capture(host_io=...): pinned input -> residual, step, residual -> pinned
    output) gives bit for bit the tokens of the device-resident loop (batch 1:
    every output element has one writer and a fixed summation order)."""
    w = Workload("hostio_stack", 37, d=512, h=8, d_h=128, N=2048, r=128, dtype="f16", layers=3,
                 n_prompt=30, n_gen=5, head_pct=25, neuron_pct=5)
    dev = "cuda"
    layers = [layer_weights(w, l, device=dev) for l in range(w.layers)]
    n_max = ((w.n_prompt + 8 + 15) // 16) * 16
    scale = 1.0 / math.sqrt(w.d_h)
    Xp = [embeddings(w, w.n_prompt, f"X{l}", device=dev)[None] for l in range(w.layers)]
    r0 = residual_input(w, 1, "r0", device=dev)
    outs = []
    for host in (False, True):
        dec = SparseDecoder(layers, 1, n_max, w.k_heads, w.k_neurons, scale)
        dec.prefill(Xp, w.n_prompt)
        dec.r_stream.copy_(r0)
        dec.step_ops()  # layer 0's first token eagerly, as in the stack tests
        dv.dv_positions_advance(dec.pos, 0, n_max)
        seq = []
        if host:
            h_in = torch.empty((1, w.d), dtype=torch.float32, pin_memory=True)
            h_out = torch.empty((1, w.d), dtype=torch.float32, pin_memory=True)
            h_in.copy_(dec.r_stream.cpu())
            dec.capture(advance=(0, n_max), host_io=(h_in, h_out))
            for _ in range(4):
                dec.replay()
                torch.cuda.current_stream().synchronize()
                seq.append(h_out.clone())
                h_in.copy_(h_out)
        else:
            dec.capture(advance=(0, n_max))
            for _ in range(4):
                dec.replay()
                seq.append(dec.r_stream.cpu())
        dec.check()
        outs.append(seq)
    for t, (a, b) in enumerate(zip(*outs)):
        assert torch.equal(a, b), f"token {t}"

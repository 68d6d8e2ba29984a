"""Decoder stack driver: one decoded token through L sparse layers, with the
next layer's heads and neurons predicted on a side CUDA stream from the
current layer's attention input ("用Deja Vu来提高 LLM 的推理速度" §3.1, parallel
sparsity prediction; Deja Vu reading notes, "Reducing Overhead with
Asynchronous Execution").

Per layer l (main stream):
    y_a = LN(r)                      dv_layernorm
    (layer 0 only) S_A, S_M = predict(y_a)          dv_predict, synchronous
    wait for layer l's look-ahead sets (event)
    record "y_a of layer l ready"; side stream: dv_lookahead(y_a, P^{l+1})
    r += MHA_{S_A}(y_a)              dv_sparse_attn (append, repair, attend)
    y_m = LN(r);  r += MLP_{S_M}(y_m)    dv_layernorm, dv_sparse_mlp
The whole token (both streams) is captured once into a CUDA graph and
replayed.  This module only orders calls; every step runs in libdv's kernels.
"""

from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import binding as dv


class SparseDecoder:
    """Device state of an L-layer sparse decoder for a batch of B sequences.

    layers: per layer a dict of weight tensors in the library layouts
            (Wqkv, Wo, W1n, W2n, PA1t, PA2t, PM1t, PM2t), all of one dtype.
    trace:  keep a copy of the residual stream before layer 0 (r_in0) and
            after every block of every layer (r_mid[l] after the attention,
            r_out[l] after the MLP), so that each block can be checked on its
            own inputs (plain device copies between the calls).
    """

    def __init__(self, layers: List[Dict[str, torch.Tensor]], B: int, n_max: int,
                 k_heads: int, k_neurons: int, scale: float, eps: float = 1e-5,
                 trace: bool = False):
        W0 = layers[0]
        self.layers = layers
        self.L = len(layers)
        self.h, _, self.d_h, self.d = W0["Wqkv"].shape
        self.N = W0["W1n"].shape[0]
        self.r = W0["PM1t"].shape[0]
        self.B, self.n_max = B, n_max
        self.k_heads, self.k_neurons = k_heads, k_neurons
        self.scale, self.eps = float(scale), float(eps)
        self.dtype = W0["W1n"].dtype
        dev = W0["W1n"].device
        self.device = dev
        i32 = dict(dtype=torch.int32, device=dev)
        B, d = self.B, self.d
        self.kv = [dv.KV.empty(B, self.h, n_max, self.d_h, d, self.dtype, dev) for _ in layers]
        self.head_idx = [torch.zeros(B, k_heads, **i32) for _ in layers]
        self.head_cnt = [torch.zeros(B, **i32) for _ in layers]
        self.neur_idx = [torch.zeros(B, k_neurons, **i32) for _ in layers]
        self.neur_cnt = [torch.zeros(B, **i32) for _ in layers]
        self.y_a = [torch.zeros(B, d, dtype=self.dtype, device=dev) for _ in layers]
        self.y_m = [torch.zeros(B, d, dtype=self.dtype, device=dev) for _ in layers]
        self.r_stream = torch.zeros(B, d, dtype=torch.float32, device=dev)   # residual
        self.trace = bool(trace)
        if self.trace:
            f32 = dict(dtype=torch.float32, device=dev)
            self.r_in0 = torch.zeros(B, d, **f32)
            self.r_mid = [torch.zeros(B, d, **f32) for _ in layers]
            self.r_out = [torch.zeros(B, d, **f32) for _ in layers]
        self.pos = torch.zeros(B, **i32)
        self.ws_pred_main = dv.workspace(dv.dv_predict_workspace_size(B, 2, self.r, self.N), dev)
        self.ws_pred_side = dv.workspace(dv.dv_predict_workspace_size(B, 2, self.r, self.N), dev)
        self.ws_attn = dv.workspace(
            dv.dv_sparse_attn_workspace_size(B, d, self.h, self.d_h, k_heads, n_max), dev)
        self.ws_mlp = dv.workspace(dv.dv_sparse_mlp_workspace_size(B, d, self.N, k_neurons), dev)
        self.side = torch.cuda.Stream(device=dev)
        self.ev_y = [dv.make_event() for _ in layers]
        self.ev_pred = [dv.make_event() for _ in layers]
        torch.cuda.synchronize(dev)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        # optional timing of one kernel family inside the step (events recorded
        # around every call of it on the main stream)
        self.timed: Optional[str] = None
        self.t_ev: List[torch.cuda.Event] = []

    def set_keep(self, k_heads: int, k_neurons: int):
        """Change the number of heads and neurons kept per layer (new index
        lists and block workspaces; the KV caches are kept).  Re-capture
        the graph afterwards."""
        dev, B = self.device, self.B
        i32 = dict(dtype=torch.int32, device=dev)
        self.k_heads, self.k_neurons = k_heads, k_neurons
        self.head_idx = [torch.zeros(B, k_heads, **i32) for _ in self.layers]
        self.head_cnt = [torch.zeros(B, **i32) for _ in self.layers]
        self.neur_idx = [torch.zeros(B, k_neurons, **i32) for _ in self.layers]
        self.neur_cnt = [torch.zeros(B, **i32) for _ in self.layers]
        self.ws_attn = dv.workspace(
            dv.dv_sparse_attn_workspace_size(B, self.d, self.h, self.d_h, k_heads, self.n_max), dev)
        self.ws_mlp = dv.workspace(dv.dv_sparse_mlp_workspace_size(B, self.d, self.N, k_neurons), dev)
        self.graph = None

    # ------------------------------------------------------------------ pieces
    def predictors(self, l: int):
        W = self.layers[l]
        return [dv.Predictor(W["PA1t"], W["PA2t"], self.head_idx[l], self.head_cnt[l],
                             dv.DV_TOPK, self.k_heads),
                dv.Predictor(W["PM1t"], W["PM2t"], self.neur_idx[l], self.neur_cnt[l],
                             dv.DV_TOPK, self.k_neurons)]

    def prefill(self, X_prompt: List[torch.Tensor], n_prompt: int):
        """Synthetic prompt: X[b][0:n_prompt] = X_prompt[l] for every layer and
        K/V of every head computed from it (dv_kv_repair with all heads)."""
        all_heads = torch.arange(self.h, dtype=torch.int32, device=self.device).repeat(self.B, 1)
        cnt = torch.full((self.B,), self.h, dtype=torch.int32, device=self.device)
        pos = torch.full((self.B,), n_prompt, dtype=torch.int32, device=self.device)
        ws = dv.workspace(dv.dv_sparse_attn_workspace_size(self.B, self.d, self.h, self.d_h, self.h,
                                                           self.n_max), self.device)
        for l in range(self.L):
            kv = self.kv[l]
            kv.valid.zero_()
            kv.X[:, :n_prompt].copy_(X_prompt[l][:, :n_prompt])
            dv.dv_kv_repair(kv, self.layers[l]["Wqkv"], pos, all_heads, cnt, ws)
        self.pos.fill_(n_prompt)
        st, info = dv.dv_check(ws)
        if st != 0:
            raise dv.DvError(st, "prefill", f"info={info}")

    def _dense_ops(self):
        """One prompt position through every layer with all heads and all
        neurons selected (no predictor), on the current stream."""
        if self.trace:
            self.r_in0.copy_(self.r_stream)
        for l in range(self.L):
            W = self.layers[l]
            dv.dv_layernorm(self.r_stream, self.y_a[l], self.eps)
            dv.dv_sparse_attn(self.y_a[l], W["Wqkv"], W["Wo"], self.kv[l], self.pos,
                              self.head_idx[l], self.head_cnt[l], self.scale, self.r_stream,
                              self.ws_attn, accumulate=True)
            if self.trace:
                self.r_mid[l].copy_(self.r_stream)
            dv.dv_layernorm(self.r_stream, self.y_m[l], self.eps)
            dv.dv_sparse_mlp(self.y_m[l], W["W1n"], W["W2n"], self.neur_idx[l], self.neur_cnt[l],
                             self.r_stream, self.ws_mlp, accumulate=True)
            if self.trace:
                self.r_out[l].copy_(self.r_stream)

    def prefill_dense(self, E: torch.Tensor, n_prompt: int, on_position=None):
        """Dense causal prompt pass (Deja Vu reading notes, "Typical LLM
        procedure": the prompt runs through every layer, which builds each
        layer's KV cache; generation then goes token by token).  Positions
        0..n_prompt-1 in order, each through every layer with all heads and
        all neurons selected -- the decode step's own kernels with S = all,
        one CUDA graph replayed per position -- so position t attends over
        positions 0..t (causal attention) and every layer's X, K, V and valid
        flags below n_prompt are the model's own.  E [B][n_prompt][d] (fp32)
        is the residual stream entering layer 0.  Afterwards the decoder
        continues at n_prompt with its keep counts.  ``on_position(t)`` runs
        after position t (the tests read the traced activations there)."""
        keep = (self.k_heads, self.k_neurons)
        dev, B = self.device, self.B
        if n_prompt > self.n_max:
            raise ValueError("prompt longer than the cache")
        self.set_keep(self.h, self.N)
        heads = torch.arange(self.h, dtype=torch.int32, device=dev).repeat(B, 1)
        neurons = torch.arange(self.N, dtype=torch.int32, device=dev).repeat(B, 1)
        for l in range(self.L):
            self.kv[l].valid.zero_()
            self.head_idx[l].copy_(heads)
            self.head_cnt[l].fill_(self.h)
            self.neur_idx[l].copy_(neurons)
            self.neur_cnt[l].fill_(self.N)
        self.pos.zero_()
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        # every attention / MLP call follows the layernorm that produces its
        # input and no predictor runs: launch overlap holds for all of them
        prev = dv.dv_set_launch_overlap(1)
        try:
            with torch.cuda.stream(s):
                with torch.cuda.graph(graph, stream=s):
                    self._dense_ops()
                    dv.dv_positions_advance(self.pos, 0, self.n_max)
        finally:
            dv.dv_set_launch_overlap(prev)
        torch.cuda.current_stream().wait_stream(s)
        for t in range(n_prompt):
            self.r_stream.copy_(E[:, t])
            graph.replay()
            if on_position is not None:
                on_position(t)
        self.check()
        self.set_keep(*keep)

    def _time(self, kind: str, stream=None):
        """Record a timing event (kept in self.t_ev) when timing ``kind``.
        Events are 'external' so that they are real event records inside a
        captured graph."""
        if self.timed != kind:
            return
        try:
            ev = torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:  # older torch: events still work outside graphs
            ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream if stream is not None else torch.cuda.current_stream())
        self.t_ev.append(ev)

    def step_ops(self):
        """Enqueue one token on the current stream (+ the side stream)."""
        # Every attention / MLP call here directly follows the layernorm that
        # produces its input, except layer 0's attention (after its predictor
        # on the same stream): launch overlap is on for all the others.
        prev = dv.dv_set_launch_overlap(1)
        try:
            self._step_ops()
        finally:
            dv.dv_set_launch_overlap(prev)

    def _step_ops(self):
        main = torch.cuda.current_stream()
        if self.trace:
            self.r_in0.copy_(self.r_stream)
        for l in range(self.L):
            W = self.layers[l]
            self._time("ln")
            dv.dv_layernorm(self.r_stream, self.y_a[l], self.eps)
            self._time("ln")
            if l == 0:
                self._time("predict")
                dv.dv_predict(self.y_a[0], self.predictors(0), self.ws_pred_main)
                self._time("predict")
            else:
                main.wait_event(self.ev_pred[l])
            if l + 1 < self.L:
                self.ev_y[l].record(main)
                if self.timed == "predict":
                    # dv_lookahead spelled out so the timing events bracket
                    # only the predictor kernels on the side stream
                    self.side.wait_event(self.ev_y[l])
                    self._time("predict", self.side)
                    dv.dv_predict(self.y_a[l], self.predictors(l + 1), self.ws_pred_side,
                                  stream=self.side)
                    self._time("predict", self.side)
                    self.ev_pred[l + 1].record(self.side)
                else:
                    dv.dv_lookahead(self.y_a[l], self.predictors(l + 1), self.ws_pred_side,
                                    self.ev_y[l], self.side, self.ev_pred[l + 1])
            self._time("attn")
            if l == 0:
                dv.dv_set_launch_overlap(0)  # the predictor just wrote this call's head list
            dv.dv_sparse_attn(self.y_a[l], W["Wqkv"], W["Wo"], self.kv[l], self.pos,
                              self.head_idx[l], self.head_cnt[l], self.scale, self.r_stream,
                              self.ws_attn, accumulate=True)
            dv.dv_set_launch_overlap(1)
            self._time("attn")
            if self.trace:
                self.r_mid[l].copy_(self.r_stream)
            self._time("ln")
            dv.dv_layernorm(self.r_stream, self.y_m[l], self.eps)
            self._time("ln")
            self._time("mlp")
            dv.dv_sparse_mlp(self.y_m[l], W["W1n"], W["W2n"], self.neur_idx[l], self.neur_cnt[l],
                             self.r_stream, self.ws_mlp, accumulate=True)
            self._time("mlp")
            if self.trace:
                self.r_out[l].copy_(self.r_stream)

    def capture(self, advance: Optional[tuple] = None, host_io: Optional[tuple] = None):
        """Capture one token (optionally followed by pos advance (lo, hi))
        into a CUDA graph.  host_io = (h_in, h_out), pinned host tensors of
        the residual's shape: the graph then starts with the copy of h_in
        into the residual stream and ends with the copy of the result into
        h_out, so a host-driven loop costs one graph launch per token."""
        self.graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        if host_io is not None:
            for t in host_io:
                if t.device.type != "cpu" or not t.is_pinned() or t.shape != self.r_stream.shape \
                        or t.dtype != self.r_stream.dtype:
                    raise ValueError("host_io: pinned host fp32 tensors of the residual's shape")
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                if host_io is not None:
                    self.r_stream.copy_(host_io[0], non_blocking=True)
                self.step_ops()
                if advance is not None:
                    dv.dv_positions_advance(self.pos, advance[0], advance[1])
                if host_io is not None:
                    host_io[1].copy_(self.r_stream, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s)

    def replay(self):
        self.graph.replay()

    def check(self):
        for ws in (self.ws_pred_main, self.ws_pred_side, self.ws_attn, self.ws_mlp):
            st, info = dv.dv_check(ws)
            if st != 0:
                raise dv.DvError(st, "decode step", f"info={info}")

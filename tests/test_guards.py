"""Guard regions around every buffer the library writes.

Race and bounds detection without a sanitizer: each output, index list,
score row, KV-cache tensor and workspace is the middle of a larger
allocation whose two ends hold a sentinel pattern.  After the calls of a
decode loop (batch 1, the batched tensor-core paths, the streaming paths
for long selections, the predictor, the selection and the labeller) every
sentinel must be intact, so no kernel wrote outside its buffer.  The
results themselves are checked against the oracle by the parity tests; here
only the byte ranges matter.
"""

import math

import pytest
import torch

from contextual_sparsity_decode_gb300 import binding as dv
from synth import draw

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096  # each side; keeps the guarded view 256-byte aligned


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD_BYTES of sentinel on
    both sides."""

    def __init__(self, shape, dtype, fill=0, device="cuda"):
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esize
        n = math.prod(shape)
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device=device)
        if dtype == torch.uint8:
            self.sentinel = 0xA5
        elif dtype == torch.int32:
            self.sentinel = -777
        else:
            self.sentinel = 3.0
        self.buf.fill_(self.sentinel)
        self.t = self.buf[self.g: self.g + n].view(shape)
        self.t.fill_(fill)

    def intact(self) -> bool:
        lo, hi = self.buf[: self.g], self.buf[-self.g:]
        return bool((lo == self.sentinel).all()) and bool((hi == self.sentinel).all())


def _ws(nbytes):
    w = Guarded((max(int(nbytes), 256),), torch.uint8)
    dv.dv_workspace_init(w.t)
    return w


def _kv(B, h, n_max, d_h, d, dtype):
    parts = [Guarded((B, h, n_max, d_h), dtype), Guarded((B, h, n_max, d_h), dtype),
             Guarded((B, n_max, d), dtype), Guarded((B, h, n_max), torch.uint8)]
    return dv.KV(*(p.t for p in parts)), parts


def _all_intact(items, what):
    for i, it in enumerate(items):
        assert it.intact(), f"{what}: buffer {i} written outside its range"


@pytest.mark.parametrize("B,d,h,d_h,k,n_prompt,dt", [
    (1, 512, 8, 128, 3, 40, torch.float16),    # batch-1 tensor-core projection
    (1, 256, 6, 64, 2, 37, torch.float16),     # CUDA-core projection
    (5, 512, 8, 128, 3, 30, torch.bfloat16),   # batched tensor-core attention
    (1, 12288, 24, 128, 16, 20, torch.float16),  # streaming output projection (>= 48 MB)
])
def test_attention_writes_stay_in_bounds(B, d, h, d_h, k, n_prompt, dt):
    dev = "cuda"
    name = f"guard_attn_{B}_{d}_{h}"
    sdt = "f16" if dt == torch.float16 else "bf16"
    Wqkv = draw((h, 3, d_h, d), d ** -0.5, 401, name + "/Wqkv", sdt).to(dev)
    Wo = draw((h, d_h, d), d ** -0.5, 401, name + "/Wo", sdt).to(dev)
    n_max = ((n_prompt + 8 + 15) // 16) * 16
    kv, kv_parts = _kv(B, h, n_max, d_h, d, dt)
    kv.X[:, :n_prompt].copy_(draw((B, n_prompt, d), 1.0, 401, name + "/X", sdt).to(dev))
    pos = torch.full((B,), n_prompt, dtype=torch.int32, device=dev)
    ws_fill = _ws(dv.dv_sparse_attn_workspace_size(B, d, h, d_h, h, n_max))
    all_heads = torch.arange(h, dtype=torch.int32, device=dev).repeat(B, 1)
    dv.dv_kv_repair(kv, Wqkv, pos, all_heads, torch.full((B,), h, dtype=torch.int32, device=dev), ws_fill.t)
    assert dv.dv_check(ws_fill.t)[0] == 0
    ws = _ws(dv.dv_sparse_attn_workspace_size(B, d, h, d_h, k, n_max))
    idx = Guarded((B, k), torch.int32)
    cnt = Guarded((B,), torch.int32)
    out = Guarded((B, d), torch.float32)
    g = torch.Generator().manual_seed(B * 1000 + d)
    for step in range(4):
        for b in range(B):
            idx.t[b] = torch.sort(torch.randperm(h, generator=g)[:k]).values.to(torch.int32).to(dev)
        cnt.t.fill_(k)
        y = draw((B, d), 1.0, 401, f"{name}/y{step}", sdt).to(dev)
        dv.dv_sparse_attn(y, Wqkv, Wo, kv, pos, idx.t, cnt.t, 1.0 / math.sqrt(d_h), out.t, ws.t, accumulate=True)
        assert dv.dv_check(ws.t)[0] == 0
        pos += 1
    _all_intact(kv_parts + [ws_fill, ws, idx, cnt, out], "attention")


@pytest.mark.parametrize("B,d,N,k,dt", [
    (1, 512, 2048, 100, torch.float16),     # one-launch MLP
    (4, 512, 2048, 100, torch.bfloat16),    # tensor-core union
    (3, 256, 1024, 37, torch.float32),      # CUDA-core union
    (1, 12288, 4096, 2048, torch.float16),  # streaming MLP (>= 96 MB of selected rows)
])
def test_mlp_writes_stay_in_bounds(B, d, N, k, dt):
    dev = "cuda"
    sdt = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[dt]
    name = f"guard_mlp_{B}_{d}_{N}"
    W1n = draw((N, d), d ** -0.5, 402, name + "/W1", sdt).to(dev)
    W2n = draw((N, d), d ** -0.5, 402, name + "/W2", sdt).to(dev)
    ws = _ws(dv.dv_sparse_mlp_workspace_size(B, d, N, k))
    idx = Guarded((B, k), torch.int32)
    cnt = Guarded((B,), torch.int32)
    out = Guarded((B, d), torch.float32)
    g = torch.Generator().manual_seed(B * 77 + N)
    for step in range(3):
        for b in range(B):
            kk = k - (b % 3)  # ragged counts
            idx.t[b, :kk] = torch.sort(torch.randperm(N, generator=g)[:kk]).values.to(torch.int32).to(dev)
            cnt.t[b] = kk
        y = draw((B, d), 1.0, 402, f"{name}/y{step}", sdt).to(dev)
        dv.dv_sparse_mlp(y, W1n, W2n, idx.t, cnt.t, out.t, ws.t, accumulate=step > 0)
        assert dv.dv_check(ws.t)[0] == 0
    _all_intact([ws, idx, cnt, out], "mlp")


@pytest.mark.parametrize("B", [1, 3, 16])
def test_predictor_and_selection_writes_stay_in_bounds(B):
    dev = "cuda"
    d, r, NA, NM = 1024, 256, 40, 8192
    name = f"guard_pred_{B}"
    y = draw((B, d), 1.0, 403, name + "/y", "f16").to(dev)
    PA1 = draw((r, d), d ** -0.5, 403, name + "/PA1", "f16").to(dev)
    PA2 = draw((NA, r), r ** -0.5, 403, name + "/PA2", "f16").to(dev)
    PM1 = draw((r, d), d ** -0.5, 403, name + "/PM1", "f16").to(dev)
    PM2 = draw((NM, r), r ** -0.5, 403, name + "/PM2", "f16").to(dev)
    outs = []
    preds = []
    for P1, P2, mode, k in ((PA1, PA2, dv.DV_TOPK, 8), (PM1, PM2, dv.DV_THRESHOLD, 0)):
        N = P2.shape[0]
        cap = N if mode == dv.DV_THRESHOLD else k
        idx, cnt, sc = Guarded((B, cap), torch.int32, -1), Guarded((B,), torch.int32), Guarded((B, N), torch.float32)
        preds.append(dv.Predictor(P1, P2, idx.t, cnt.t, mode, k, 0.5, sc.t))
        outs += [idx, cnt, sc]
    ws = _ws(dv.dv_predict_workspace_size(B, 2, r, NM))
    dv.dv_predict(y, preds, ws.t)
    assert dv.dv_check(ws.t)[0] == 0
    # the selection alone on the scores just written
    sidx, scnt = Guarded((B, 500), torch.int32, -1), Guarded((B,), torch.int32)
    ws2 = _ws(256)
    dv.dv_select_scores(preds[1].scores, dv.DV_TOPK, 500, 0.0, sidx.t, scnt.t, ws2.t)
    assert dv.dv_check(ws2.t)[0] == 0
    _all_intact(outs + [ws, sidx, scnt, ws2], "predictor / selection")


def test_labeller_writes_stay_in_bounds():
    dev = "cuda"
    T, d, N, h, d_h = 300, 512, 1000, 4, 128
    X = draw((T, d), 1.0, 404, "guard_label/X", "bf16").to(dev)
    W1n = draw((N, d), d ** -0.5, 404, "guard_label/W1", "bf16").to(dev)
    Wqkv = draw((h, 3, d_h, d), d ** -0.5, 404, "guard_label/Wqkv", "bf16").to(dev)
    nn, hn = Guarded((N,), torch.float32), Guarded((h,), torch.float32)
    ws = _ws(dv.dv_label_workspace_size(T, d, N, h, d_h))
    dv.dv_label_neurons(X, W1n, nn.t, ws.t)
    dv.dv_label_heads(X, Wqkv, 1.0 / math.sqrt(d_h), hn.t, ws.t)
    assert dv.dv_check(ws.t)[0] == 0
    _all_intact([nn, hn, ws], "labeller")

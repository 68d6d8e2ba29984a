"""dv_predict_static -- the predictor entry point that allocates nothing --
against dv_predict, through the C ABI, on two calls in a row.

Callers that cannot allocate device memory (a plugin whose host engine owns
all device allocations, or a loop where a cudaMalloc could stall the device)
use dv_predict_static, whose scratch is a fixed array inside the library.
This file is collected last so that a failure here leaves every other test
already run; it also passes on its own in a fresh process, where its first
call performs the per-device set-up.
"""

import numpy as np
import pytest
import torch

from contextual_sparsity_decode_gb300 import binding as dv
from synth import draw

pytestmark = pytest.mark.gpu


def _preds(B, PA1, PA2, PM1, PM2, kA, kM, dev, with_scores=True):
    outs = []
    preds = []
    for P1, P2, k in ((PA1, PA2, kA), (PM1, PM2, kM)):
        idx = torch.full((B, k), -3, dtype=torch.int32, device=dev)
        cnt = torch.full((B,), -1, dtype=torch.int32, device=dev)
        sc = torch.zeros((B, P2.shape[0]), dtype=torch.float32, device=dev) if with_scores else None
        preds.append(dv.Predictor(P1, P2, idx, cnt, dv.DV_TOPK, k, 0.5, sc))
        outs.append((idx, cnt, sc))
    return preds, outs


def test_predict_static_matches_predict_twice():
    dev = "cuda"
    B, d, r, h, N = 2, 2048, 1024, 32, 8192
    kA, kM = 7, 410
    PA1 = draw((r, d), d ** -0.5, 401, "PA1", "f16").to(dev)
    PA2 = draw((h, r), r ** -0.5, 401, "PA2", "f16").to(dev)
    PM1 = draw((r, d), d ** -0.5, 401, "PM1", "f16").to(dev)
    PM2 = draw((N, r), r ** -0.5, 401, "PM2", "f16").to(dev)
    ws = dv.workspace(dv.dv_predict_workspace_size(B, 2, r, N))
    # the second call leaves the score outputs NULL, so the scores live in
    # the library's own array between the two GEMVs and the selection
    for call in range(2):
        y = draw((B, d), 1.0, 401, f"y{call}", "f16").to(dev)
        ref_p, ref_o = _preds(B, PA1, PA2, PM1, PM2, kA, kM, dev)
        dv.dv_predict(y, ref_p, ws)
        assert dv.dv_check(ws)[0] == 0
        new_p, new_o = _preds(B, PA1, PA2, PM1, PM2, kA, kM, dev, with_scores=call == 0)
        dv.dv_predict_static(y, new_p)
        torch.cuda.synchronize()
        for (i0, c0, s0), (i1, c1, s1) in zip(ref_o, new_o):
            assert torch.equal(c0, c1)
            assert torch.equal(i0, i1)
            if s1 is not None:
                assert float((s0 - s1).abs().max()) <= 1e-5


def test_predict_static_rejects_shapes_beyond_its_array():
    dev = "cuda"
    B, d, r, N = 1, 256, 64, 40000   # N above the static limit
    P1 = torch.zeros((r, d), dtype=torch.float16, device=dev)
    P2 = torch.zeros((N, r), dtype=torch.float16, device=dev)
    idx = torch.zeros((B, 8), dtype=torch.int32, device=dev)
    cnt = torch.zeros((B,), dtype=torch.int32, device=dev)
    y = torch.zeros((B, d), dtype=torch.float16, device=dev)
    with pytest.raises(dv.DvError) as e:
        dv.dv_predict_static(y, [dv.Predictor(P1, P2, idx, cnt, dv.DV_TOPK, 8)])
    assert e.value.status == 3

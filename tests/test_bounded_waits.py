"""Device-side bounded waits run out, report DV_ERR_TIMEOUT, and leave the
GPU context and the workspace usable.

The failure is made on the host, never by a fault: a workspace whose arrival
counter was never zero-filled (so the up-projection CTAs of the one-launch
MLP can never bring it to its target), or a wait limit so short
(dv_set_wait_limit_ns) that the tensor-core pipeline's first waits give up
before the copies they wait for have landed.  Each kernel still waits for
its own copies and tensor-core work before it exits.  The call after the
failed one must match the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_decode_gb300 import binding as dv
from dvtest import assert_rel_l2, f64
from synth import draw

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _mlp_case(tag, B, d, N, k, dtype, wid=211):
    W1n = draw((N, d), 0.02, wid, tag + "/W1", dtype)
    W2n = draw((N, d), 0.02, wid, tag + "/W2", dtype)
    y = draw((B, d), 1.0, wid, tag + "/y", dtype)
    g = torch.Generator().manual_seed(5)
    sets = [torch.sort(torch.randperm(N, generator=g)[:k]).values.to(torch.int32) for _ in range(B)]
    idx = torch.stack(sets)
    cnt = torch.full((B,), k, dtype=torch.int32)
    dev = "cuda"
    return (W1n, W2n, y, sets, W1n.to(dev), W2n.to(dev), y.to(dev), idx.to(dev), cnt.to(dev))


def _ref(W1n, W2n, y, sets):
    return oracle.sparse_mlp_batched(f64(y), f64(W1n), f64(W2n), [s.numpy() for s in sets])


@pytest.fixture
def short_wait():
    prev = dv.dv_set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        yield
    finally:
        dv.dv_set_wait_limit_ns(prev)


def test_wait_limit_setting_round_trips():
    prev = dv.dv_set_wait_limit_ns(12345)
    try:
        assert dv.dv_set_wait_limit_ns(0) == 12345     # 0 restores the default
        assert dv.dv_set_wait_limit_ns(-7) == 1_000_000_000
    finally:
        dv.dv_set_wait_limit_ns(prev)


def test_fused_mlp_wait_times_out_on_unzeroed_workspace(short_wait):
    """OPT-13B-shaped batch-1 MLP (one launch).  Every workspace byte past the
    error header is 0xff, so the arrival counter starts at -1 and the nA
    arrivals reach nA - 1 only: the down-projection CTAs' wait gives up."""
    W1n, W2n, y, sets, W1d, W2d, yd, idx, cnt = _mlp_case("tmo13b", 1, 5120, 20480, 1024, "f16")
    nbytes = dv.dv_sparse_mlp_workspace_size(1, 5120, 20480, 1024)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0
    out = torch.zeros(1, 5120, device="cuda")
    dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
    st, info = dv.dv_check(ws)
    assert st == TIMEOUT, (st, info)
    # zero-filled again, the same workspace serves a correct call
    dv.dv_workspace_init(ws)
    dv.dv_set_wait_limit_ns(0)
    out.zero_()
    dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
    assert dv.dv_check(ws) == (0, 0)
    assert_rel_l2(f64(out)[0], _ref(W1n, W2n, y, sets)[0], "f16", "after re-init")


def test_fused_mlp_recovers_after_a_wait_that_gave_up_early():
    """A 1 ns limit makes the down-projection CTAs give up before the
    up-projection CTAs arrive (whether they do depends on timing, so either
    status is accepted).  The late arrivals must still bring the counters
    back to zero: the next calls on the same workspace, with the normal
    limit, match the oracle."""
    W1n, W2n, y, sets, W1d, W2d, yd, idx, cnt = _mlp_case("late13b", 1, 5120, 20480, 1024, "f16")
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(1, 5120, 20480, 1024))
    out = torch.zeros(1, 5120, device="cuda")
    prev = dv.dv_set_wait_limit_ns(1)
    try:
        dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
        st, _ = dv.dv_check(ws)
    finally:
        dv.dv_set_wait_limit_ns(prev)
    assert st in (0, TIMEOUT)
    ref = _ref(W1n, W2n, y, sets)[0]
    for _ in range(2):
        out.zero_()
        dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
        assert dv.dv_check(ws) == (0, 0)
        assert_rel_l2(f64(out)[0], ref, "f16", "after an early give-up")


@pytest.mark.tc
def test_tensor_core_pipeline_waits_time_out_and_unwind():
    """Batch 16 (tcgen05 path) with a 1 ns pipeline limit: the TMA producer
    and MMA issuer give up at their first waits and report DV_ERR_TIMEOUT;
    each CTA still waits (at least two seconds) for the copies and MMAs it
    started before freeing its tensor memory.  With the limit restored the
    next call matches the oracle."""
    W1n, W2n, y, sets, W1d, W2d, yd, idx, cnt = _mlp_case("tmotc", 16, 2048, 8192, 410, "f16")
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(16, 2048, 8192, 410))
    out = torch.zeros(16, 2048, device="cuda")
    prev = dv.dv_set_wait_limit_ns(1)
    statuses = []
    try:
        for _ in range(3):
            dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
            statuses.append(dv.dv_check(ws)[0])
            if statuses[-1] == TIMEOUT:
                break
    finally:
        dv.dv_set_wait_limit_ns(prev)
    assert TIMEOUT in statuses and set(statuses) <= {0, TIMEOUT}, statuses
    out.zero_()
    dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
    assert dv.dv_check(ws) == (0, 0)
    ref = _ref(W1n, W2n, y, sets)
    for b in range(16):
        assert_rel_l2(f64(out)[b], ref[b], "f16", f"row {b} after the timed-out call")


def test_streaming_mlp_recovers_after_a_short_wait_limit():
    """The streaming batch-1 MLP pass (selected rows >= 96 MB) under a 1 ns
    limit.  Its bulk copies usually land inside the hardware's own suspend
    window of mbarrier.try_wait, so whether a wait gives up depends on
    timing and either status is accepted; a CTA that gives up still waits
    for the copies it issued.  The next calls, with the normal limit, match
    the oracle."""
    W1n, W2n, y, sets, W1d, W2d, yd, idx, cnt = _mlp_case("tmostrm", 1, 12288, 49152, 2458, "f16")
    ws = dv.workspace(dv.dv_sparse_mlp_workspace_size(1, 12288, 49152, 2458))
    out = torch.zeros(1, 12288, device="cuda")
    prev = dv.dv_set_wait_limit_ns(1)
    statuses = []
    try:
        for _ in range(3):
            dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
            statuses.append(dv.dv_check(ws)[0])
    finally:
        dv.dv_set_wait_limit_ns(prev)
    assert set(statuses) <= {0, TIMEOUT}, statuses
    ref = _ref(W1n, W2n, y, sets)[0]
    for _ in range(2):
        out.zero_()
        dv.dv_sparse_mlp(yd, W1d, W2d, idx, cnt, out, ws)
        assert dv.dv_check(ws) == (0, 0)
        assert_rel_l2(f64(out)[0], ref, "f16", "after the short-limit calls")

"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point that include/dv.h declares, answers
workspace queries, and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import pytest

from contextual_sparsity_decode_gb300 import binding as dv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = dv.lib()
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dv.EXPORTS)


def test_version_and_status_strings():
    assert dv.dv_version() >= 100
    assert dv.dv_status_str(0) == "ok"
    for st in range(1, 10):
        assert dv.dv_status_str(st) not in ("", "unknown status")
    assert dv.dv_status_str(99) == "unknown status"


def test_workspace_sizes():
    a = dv.dv_predict_workspace_size(1, 2, 1024, 20480)
    b = dv.dv_predict_workspace_size(4, 2, 1024, 20480)
    assert 0 < a < b
    assert dv.dv_sparse_mlp_workspace_size(1, 5120, 20480, 1024) > 0
    s1 = dv.dv_sparse_attn_workspace_size(1, 5120, 40, 128, 8, 1152)
    s2 = dv.dv_sparse_attn_workspace_size(1, 5120, 40, 128, 16, 1152)
    assert 0 < s1 < s2   # grows with the selected heads (per-head q and H)
    # the split-KV partials live in shared memory: no dependence on n_max
    assert dv.dv_sparse_attn_workspace_size(1, 5120, 40, 128, 8, 2304) == s1
    with pytest.raises(dv.DvError) as e:
        dv.dv_predict_workspace_size(0, 2, 1024, 20480)
    assert e.value.status == 1


def _vp(x):
    return ctypes.c_void_p(x)


def test_null_and_misaligned_arguments_rejected_on_host():
    lib = dv.lib()
    fake = 1 << 20  # never dereferenced: validation fails first
    s = _vp(0)
    # dv_sparse_mlp: null y
    st = lib.dv_sparse_mlp(None, 1, 64, 128, _vp(fake), _vp(fake), _vp(fake), 8, _vp(fake), 1,
                           _vp(fake), 0, _vp(fake), 1 << 20, s)
    assert st == 1
    # misaligned weight pointer
    st = lib.dv_sparse_mlp(_vp(fake), 1, 64, 128, _vp(fake + 2), _vp(fake), _vp(fake), 8, _vp(fake),
                           1, _vp(fake), 0, _vp(fake), 1 << 20, s)
    assert st == 1
    # bad dtype
    st = lib.dv_sparse_mlp(_vp(fake), 1, 64, 128, _vp(fake), _vp(fake), _vp(fake), 8, _vp(fake), 7,
                           _vp(fake), 0, _vp(fake), 1 << 20, s)
    assert st == 2
    # d not a multiple of the 16-byte vector
    st = lib.dv_sparse_mlp(_vp(fake), 1, 60, 128, _vp(fake), _vp(fake), _vp(fake), 8, _vp(fake), 1,
                           _vp(fake), 0, _vp(fake), 1 << 20, s)
    assert st == 1
    # batch too large
    st = lib.dv_sparse_mlp(_vp(fake), 33, 64, 128, _vp(fake), _vp(fake), _vp(fake), 8, _vp(fake), 1,
                           _vp(fake), 0, _vp(fake), 1 << 20, s)
    assert st == 1
    # workspace too small
    st = lib.dv_sparse_mlp(_vp(fake), 1, 64, 128, _vp(fake), _vp(fake), _vp(fake), 8, _vp(fake), 1,
                           _vp(fake), 0, _vp(fake), 16, s)
    assert st == 3


def test_predictor_arguments_rejected_on_host():
    lib = dv.lib()
    fake = 1 << 20
    p = dv.dv_predictor(fake, fake, 64, 100, dv.DV_TOPK, 10, 0.5, fake, 8, fake, None)
    # k > cap
    st = lib.dv_predict(_vp(fake), 1, 64, dv.DV_F16, ctypes.byref(p), 1, _vp(fake), 1 << 24, _vp(0))
    assert st == 1
    p.cap = 16
    p.r = 60  # not a multiple of 8 halves
    st = lib.dv_predict(_vp(fake), 1, 64, dv.DV_F16, ctypes.byref(p), 1, _vp(fake), 1 << 24, _vp(0))
    assert st == 1
    p.r = 64
    p.N = 100000  # beyond the selection limit
    st = lib.dv_predict(_vp(fake), 1, 64, dv.DV_F16, ctypes.byref(p), 1, _vp(fake), 1 << 24, _vp(0))
    assert st == 1
    p.N = 100
    st = lib.dv_predict(_vp(fake), 1, 64, dv.DV_F16, ctypes.byref(p), 3, _vp(fake), 1 << 24, _vp(0))
    assert st == 1  # more than two predictors


def test_attention_arguments_rejected_on_host():
    lib = dv.lib()
    fake = 1 << 20
    kv = dv.dv_kv(fake, fake, fake, fake, 64)
    args = lambda d_h, cap, nmax: (_vp(fake), 1, 256, 8, d_h, _vp(fake), _vp(fake),
                                   ctypes.byref(dv.dv_kv(fake, fake, fake, fake, nmax)), _vp(fake),
                                   _vp(fake), cap, _vp(fake), 1.0, dv.DV_F16, _vp(fake), 0,
                                   _vp(fake), 1 << 26, _vp(0))
    assert lib.dv_sparse_attn(*args(96, 4, 64)) == 7   # head dim unsupported
    assert lib.dv_sparse_attn(*args(64, 9, 64)) == 1   # cap > h
    assert lib.dv_sparse_attn(*args(64, 4, 40)) == 1   # n_max not a multiple of 16
    st = lib.dv_kv_repair(ctypes.byref(kv), 1, 256, 8, 64, None, _vp(fake), _vp(fake), 4, _vp(fake),
                          dv.DV_F16, _vp(fake), 1 << 26, _vp(0))
    assert st == 1
    assert lib.dv_layernorm(None, 1, 64, 1e-5, _vp(fake), dv.DV_F16, _vp(0)) == 1
    assert lib.dv_positions_advance(_vp(fake), 1, 5, 5, _vp(0)) == 1


def test_launch_overlap_policy_round_trips():
    """The launch policy is a host-side setting: it returns the previous level
    and clamps to {0, 1}."""
    prev = dv.dv_set_launch_overlap(1)
    try:
        assert dv.dv_set_launch_overlap(5) == 1
        assert dv.dv_set_launch_overlap(0) == 1
        assert dv.dv_set_launch_overlap(-3) == 0
    finally:
        dv.dv_set_launch_overlap(prev)

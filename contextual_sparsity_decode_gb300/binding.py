"""Thin ctypes binding of libdv (include/dv.h).

Each ``dv_*`` function here has the name of the C entry point it calls and
only marshals arguments: it takes torch CUDA tensors (PyTorch is used for
device memory and streams), derives sizes from their shapes, passes raw
pointers and the stream handle, and raises ``DvError`` on a non-OK status.
All computation happens in the library's CUDA kernels.  There is no
fallback: if libdv.so cannot be built or loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from . import build as _build

DV_F32, DV_F16, DV_BF16 = 0, 1, 2
DV_TOPK, DV_THRESHOLD = 0, 1

STATUS = {
    0: "DV_OK", 1: "DV_ERR_INVALID_ARG", 2: "DV_ERR_DTYPE", 3: "DV_ERR_WORKSPACE",
    4: "DV_ERR_CUDA", 5: "DV_ERR_INDEX_RANGE", 6: "DV_ERR_TIMEOUT", 7: "DV_ERR_UNSUPPORTED",
    8: "DV_ERR_CAPACITY", 9: "DV_ERR_POSITION",
}

_DT = {torch.float32: DV_F32, torch.float16: DV_F16, torch.bfloat16: DV_BF16}

# every entry point declared in include/dv.h
EXPORTS = (
    "dv_status_str", "dv_last_cuda_error", "dv_version", "dv_workspace_init", "dv_check",
    "dv_predict_workspace_size", "dv_predict", "dv_lookahead", "dv_predict_static",
    "dv_sparse_mlp_workspace_size", "dv_sparse_mlp",
    "dv_sparse_attn_workspace_size", "dv_sparse_attn", "dv_kv_repair",
    "dv_layernorm", "dv_positions_advance", "dv_set_launch_overlap", "dv_set_wait_limit_ns",
    "dv_kernel_launches", "dv_label_workspace_size", "dv_label_neurons", "dv_label_heads",
    "dv_select_scores",
)


class DvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} {detail}".rstrip())


class dv_predictor(ctypes.Structure):
    _fields_ = [("P1t", ctypes.c_void_p), ("P2t", ctypes.c_void_p), ("r", ctypes.c_int),
                ("N", ctypes.c_int), ("mode", ctypes.c_int), ("k", ctypes.c_int),
                ("t", ctypes.c_float), ("idx", ctypes.c_void_p), ("cap", ctypes.c_int),
                ("count", ctypes.c_void_p), ("scores", ctypes.c_void_p)]


class dv_kv(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("X", ctypes.c_void_p),
                ("valid", ctypes.c_void_p), ("n_max", ctypes.c_int)]


_lib = None
_lock = threading.Lock()

_c_int, _c_float, _vp, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_SIGS = {
    "dv_status_str": ([_c_int], ctypes.c_char_p),
    "dv_last_cuda_error": ([], _c_int),
    "dv_version": ([], _c_int),
    "dv_workspace_init": ([_vp, _sz, _vp], _c_int),
    "dv_check": ([_vp, _vp, ctypes.POINTER(_c_int)], _c_int),
    "dv_predict_workspace_size": ([_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_sz)], _c_int),
    "dv_predict": ([_vp, _c_int, _c_int, _c_int, ctypes.POINTER(dv_predictor), _c_int, _vp, _sz, _vp],
                   _c_int),
    "dv_lookahead": ([_vp, _c_int, _c_int, _c_int, ctypes.POINTER(dv_predictor), _c_int, _vp, _sz,
                      _vp, _vp, _vp], _c_int),
    "dv_predict_static": ([_vp, _c_int, _c_int, _c_int, ctypes.POINTER(dv_predictor), _c_int, _vp],
                          _c_int),
    "dv_sparse_mlp_workspace_size": ([_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_sz)], _c_int),
    "dv_sparse_mlp": ([_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp, _c_int,
                       _vp, _sz, _vp], _c_int),
    "dv_sparse_attn_workspace_size": ([_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       ctypes.POINTER(_sz)], _c_int),
    "dv_sparse_attn": ([_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, ctypes.POINTER(dv_kv), _vp,
                        _vp, _c_int, _vp, _c_float, _c_int, _vp, _c_int, _vp, _sz, _vp], _c_int),
    "dv_kv_repair": ([ctypes.POINTER(dv_kv), _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_int,
                      _vp, _c_int, _vp, _sz, _vp], _c_int),
    "dv_layernorm": ([_vp, _c_int, _c_int, _c_float, _vp, _c_int, _vp], _c_int),
    "dv_positions_advance": ([_vp, _c_int, _c_int, _c_int, _vp], _c_int),
    "dv_set_launch_overlap": ([_c_int], _c_int),
    "dv_set_wait_limit_ns": ([ctypes.c_longlong], ctypes.c_longlong),
    "dv_kernel_launches": ([], ctypes.c_longlong),
    "dv_label_workspace_size": ([_c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_sz)], _c_int),
    "dv_label_neurons": ([_vp, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _sz, _vp], _c_int),
    "dv_label_heads": ([_vp, _c_int, _c_int, _c_int, _c_int, _vp, _c_float, _c_int, _vp, _vp, _sz, _vp],
                       _c_int),
    "dv_select_scores": ([_vp, _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _c_int, _vp, _vp, _sz, _vp],
                         _c_int),
}


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libdv.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    h = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(h)


def _event(ev) -> ctypes.c_void_p:
    if ev is None:
        return ctypes.c_void_p(0)
    h = ev.cuda_event if hasattr(ev, "cuda_event") else int(ev)
    if not h:
        raise ValueError("CUDA event not created yet: use make_event()")
    return ctypes.c_void_p(h)


def make_event(stream=None) -> torch.cuda.Event:
    """A torch CUDA event whose underlying cudaEvent_t already exists (torch
    creates it lazily on the first record)."""
    ev = torch.cuda.Event()
    ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ev


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise DvError(2, "dtype", str(t.dtype))


def _ok(st: int, where: str):
    if st != 0:
        detail = ""
        if st == 4:
            detail = f"(cudaError {lib().dv_last_cuda_error()})"
        raise DvError(st, where, detail)


# --------------------------------------------------------------------- utility

def dv_version() -> int:
    return lib().dv_version()


def dv_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far (captured
    launches included)."""
    return int(lib().dv_kernel_launches())


def dv_status_str(st: int) -> str:
    return lib().dv_status_str(st).decode()


def dv_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _ok(lib().dv_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
        "dv_workspace_init")


def workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """Allocate (through torch) and zero-fill a workspace of ``nbytes``."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    dv_workspace_init(ws, stream)
    return ws


def dv_check(ws: torch.Tensor, stream=None):
    """Synchronise and return (status, info) of the workspace's error word."""
    info = ctypes.c_int(0)
    st = lib().dv_check(_ptr(ws), _stream(stream), ctypes.byref(info))
    return st, info.value


# --------------------------------------------------------------------- predictor

class Predictor:
    """Arguments of one predictor (see dv_predictor in dv.h)."""

    def __init__(self, P1t, P2t, idx, count, mode=DV_TOPK, k=0, t=0.5, scores=None):
        self.P1t, self.P2t, self.idx, self.count, self.scores = P1t, P2t, idx, count, scores
        self.mode, self.k, self.t = int(mode), int(k), float(t)

    def c(self) -> dv_predictor:
        return dv_predictor(self.P1t.data_ptr(), self.P2t.data_ptr(), self.P1t.shape[0],
                            self.P2t.shape[0], self.mode, self.k, self.t, self.idx.data_ptr(),
                            self.idx.shape[-1], self.count.data_ptr(),
                            self.scores.data_ptr() if self.scores is not None else None)


def dv_predict_workspace_size(B: int, n_preds: int, r_max: int, N_max: int) -> int:
    n = ctypes.c_size_t(0)
    _ok(lib().dv_predict_workspace_size(B, n_preds, r_max, N_max, ctypes.byref(n)),
        "dv_predict_workspace_size")
    return n.value


def _preds(preds: Sequence[Predictor]):
    arr = (dv_predictor * len(preds))(*[p.c() for p in preds])
    return arr, len(preds)


def dv_predict(y: torch.Tensor, preds: Sequence[Predictor], ws: torch.Tensor, stream=None):
    arr, n = _preds(preds)
    B, d = y.shape
    _ok(lib().dv_predict(_ptr(y), B, d, _dt(y), arr, n, _ptr(ws), ws.numel(), _stream(stream)),
        "dv_predict")


def dv_predict_static(y: torch.Tensor, preds: Sequence[Predictor], stream=None):
    """dv_predict without a workspace: the library's fixed scratch array is
    used instead (for callers that cannot allocate; see dv.h for limits)."""
    arr, n = _preds(preds)
    B, d = y.shape
    _ok(lib().dv_predict_static(_ptr(y), B, d, _dt(y), arr, n, _stream(stream)),
        "dv_predict_static")


def dv_lookahead(y: torch.Tensor, preds: Sequence[Predictor], ws: torch.Tensor,
                 input_ready, side, done):
    arr, n = _preds(preds)
    B, d = y.shape
    _ok(lib().dv_lookahead(_ptr(y), B, d, _dt(y), arr, n, _ptr(ws), ws.numel(), _event(input_ready),
                           _stream(side), _event(done)), "dv_lookahead")


# --------------------------------------------------------------------- sparse MLP

def dv_sparse_mlp_workspace_size(B: int, d: int, N: int, cap: int) -> int:
    n = ctypes.c_size_t(0)
    _ok(lib().dv_sparse_mlp_workspace_size(B, d, N, cap, ctypes.byref(n)),
        "dv_sparse_mlp_workspace_size")
    return n.value


def dv_sparse_mlp(y, W1n, W2n, idx, count, out, ws, accumulate=False, stream=None):
    B, d = y.shape
    N = W1n.shape[0]
    _ok(lib().dv_sparse_mlp(_ptr(y), B, d, N, _ptr(W1n), _ptr(W2n), _ptr(idx), idx.shape[-1],
                            _ptr(count), _dt(y), _ptr(out), int(bool(accumulate)), _ptr(ws),
                            ws.numel(), _stream(stream)), "dv_sparse_mlp")


# --------------------------------------------------------------------- attention

class KV:
    """A batch's per-layer KV cache: K, V [B][h][n_max][d_h], X [B][n_max][d],
    valid [B][h][n_max] (uint8)."""

    def __init__(self, K, V, X, valid):
        self.K, self.V, self.X, self.valid = K, V, X, valid
        self.n_max = K.shape[2]

    @classmethod
    def empty(cls, B, h, n_max, d_h, d, dtype, device="cuda"):
        return cls(torch.zeros(B, h, n_max, d_h, dtype=dtype, device=device),
                   torch.zeros(B, h, n_max, d_h, dtype=dtype, device=device),
                   torch.zeros(B, n_max, d, dtype=dtype, device=device),
                   torch.zeros(B, h, n_max, dtype=torch.uint8, device=device))

    def c(self) -> dv_kv:
        return dv_kv(self.K.data_ptr(), self.V.data_ptr(), self.X.data_ptr(),
                     self.valid.data_ptr(), self.n_max)


def dv_sparse_attn_workspace_size(B, d, h, d_h, cap, n_max) -> int:
    n = ctypes.c_size_t(0)
    _ok(lib().dv_sparse_attn_workspace_size(B, d, h, d_h, cap, n_max, ctypes.byref(n)),
        "dv_sparse_attn_workspace_size")
    return n.value


def dv_sparse_attn(y, Wqkv, Wo, kv: KV, pos, head_idx, head_count, scale, out, ws,
                   accumulate=False, stream=None):
    B, d = y.shape
    h, _, d_h, _ = Wqkv.shape
    c = kv.c()
    _ok(lib().dv_sparse_attn(_ptr(y), B, d, h, d_h, _ptr(Wqkv), _ptr(Wo), ctypes.byref(c), _ptr(pos),
                             _ptr(head_idx), head_idx.shape[-1], _ptr(head_count), float(scale),
                             _dt(y), _ptr(out), int(bool(accumulate)), _ptr(ws), ws.numel(),
                             _stream(stream)), "dv_sparse_attn")


def dv_kv_repair(kv: KV, Wqkv, pos, head_idx, head_count, ws, stream=None):
    B = kv.K.shape[0]
    h, _, d_h, d = Wqkv.shape
    c = kv.c()
    _ok(lib().dv_kv_repair(ctypes.byref(c), B, d, h, d_h, _ptr(Wqkv), _ptr(pos), _ptr(head_idx),
                           head_idx.shape[-1], _ptr(head_count), _dt(Wqkv), _ptr(ws), ws.numel(),
                           _stream(stream)), "dv_kv_repair")


# --------------------------------------------------------------------- labels

def dv_label_workspace_size(T: int, d: int, N: int, h: int, d_h: int) -> int:
    n = ctypes.c_size_t(0)
    _ok(lib().dv_label_workspace_size(T, d, N, h, d_h, ctypes.byref(n)), "dv_label_workspace_size")
    return n.value


def dv_label_neurons(X, W1n, norms, ws, stream=None):
    T, d = X.shape
    _ok(lib().dv_label_neurons(_ptr(X), T, d, W1n.shape[0], _ptr(W1n), _dt(X), _ptr(norms), _ptr(ws),
                               ws.numel(), _stream(stream)), "dv_label_neurons")


def dv_label_heads(X, Wqkv, scale, norms, ws, stream=None):
    T, d = X.shape
    h, _, d_h, _ = Wqkv.shape
    _ok(lib().dv_label_heads(_ptr(X), T, d, h, d_h, _ptr(Wqkv), float(scale), _dt(X), _ptr(norms), _ptr(ws),
                             ws.numel(), _stream(stream)), "dv_label_heads")


def dv_select_scores(scores, mode, k, t, idx, count, ws, stream=None):
    B, N = scores.shape
    _ok(lib().dv_select_scores(_ptr(scores), B, N, int(mode), int(k), float(t), _ptr(idx), idx.shape[-1],
                               _ptr(count), _ptr(ws), ws.numel(), _stream(stream)), "dv_select_scores")


# --------------------------------------------------------------------- helpers

def dv_layernorm(x: torch.Tensor, y: torch.Tensor, eps: float = 1e-5, stream=None):
    B, d = x.shape
    _ok(lib().dv_layernorm(_ptr(x), B, d, float(eps), _ptr(y), _dt(y), _stream(stream)),
        "dv_layernorm")


def dv_positions_advance(pos: torch.Tensor, lo: int, hi: int, stream=None):
    _ok(lib().dv_positions_advance(_ptr(pos), pos.numel(), int(lo), int(hi), _stream(stream)),
        "dv_positions_advance")


def dv_set_launch_overlap(level: int) -> int:
    """Process-wide launch policy (see dv_set_launch_overlap in dv.h);
    returns the previous level."""
    return int(lib().dv_set_launch_overlap(int(level)))


def dv_set_wait_limit_ns(ns: int) -> int:
    """Process-wide bound of the device-side waits in nanoseconds (see
    dv_set_wait_limit_ns in dv.h; ns <= 0 restores one second); returns the
    previous bound."""
    return int(lib().dv_set_wait_limit_ns(int(ns)))

"""Helpers shared by the parity tests: conversions to the oracle's float64
arrays, tolerances, and the index-window comparison.

Tolerances (relative L2 of fp32 outputs against the float64 oracle):
  fp16 / bf16 inputs, fp32 accumulation: 1e-3;   fp32 inputs: 1e-5.
Index lists must match exactly, except a unit whose oracle score lies within
1e-5 of the threshold t or of the k-th largest score.
Stored K/V rows must lie within one unit in the last place (of the storage
type) of the exact float64 product.
"""

from __future__ import annotations

import math

import numpy as np
import torch

REL_L2 = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}
WINDOW = 1e-5
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
MANT = {"f32": 23, "f16": 10, "bf16": 7}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def rel_l2(x: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(np.asarray(x) - ref))
    return num / den if den > 0 else num


def assert_rel_l2(x, ref, dtype: str, what: str = ""):
    e = rel_l2(x, ref)
    assert e <= REL_L2[dtype], f"{what}: rel-L2 {e:.3g} > {REL_L2[dtype]:g}"
    return e


def within_ulp(got: np.ndarray, exact: np.ndarray, dtype: str, ulps: float = 1.0,
               acc_floor=None) -> bool:
    """|got - exact| <= ulps * ulp(exact) in the storage type (+ acc_floor).

    acc_floor, when given, is an absolute allowance per element for the fp32
    accumulation of the kernel's dot product (it matters only for values so
    small that one storage ulp is below the fp32 summation error)."""
    ax = np.maximum(np.abs(exact), 2.0 ** -14)
    ulp = np.exp2(np.floor(np.log2(ax)) - MANT[dtype])
    tol = ulps * ulp + (0.0 if acc_floor is None else acc_floor)
    return bool(np.all(np.abs(got - exact) <= tol))


def within_ulp_product(got: np.ndarray, X: np.ndarray, W: np.ndarray, dtype: str) -> bool:
    """Stored rows got = RNE(X W^T) computed with fp32 accumulation: within one
    storage ulp of the exact float64 product, plus an fp32 summation allowance
    of 4 * d * 2^-24 * rms_i(x_i w_i) per element."""
    exact = X @ W.T
    d = X.shape[1]
    rms = np.sqrt(((X * X) @ (W * W).T) / d)
    return within_ulp(got, exact, dtype, acc_floor=4.0 * d * 2.0 ** -24 * rms)


def topk_list_is_valid(lst: np.ndarray, s: np.ndarray, k: int) -> bool:
    """The kernel's own top-k decision on its own fp32 scores: k ascending
    unique units, every selected score >= every unselected score, and equal
    scores resolved in favour of the lower index."""
    if len(lst) != k or not ascending_unique(lst):
        return False
    if k == 0 or k == len(s):
        return k == 0 or lst.tolist() == list(range(len(s)))
    sel = np.zeros(len(s), dtype=bool)
    sel[lst] = True
    lo = s[sel].min()
    hi = s[~sel].max()
    if lo < hi:
        return False
    if lo == hi:  # a tie at the boundary: no unselected index below a selected one
        tied_sel = np.flatnonzero(sel & (s == lo))
        tied_out = np.flatnonzero(~sel & (s == lo))
        return tied_sel.max() < tied_out.min()
    return True


def check_selection(gpu: np.ndarray, ref: np.ndarray, s_ref: np.ndarray, mode: str,
                    k: int = 0, t: float = 0.5, window: float = WINDOW):
    """Compare one index list with the oracle's: every unit in the symmetric
    difference must have an oracle score within ``window`` of the boundary
    (the k-th largest score, or t).  Returns the number of such units."""
    g, r = set(gpu.tolist()), set(ref.tolist())
    diff = sorted(g ^ r)
    if not diff:
        return 0
    if mode == "topk":
        kth = np.sort(s_ref)[::-1][k - 1] if k > 0 else math.inf
        bound = kth
    else:
        bound = t
    bad = [j for j in diff if abs(s_ref[j] - bound) > window]
    assert not bad, f"index mismatch outside the {window} window: {bad[:10]} (bound {bound})"
    assert len(g) == len(r) or mode == "threshold"
    return len(diff)


def ascending_unique(x: np.ndarray) -> bool:
    return bool(np.all(np.diff(x) > 0))

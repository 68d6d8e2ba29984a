"""Float64 oracle: the method's steps, in the pages' order and notation.

TEST INFRASTRUCTURE ONLY (see the package docstring for the pages cited and
the readings taken).  Numpy's matmul is the only library primitive used; no
step is blocked, fused or reordered beyond what the formulas state.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

EPS_LN = 1e-5


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------

def round_to(x, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``dtype`` (ties to even)
    and return them as float64.  ``dtype`` is "f64" (no rounding), "f32",
    "f16" or "bf16".

    bf16 keeps 8 significant bits: with x = m * 2^e and 1/2 <= |m| < 1, the
    rounded value is rint(m * 2^8) * 2^(e-8), rint rounding halves to even.
    (Values are assumed inside bf16's normal range, as all inputs here are.)
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        m, e = np.frexp(x)
        return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# sparsity predictor  ([blog] §2; [notes] "Sparsity operator for MLP/Attention")
# --------------------------------------------------------------------------

def predictor_hidden(y: np.ndarray, P1t: np.ndarray) -> np.ndarray:
    """First predictor layer h = ReLU(y P1).  y [B][d]; P1t [r][d] holds the
    columns of P1 as rows.  Returns h [B][r]."""
    return np.maximum(0.0, np.atleast_2d(y) @ P1t.T)


def predictor_logits(h: np.ndarray, P2t: np.ndarray) -> np.ndarray:
    """Second predictor layer z = h P2, one output per head / neuron.
    P2t [N][r].  Returns z [B][N]."""
    return np.atleast_2d(h) @ P2t.T


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Per-unit binary classifier output s = 1 / (1 + exp(-z)) ([blog] §2)."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def select_threshold(s: np.ndarray, t: float) -> np.ndarray:
    """Units whose classifier says "select": s > t, ascending."""
    return np.flatnonzero(np.asarray(s) > t).astype(np.int32)


def select_topk(key: np.ndarray, k: int) -> np.ndarray:
    """The k units with the largest key (ties: lower index first), returned
    in ascending index order."""
    key = np.asarray(key)
    n = key.shape[0]
    if not 0 <= k <= n:
        raise ValueError("k out of range")
    order = np.lexsort((np.arange(n), -key))  # primary: key desc, then index asc
    return np.sort(order[:k]).astype(np.int32)


def predict(y, P1t, P2t, mode: str, k: Optional[int] = None, t: float = 0.5):
    """Two-layer predictor then selection, per batch row.

    Returns (lists, s, z): lists[b] is the ascending index list of row b,
    s and z are [B][N] float64 scores and logits.  Top-k ranks by the logit z,
    which orders units exactly as s = sigmoid(z) does (sigmoid is strictly
    increasing) without float64 saturation of s near 1.
    """
    h = predictor_hidden(y, P1t)
    z = predictor_logits(h, P2t)
    s = sigmoid(z)
    if mode == "topk":
        lists = [select_topk(z[b], k) for b in range(z.shape[0])]
    elif mode == "threshold":
        lists = [select_threshold(s[b], t) for b in range(z.shape[0])]
    else:
        raise ValueError(mode)
    return lists, s, z


# --------------------------------------------------------------------------
# sparsified MLP  ([notes] "Sparsified MLP"; [blog] §3.2 for the fused gather)
# --------------------------------------------------------------------------

def sparse_mlp(y: np.ndarray, W1n: np.ndarray, W2n: np.ndarray,
               S_M: Sequence[int]) -> np.ndarray:
    """MLP_{S_M}(y) = sigma(y W^1_{S_M}) (W^2_{S_M})^T for one token.

    y [d]; W1n, W2n [N][d] with row j = column j of W^1 / W^2.
    a_j = ReLU(y . W^1[:, j]) for j in S_M, then out = sum_j a_j W^2[:, j].
    """
    S = np.asarray(S_M, dtype=np.int64)
    y = np.asarray(y, dtype=np.float64).reshape(-1)
    if S.size == 0:
        return np.zeros(W2n.shape[1])
    a = np.maximum(0.0, W1n[S] @ y)
    return W2n[S].T @ a


def sparse_mlp_batched(Y, W1n, W2n, S_list) -> np.ndarray:
    """Batched reading: every row b uses its own S_M^b (units of the batch
    union outside S_M^b contribute nothing to row b)."""
    return np.stack([sparse_mlp(Y[b], W1n, W2n, S_list[b])
                     for b in range(len(S_list))])


def dense_mlp_zeroed(y, W1n, W2n, S_M) -> np.ndarray:
    """The dense MLP sigma(y W^1) (W^2)^T with the columns of W^1 outside S_M
    set to zero (an independent statement of the same result)."""
    keep = np.zeros(W1n.shape[0], dtype=bool)
    keep[np.asarray(S_M, dtype=np.int64)] = True
    W1z = np.where(keep[:, None], W1n, 0.0)
    return np.maximum(0.0, np.asarray(y).reshape(-1) @ W1z.T) @ W2n


# --------------------------------------------------------------------------
# sparsified attention with KV repair  ([notes] "Sparsified Attention",
# "Sparsity operator for Attention")
# --------------------------------------------------------------------------

@dataclasses.dataclass
class KVCache:
    """One sequence's per-layer cache.

    K, V [h][n_max][d_h]  key / value rows, values of the storage type
    X    [n_max][d]       the attention input y of every position
    valid [h][n_max]      whether K/V of (head, position) were computed
    dtype                 storage type used to round new K/V rows
    """

    K: np.ndarray
    V: np.ndarray
    X: np.ndarray
    valid: np.ndarray
    dtype: str

    @classmethod
    def empty(cls, h: int, n_max: int, d_h: int, d: int, dtype: str):
        return cls(np.zeros((h, n_max, d_h)), np.zeros((h, n_max, d_h)),
                   np.zeros((n_max, d)), np.zeros((h, n_max), dtype=bool), dtype)

    def copy(self) -> "KVCache":
        return KVCache(self.K.copy(), self.V.copy(), self.X.copy(),
                       self.valid.copy(), self.dtype)


def _proj(Wqkv, i: int, m: int, x: np.ndarray) -> np.ndarray:
    """x W_i^m for m = 0 (Q), 1 (K), 2 (V); Wqkv[i][m] holds W_i^m's columns."""
    return Wqkv[i, m] @ x


def kv_append(cache: KVCache, y: np.ndarray, Wqkv: np.ndarray, n: int,
              S_A: Sequence[int]) -> None:
    """Store the current token at position n: X[n] = y; for each selected
    head its key y W_i^K and value y W_i^V (rounded to the storage type) with
    valid = 1; the other heads' rows at n are marked missing (their K/V are
    recomputed from X[n] if the head is selected later)."""
    cache.X[n] = y
    cache.valid[:, n] = False
    for i in S_A:
        cache.K[i, n] = round_to(_proj(Wqkv, i, 1, y), cache.dtype)
        cache.V[i, n] = round_to(_proj(Wqkv, i, 2, y), cache.dtype)
        cache.valid[i, n] = True


def kv_prefill(cache: KVCache, Wqkv: np.ndarray, n: int,
               heads: Optional[Sequence[int]] = None) -> None:
    """A dense prompt of n positions: K/V of the given heads (default: all)
    at positions < n from the stored X (all rows of a head in one product),
    valid = 1.  Equal to kv_append at every prompt position up to float64
    summation order; used to set up large cases, not by the pins."""
    for i in (range(Wqkv.shape[0]) if heads is None else heads):
        cache.K[i, :n] = round_to(cache.X[:n] @ Wqkv[i, 1].T, cache.dtype)
        cache.V[i, :n] = round_to(cache.X[:n] @ Wqkv[i, 2].T, cache.dtype)
        cache.valid[i, :n] = True


def kv_repair(cache: KVCache, Wqkv: np.ndarray, n: int,
              S_A: Sequence[int]) -> int:
    """KV repair: for every selected head and every earlier position j < n
    whose K/V were skipped, reload the stored embedding X[j] and recompute
    K[i][j] = X[j] W_i^K, V[i][j] = X[j] W_i^V with the same product as the
    append step.  Returns the rows repaired."""
    fixed = 0
    for i in S_A:
        for j in np.flatnonzero(~cache.valid[i, :n]):
            cache.K[i, j] = round_to(_proj(Wqkv, i, 1, cache.X[j]), cache.dtype)
            cache.V[i, j] = round_to(_proj(Wqkv, i, 2, cache.X[j]), cache.dtype)
            cache.valid[i, j] = True
            fixed += 1
    return fixed


def head_output(q_i: np.ndarray, K_i: np.ndarray, V_i: np.ndarray,
                c: float) -> np.ndarray:
    """H_i(y) = D_i(y)^-1 exp(c q_i K_i^T) V_i with D_i = exp(c q_i K_i^T) 1_n.

    K_i, V_i [n+1][d_h] are the head's key and value rows (X W_i^K, X W_i^V).
    The common factor exp(-max logit) is taken out of numerator and
    denominator, which leaves the ratio unchanged.
    """
    logits = c * (K_i @ q_i)
    w = np.exp(logits - logits.max())
    return (w @ V_i) / w.sum()


def sparse_attn(y: np.ndarray, Wqkv: np.ndarray, Wo: np.ndarray,
                cache: KVCache, n: int, S_A: Sequence[int], c: float):
    """MHA_{S_A}(y) = sum_{i in S_A} H_i(y) W_i^O for the token at position n.

    Order: append the token (X[n], the selected heads' K/V at n), repair the
    selected heads' missing rows, then for each selected head
    q_i = y W_i^Q, H_i over positions 0..n, and the projected sum.
    Mutates ``cache``; returns out [d].
    """
    y = np.asarray(y, dtype=np.float64).reshape(-1)
    kv_append(cache, y, Wqkv, n, S_A)
    kv_repair(cache, Wqkv, n, S_A)
    out = np.zeros(Wo.shape[2])
    for i in S_A:
        q_i = _proj(Wqkv, i, 0, y)
        H_i = head_output(q_i, cache.K[i, :n + 1], cache.V[i, :n + 1], c)
        out += H_i @ Wo[i]
    return out


def sparse_attn_batched(Y, Wqkv, Wo, caches: List[KVCache], pos, S_list, c):
    """Batched reading: row b attends over its own cache with its own S_A^b."""
    return np.stack([sparse_attn(Y[b], Wqkv, Wo, caches[b], int(pos[b]),
                                 S_list[b], c) for b in range(len(S_list))])


# --------------------------------------------------------------------------
# decoder layer and stack with look-ahead prediction
# ([blog] §3.1; [notes] "Reducing Overhead with Asynchronous Execution")
# --------------------------------------------------------------------------

def layernorm(x: np.ndarray, eps: float = EPS_LN) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) over the last axis, no affine terms."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def decode_layer(r: np.ndarray, W: dict, cache: KVCache, n: int, S_A, S_M,
                 c: float, dtype: str):
    """One pre-LN decoder layer on the residual stream r [d]:
    y_a = LN(r) (stored as the layer's attention input), r += MHA_{S_A}(y_a),
    y_m = LN(r), r += MLP_{S_M}(y_m).  The LayerNorm outputs are rounded to
    the storage type, which is what the sparse blocks read.
    Returns (r_new, y_a)."""
    y_a = round_to(layernorm(r), dtype)
    r = r + sparse_attn(y_a, W["Wqkv"], W["Wo"], cache, n, S_A, c)
    y_m = round_to(layernorm(r), dtype)
    r = r + sparse_mlp(y_m, W["W1n"], W["W2n"], S_M)
    return r, y_a


def lookahead(y_l: np.ndarray, W_next: dict, k_heads: int, k_neurons: int):
    """Look-ahead prediction: layer l+1's head set S_A and neuron set S_M,
    both predicted from layer l's attention input y_l (top-k)."""
    S_A = predict(y_l, W_next["PA1t"], W_next["PA2t"], "topk", k_heads)[0][0]
    S_M = predict(y_l, W_next["PM1t"], W_next["PM2t"], "topk", k_neurons)[0][0]
    return S_A, S_M


def decode_stack(r: np.ndarray, layers: List[dict], caches: List[KVCache],
                 n: int, c: float, dtype: str, k_heads: int, k_neurons: int,
                 force_sets=None, trace: Optional[list] = None):
    """One decoded token through the stack at position n.

    Layer 0 predicts its own sets from its own attention input; every later
    layer l+1 uses the sets predicted from layer l's attention input.
    ``force_sets`` (list of (S_A, S_M) per layer) replaces the predictions.
    If ``trace`` is a list, the input each layer's sets were predicted from
    is appended to it.  Returns (r_out, sets) with sets[l] = (S_A, S_M) used
    by layer l.
    """
    sets = []
    pending = None
    src = None
    for l, W in enumerate(layers):
        if force_sets is not None:
            S_A, S_M = force_sets[l]
        elif pending is None:
            src = round_to(layernorm(r), dtype)
            S_A, S_M = lookahead(src, W, k_heads, k_neurons)
        else:
            S_A, S_M = pending
        if trace is not None:
            trace.append(src)
        sets.append((np.asarray(S_A), np.asarray(S_M)))
        r, y_a = decode_layer(r, W, caches[l], n, S_A, S_M, c, dtype)
        if l + 1 < len(layers) and force_sets is None:
            pending = lookahead(y_a, layers[l + 1], k_heads, k_neurons)
            src = y_a
    return r, sets


def prefill_dense(E: np.ndarray, layers: List[dict], caches: List[KVCache],
                  c: float, dtype: str) -> np.ndarray:
    """The prompt phase ([notes] "Typical LLM procedure": the prompt is run
    through every layer, which builds each layer's KV cache; generation then
    goes token by token): the dense model, S_A = all heads and S_M = all
    neurons, over prompt positions 0..T-1 in order.  Position t attends over
    positions 0..t of its layer, which is causal attention; every layer
    stores its attention input X[t] and the K/V of every head at t.

    E [T][d] holds the residual stream entering layer 0 at each position.
    Mutates ``caches``; returns the residual stream after the last layer,
    [T][d]."""
    E = np.asarray(E, dtype=np.float64)
    h = layers[0]["Wqkv"].shape[0]
    N = layers[0]["W1n"].shape[0]
    every = [(np.arange(h), np.arange(N))] * len(layers)
    out = np.zeros_like(E)
    for t in range(E.shape[0]):
        out[t], _ = decode_stack(E[t], layers, caches, t, c, dtype, h, N, force_sets=every)
    return out


# --------------------------------------------------------------------------
# true-sparsity labels  ([blog] §1 Contextual Sparsity: run the sequence
# through the layer, keep the heads and MLP neurons whose outputs have the
# largest L2 norm; [blog] §2: a threshold on that norm splits units into
# positive and negative examples for the predictor)
# --------------------------------------------------------------------------

def neuron_norms(X: np.ndarray, W1n: np.ndarray) -> np.ndarray:
    """For every neuron j, the L2 norm over the sequence's tokens (the rows
    of X [T][d]) of its activation ReLU(x_t . W^1[:, j]): the MLP's T x 4d
    activation matrix read neuron by neuron (one norm per column).
    Returns [N]."""
    A = np.maximum(0.0, np.atleast_2d(X) @ W1n.T)
    return np.sqrt((A * A).sum(axis=0))


def head_outputs_causal(X: np.ndarray, Wqkv: np.ndarray, c: float,
                        dtype: str) -> np.ndarray:
    """Every head's output matrix H_i [T][d_h] over the sequence X [T][d]:
    token t attends to tokens 0..t (itself included), with its query
    x_t W_i^Q in float64 and the keys / values x_j W_i^{K,V} rounded to the
    storage type, as the KV cache holds them.  Returns [h][T][d_h]."""
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    T = X.shape[0]
    h, _, d_h, _ = Wqkv.shape
    out = np.zeros((h, T, d_h))
    for i in range(h):
        Q = X @ Wqkv[i, 0].T
        K = round_to(X @ Wqkv[i, 1].T, dtype)
        V = round_to(X @ Wqkv[i, 2].T, dtype)
        for t in range(T):
            out[i, t] = head_output(Q[t], K[: t + 1], V[: t + 1], c)
    return out


def head_norms(X: np.ndarray, Wqkv: np.ndarray, c: float, dtype: str) -> np.ndarray:
    """For every head i, the L2 (Frobenius) norm of its output matrix H_i
    over the sequence, taken before the output projection W_i^O (the page's
    example leaves the final linear layer out).  Returns [h]."""
    H = head_outputs_causal(X, Wqkv, c, dtype)
    return np.sqrt((H * H).sum(axis=(1, 2)))


def label(norms: np.ndarray, mode: str, k: Optional[int] = None,
          t: Optional[float] = None) -> np.ndarray:
    """The units labelled important: the k largest norms (ties to the lower
    index) or every norm above t; ascending."""
    if mode == "topk":
        return select_topk(np.asarray(norms), k)
    if mode == "threshold":
        return select_threshold(np.asarray(norms), t)
    raise ValueError(mode)

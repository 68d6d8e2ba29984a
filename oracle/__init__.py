"""Float64 CPU oracle of the contextually sparse decode step (Deja Vu).

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
statement of what the CUDA library computes.  Only the test suite, the smoke
check and the benchmark's CPU-baseline / reference arm may import it; the
library itself never does, and it shares no code with the library.

Pages followed (cited below by the short names in brackets):
  [blog]     "用Deja Vu来提高 LLM 的推理速度" (m.haoling.cc/wenzhang/678872):
             §1 Contextual Sparsity, §2 稀疏性预测 (sparsity prediction),
             §3.1 并行化稀疏性预测 (parallel prediction), §3.2 Kernel Fusion.
  [abstract] "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference
             Time" (arXiv 2310.17157 listing), abstract.
  [notes]    Deja Vu reading notes (pages.squarehuang.top/paper/DejaVu):
             "Sparsified MLP", "Sparsified Attention", "Deja Vu Framework"
             (sparsity operators for MLP and attention, KV repair,
             "Reducing Overhead with Asynchronous Execution").

Readings taken where the pages are silent or garbled (each is listed in the
design notes of the repository):
  * neuron j owns column j of W^1 and column j of W^2 ([notes] "Sparsified
    MLP" writes sigma(y W^1_S)(W^2_S)^T, so both matrices are d x 4d);
  * sigma in the MLP is ReLU; the predictor's hidden activation is ReLU and
    its output is a sigmoid per unit ([blog] §2);
  * top-k ranks by score, ties go to the lower index; every list is returned
    in ascending order; a threshold keeps s > t (strict);
  * the head outputs are summed ([notes] "Sparsified Attention", the sum over
    S_A), not averaged;
  * the current token is appended to the cache first and then attended to,
    so a step at position n attends over positions 0..n;
  * the softmax logits are multiplied by a caller-given scale c (the page's
    formula prints none: c = 1 is the literal reading);
  * K/V are stored in the storage type, rounded to nearest even; q, scores,
    H_i and outputs stay in float64 here;
  * the decoder stack is pre-LayerNorm without affine terms (eps 1e-5) with
    residual adds; the attention input y is what the cache's X stores;
  * the true-sparsity labels ([blog] §1) are norms over a sequence: a
    neuron's is the L2 norm of its ReLU activations over the tokens, a
    head's the Frobenius norm of its causal output matrix H_i before W_i^O;
    a label set is the top-k norms or the norms above a threshold.

Every function takes float64 numpy arrays (widened from the storage type by
the caller) and returns float64 results (int32 for index lists).
"""

from .core import (  # noqa: F401
    EPS_LN,
    round_to,
    predictor_hidden,
    predictor_logits,
    sigmoid,
    select_threshold,
    select_topk,
    predict,
    sparse_mlp,
    sparse_mlp_batched,
    dense_mlp_zeroed,
    KVCache,
    kv_append,
    kv_prefill,
    kv_repair,
    head_output,
    sparse_attn,
    sparse_attn_batched,
    layernorm,
    decode_layer,
    lookahead,
    decode_stack,
    prefill_dense,
    neuron_norms,
    head_outputs_causal,
    head_norms,
    label,
)

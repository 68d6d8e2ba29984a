/*
 * dv.h -- C ABI of the GB300 (sm_103a) contextually sparse decode library
 * (libdv.so).
 *
 * The library computes one decode step of Deja Vu's contextual sparsity:
 * a low-rank predictor picks input-dependent attention heads and MLP
 * neurons, and fused gather-and-multiply kernels compute only those.
 *
 * Pages that define the operations (cited per entry point):
 *   [blog]  "用Deja Vu来提高 LLM 的推理速度" (m.haoling.cc/wenzhang/678872),
 *           §2 稀疏性预测 (sparsity prediction), §3.1 并行化稀疏性预测
 *           (parallel / look-ahead prediction), §3.2 Kernel Fusion,
 *           §3.3 Memory coalescing.
 *   [notes] Deja Vu reading notes (pages.squarehuang.top/paper/DejaVu):
 *           "Sparsified MLP", "Sparsified Attention", "Deja Vu Framework"
 *           (sparsity operators for MLP / attention, KV repair,
 *           "Reducing Overhead with Asynchronous Execution").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument that names a tensor is DEVICE memory owned by
 *    the caller; the library never allocates, frees or keeps a pointer after
 *    the call returns.  Host-side descriptor structs (dv_kv, dv_predictor)
 *    are read during the call only.
 *  - Every compute call is asynchronous on the given stream and can be
 *    captured into a CUDA graph.  The host never reads device data (counts
 *    stay on the device); only dv_check() synchronises.
 *  - Weights, token embeddings and the KV cache share one storage type
 *    `dt` (DV_F32, DV_F16 or DV_BF16); accumulation is fp32.  Outputs of
 *    the sparse blocks are fp32.
 *  - Tensor pointers must be 16-byte aligned and row lengths (d, r, d_h)
 *    multiples of 8 elements (4 for DV_F32); otherwise DV_ERR_INVALID_ARG.
 *  - Index lists are int32, ascending, with their element count held in
 *    device memory; a list has room for `cap` entries per batch row.
 *  - Scratch space: each call takes a caller-owned device workspace of at
 *    least the size its *_workspace_size() query reports.  A workspace must
 *    be zero-filled once (dv_workspace_init) before its first use; the
 *    library leaves it reusable, also after a device wait has timed out
 *    (DV_ERR_TIMEOUT): a late arrival still brings the workspace's counters
 *    back to zero.  A workspace that was never zero-filled reports
 *    DV_ERR_TIMEOUT or DV_ERR_WORKSPACE from dv_check; zero-fill it
 *    (dv_workspace_init) before the next call.  Calls that may run
 *    concurrently (e.g. the look-ahead predictor on a side stream) need
 *    distinct workspaces.
 *  - Errors found on the host (bad arguments) are returned at once and
 *    nothing is launched.  Errors found on the device (an index outside
 *    [0, N), a count above cap, a position outside the cache) never trap:
 *    the offending element is skipped and a code is recorded in the
 *    workspace's error word, which dv_check() returns and clears.
 *
 * Storage layouts (row-major; "rows" are contiguous):
 *    y      [B][d]              token input(s) of a block
 *    P1t    [r][d]              predictor layer 1, row j = column j of P1
 *    P2t    [N][r]              predictor layer 2, row u = column u of P2
 *    W1n    [N][d]              row j = column j of W^1 (neuron j's input)
 *    W2n    [N][d]              row j = column j of W^2 (neuron j's output)
 *    Wqkv   [h][3][d_h][d]      [i][m][t] = column t of W_i^m, m = Q, K, V
 *    Wo     [h][d_h][d]         W_i^O
 *    K, V   [B][h][n_max][d_h]  KV cache, X [B][n_max][d], valid [B][h][n_max]
 */
#ifndef DV_H_
#define DV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dv_status {
  DV_OK = 0,
  DV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, cap < k */
  DV_ERR_DTYPE = 2,        /* unsupported storage / output type            */
  DV_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required   */
  DV_ERR_CUDA = 4,         /* a CUDA call failed: see dv_last_cuda_error() */
  DV_ERR_INDEX_RANGE = 5,  /* device: an index outside [0, N) was skipped  */
  DV_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up               */
  DV_ERR_UNSUPPORTED = 7,  /* shape outside what the kernels support       */
  DV_ERR_CAPACITY = 8,     /* device: a list was longer than cap; truncated */
  DV_ERR_POSITION = 9      /* device: a position outside [0, n_max)        */
} dv_status;

typedef enum dv_dtype { DV_F32 = 0, DV_F16 = 1, DV_BF16 = 2 } dv_dtype;

typedef enum dv_select {
  DV_TOPK = 0,       /* the k units with the largest score; ties -> lower index */
  DV_THRESHOLD = 1   /* every unit with score s > t (strict)                    */
} dv_select;

/* One sparsity predictor ([blog] §2: a two-layer MLP with one sigmoid per
 * head / neuron).  Used by dv_predict and dv_lookahead. */
typedef struct dv_predictor {
  const void* P1t;     /* [r][d], storage type                               */
  const void* P2t;     /* [N][r], storage type                               */
  int r;               /* predictor rank (hidden width)                      */
  int N;               /* units scored: h (heads) or 4d (neurons)            */
  dv_select mode;
  int k;               /* DV_TOPK: units kept per row, 0 <= k <= min(N, cap) */
  float t;             /* DV_THRESHOLD: keep s > t                           */
  int32_t* idx;        /* out [B][cap]: selected units, ascending            */
  int cap;             /* room per row in idx                                */
  int32_t* count;      /* out [B]: entries written per row                   */
  float* scores;       /* out [B][N] fp32 sigmoid scores, or NULL            */
} dv_predictor;

/* Per-layer KV cache of a batch of sequences ([notes] "Sparsity operator
 * for Attention": the cache holds K/V of heads that were computed and the
 * token embedding X of every position, so skipped heads can be repaired). */
typedef struct dv_kv {
  void* K;          /* [B][h][n_max][d_h], storage type                      */
  void* V;          /* [B][h][n_max][d_h], storage type                      */
  void* X;          /* [B][n_max][d], storage type: attention input per pos  */
  uint8_t* valid;   /* [B][h][n_max]: 1 where K/V of (head, pos) are present */
  int n_max;        /* positions per sequence                                */
} dv_kv;

/* ---------------------------------------------------------------- utility */

const char* dv_status_str(dv_status s);
/* The cudaError_t (as int) of the last failing CUDA call in this thread. */
int dv_last_cuda_error(void);
/* Library version, e.g. 100 for 0.1.0. */
int dv_version(void);
/* Number of kernels the library has enqueued in this process so far,
 * launches captured into a CUDA graph included (a diagnostic: the difference
 * across the calls of one step is that step's kernel count).  No
 * counterpart in the pages. */
long long dv_kernel_launches(void);

/* Zero-fill a workspace (once, before its first use). */
dv_status dv_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the workspace's device error
 * word.  Returns DV_OK or the first device-detected error code recorded
 * since the last check; *info (if not NULL) receives the offending value
 * (an index, a count or a position). */
dv_status dv_check(void* ws, cudaStream_t stream, int* info);

/* ------------------------------------------------------------- predictor */

/* Workspace bytes for dv_predict / dv_lookahead with up to `n_preds`
 * predictors of rank <= r_max scoring <= N_max units, batch B. */
dv_status dv_predict_workspace_size(int B, int n_preds, int r_max, int N_max,
                                    size_t* bytes);

/* Sparsity prediction ([blog] §2; [notes] "Sparsity operator for MLP" and
 * "... for Attention"): for each predictor p and batch row b
 *     h = ReLU(y_b P1),  z = h P2,  s = sigmoid(z)   (fp32 throughout)
 * then top-k or threshold selection into p.idx[b][...] (ascending) and
 * p.count[b].  Top-k ranks by s, ties to the lower index.  1 <= n_preds <= 2;
 * both predictors read the same y [B][d] and run in fused launches.
 * Limits: B <= 32, d <= 16384, r <= 4096, N <= 53248 (the selection stages
 * one row's scores in shared memory). */
dv_status dv_predict(const void* y, int B, int d, dv_dtype dt,
                     const dv_predictor* preds, int n_preds,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* Asynchronous look-ahead prediction ([blog] §3.1; [notes] "Reducing
 * Overhead with Asynchronous Execution"): layer l+1's predictors run on
 * `side` from layer l's attention input y.  `side` first waits for
 * `input_ready` (if not NULL), then runs dv_predict, then records `done`
 * (if not NULL), which the main stream waits on before layer l+1. */
dv_status dv_lookahead(const void* y, int B, int d, dv_dtype dt,
                       const dv_predictor* preds, int n_preds,
                       void* ws, size_t ws_bytes,
                       cudaEvent_t input_ready, cudaStream_t side,
                       cudaEvent_t done);

/* Sparsity prediction without a caller workspace.  The pages have no
 * counterpart to this entry point: it exists for callers that cannot
 * allocate device memory -- for example a plugin inside a serving engine
 * that owns every device allocation, or a latency-critical loop where a
 * cudaMalloc (which can synchronise the device) is not allowed.
 *
 * Computes exactly what dv_predict computes, with the same arguments minus
 * the workspace.  Its scratch lives in a fixed array inside the library
 * (about 1.1 MB; every GPU that loads the library holds one until the
 * process exits).  Limits: B <= 4, r <= 1024 and N <= 32768 per predictor;
 * larger shapes are rejected with DV_ERR_WORKSPACE before anything runs.
 * Nothing is allocated or freed: no cudaMalloc, no cudaFree.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call, on any stream, shares the one array and overwrites what the
 *    previous call left there: calls whose work overlaps on the GPU race and
 *    give wrong results.  Serialise them (one stream, or events).
 *  - Device-side conditions are not reported: a threshold list longer than
 *    cap is truncated to cap entries as in dv_predict, with no error word to
 *    read back. */
dv_status dv_predict_static(const void* y, int B, int d, dv_dtype dt,
                            const dv_predictor* preds, int n_preds,
                            cudaStream_t stream);

/* ------------------------------------------------------------ sparse MLP */

dv_status dv_sparse_mlp_workspace_size(int B, int d, int N, int cap,
                                       size_t* bytes);

/* Sparsified MLP ([notes] "Sparsified MLP"; fused gather [blog] §3.2):
 *     out_b (+)= sum_{j in S_b} ReLU(y_b . W1n[j]) * W2n[j]
 * computed in one pass over the selected rows of W1n and W2n (no weight
 * sub-matrix is materialised).  S_b = idx[b][0 .. count[b]).  For B > 1 the
 * rows of the batch union are read once and each row b uses its own S_b.
 * out [B][d] fp32: overwritten (accumulate = 0) or added to (accumulate = 1,
 * e.g. a residual stream).  Below 8 rows every output element has one
 * writer and a fixed summation order, so results repeat bit for bit; the
 * tensor-core path (2+ rows of a 16-bit type) adds partial sums with fp32
 * atomics, so there the last bits of out may differ between runs.
 * Limits: B <= 32, d <= 16384 (8192 for DV_F32), N <= 65536. */
dv_status dv_sparse_mlp(const void* y, int B, int d, int N,
                        const void* W1n, const void* W2n,
                        const int32_t* idx, int cap, const int32_t* count,
                        dv_dtype dt, float* out, int accumulate,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------- attention */

dv_status dv_sparse_attn_workspace_size(int B, int d, int h, int d_h, int cap,
                                        int n_max, size_t* bytes);

/* Sparsified attention for the token at position pos[b] of each sequence
 * ([notes] "Sparsified Attention" and "Sparsity operator for Attention"):
 *   1. append: X[b][pos] = y_b; for i in S_b: K/V[b][i][pos] = y_b W_i^{K,V}
 *      rounded to the storage type; valid[b][i][pos] = (i in S_b);
 *   2. KV repair: for i in S_b and every j < pos with valid[b][i][j] = 0,
 *      K/V[b][i][j] = X[b][j] W_i^{K,V}, then valid = 1;
 *   3. H_i = softmax(scale * q_i K_i^T) V_i over positions 0..pos, with
 *      q_i = y_b W_i^Q (fp32);
 *   4. out_b (+)= sum_{i in S_b} H_i W_i^O.
 * S_b = head_idx[b][0 .. head_count[b]); pos [B] is device memory.
 * scale multiplies the logits (1/sqrt(d_h) for the usual convention; the
 * page's formula prints none).  out [B][d] fp32, see dv_sparse_mlp for
 * `accumulate`.  Limits: B <= 32, d_h in {64, 128}, h <= 1024,
 * n_max <= 65536 (a multiple of 16), and one projection row of at most
 * 40 KB (d <= 20480 for 16-bit types, 10240 for DV_F32); other head
 * dimensions and rows return DV_ERR_UNSUPPORTED. */
dv_status dv_sparse_attn(const void* y, int B, int d, int h, int d_h,
                         const void* Wqkv, const void* Wo, const dv_kv* kv,
                         const int32_t* pos, const int32_t* head_idx, int cap,
                         const int32_t* head_count, float scale, dv_dtype dt,
                         float* out, int accumulate,
                         void* ws, size_t ws_bytes, cudaStream_t stream);

/* KV repair alone ([notes] "Sparsity operator for Attention"): for every
 * selected head i of sequence b and every j < pos[b] with valid = 0,
 * recompute K/V[b][i][j] from X[b][j] and set valid = 1.  With every head
 * selected and valid all 0 this is a dense prefill of positions 0..pos-1.
 * Uses the dv_sparse_attn workspace. */
dv_status dv_kv_repair(const dv_kv* kv, int B, int d, int h, int d_h,
                       const void* Wqkv, const int32_t* pos,
                       const int32_t* head_idx, int cap,
                       const int32_t* head_count, dv_dtype dt,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------- true-sparsity labels */

/* Workspace bytes for dv_label_neurons (sequence of T tokens, N neurons)
 * and dv_label_heads (h heads of d_h); one workspace serves both. */
dv_status dv_label_workspace_size(int T, int d, int N, int h, int d_h,
                                  size_t* bytes);

/* Neuron labels ([blog] §1 Contextual Sparsity: MLP neurons whose outputs
 * over the input sequence have a large L2 norm, read neuron by neuron):
 *     norms[j] = sqrt( sum_t ReLU(X[t] . W1n[j])^2 ),  j < N,
 * for a sequence X [T][d] (e.g. a prompt's MLP inputs).  The product runs
 * on the tensor cores: 16-bit storage only (DV_F32 -> DV_ERR_DTYPE);
 * d a multiple of 8; fp32 accumulation; per-tile sums added in a fixed
 * order.  norms [N] fp32, device. */
dv_status dv_label_neurons(const void* X, int T, int d, int N, const void* W1n,
                           dv_dtype dt, float* norms, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Head labels ([blog] §1: attention heads whose output matrix over the
 * sequence has a large L2 norm, taken before the output projection):
 *     norms[i] = || H_i ||_F,  H_i[t] = softmax(scale q_t K_i[0..t]^T) V_i[0..t]
 * (causal: token t attends to tokens 0..t), q_t = X[t] W_i^Q in fp32 and
 * K/V = X W_i^{K,V} rounded to the storage type as a KV cache holds them.
 * 16-bit storage only; d_h in {64, 128}; norms [h] fp32, device. */
dv_status dv_label_heads(const void* X, int T, int d, int h, int d_h,
                         const void* Wqkv, float scale, dv_dtype dt,
                         float* norms, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/* Selection over rows of non-negative, finite fp32 scores [B][N] (e.g. the
 * label norms; [blog] §2: a threshold on the norm gives the labels): top-k
 * (ties to the lower index) or score > t, ascending, into idx [B][cap] with
 * count [B]; the same selection as dv_predict's.  N <= 53248.  ws: at
 * least 256 bytes, zero-filled once (its error word: a threshold list
 * longer than cap is truncated and reported as DV_ERR_CAPACITY). */
dv_status dv_select_scores(const float* scores, int B, int N, dv_select mode,
                           int k, float t, int32_t* idx, int cap,
                           int32_t* count, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* ---------------------------------------------------- decoder-step helpers */

/* y_b = LayerNorm(x_b) without affine terms (eps given), rounded to the
 * storage type: the pre-LN input of each sparse block (the pages do not state
 * the normalisation; this is the plain pre-LN reading).  x [B][d] fp32,
 * 16-byte aligned, d a multiple of 4 and at most 16384; y [B][d] 8-byte
 * aligned.  Other shapes return DV_ERR_INVALID_ARG. */
dv_status dv_layernorm(const float* x, int B, int d, float eps,
                       void* y, dv_dtype dt, cudaStream_t stream);

/* Launch policy (no counterpart in the pages; it changes timing, never
 * results).  Inside every entry point the later kernels start during the
 * earlier ones and read only data those do not write.  At level 0 (the
 * default) the first kernel of each call waits for everything before it.
 * At level 1, for batch 1, the first kernel of dv_sparse_attn and of
 * dv_sparse_mlp may also start while the kernel before the call is still
 * running, and reads before waiting for it: the head / neuron lists and
 * counts, pos, the valid flags and the weights.  Enable it only when the
 * kernel issued just before each such call (on the same stream) writes none
 * of those -- true when that kernel is the dv_layernorm producing the call's
 * y, as in a pre-LN decoder -- and neither does the kernel before that
 * layernorm, which lets its consumer start at once (in a pre-LN decoder it
 * is the previous block's dv_sparse_attn or dv_sparse_mlp).  Process-wide;
 * returns the previous level. */
int dv_set_launch_overlap(int level);

/* Bound of every device-side wait (no counterpart in the pages): the
 * one-launch MLP's wait for its up-projection CTAs and the tensor-core
 * path's pipeline waits give up after `ns` nanoseconds of the GPU's global
 * timer, record DV_ERR_TIMEOUT in the workspace (read it with dv_check) and
 * unwind; the kernel still waits for its own tensor-core and copy work in
 * flight before it exits.  ns <= 0 restores the default of one second.
 * Read at launch (a captured graph keeps the value it was captured with);
 * process-wide; returns the previous bound. */
long long dv_set_wait_limit_ns(long long ns);

/* pos[b] = pos[b] + 1, or `lo` when that reaches `hi` (decode loop). */
dv_status dv_positions_advance(int32_t* pos, int B, int lo, int hi,
                               cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DV_H_ */

// Host-side launchers of libdv's kernels (one translation unit each).
// Shapes have been validated by the C-ABI layer before any launcher runs.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "dv_common.cuh"
#include "per_device.h"

namespace dv {

// The current device id (-1 if it cannot be read): the key of PerDevice caches.
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  return dev;
}

// Bound of every device-side wait, in nanoseconds of %globaltimer
// (dv_set_wait_limit_ns; default one second).  A wait that runs out records
// DV_ERR_TIMEOUT in the workspace and the kernel unwinds.
long long wait_limit_ns();
long long set_wait_limit_ns(long long ns);

// Record a failed CUDA call for dv_last_cuda_error() and return DV_ERR_CUDA.
dv_status cuda_fail(cudaError_t e);

// Kernels this library has enqueued in this process (dv_kernel_launches):
// every launch site adds its launches once they are accepted.
void count_launches(int n);
long long launches_total();

// Launch with an optional programmatic dependency on the previous kernel of
// the stream (see grid_dep_wait / grid_dep_launch).  Used only between the
// kernels of one entry point, whose data dependencies are known; the first
// kernel of every entry point is launched the ordinary way.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     bool pdl, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? at : nullptr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

// SM count of the current device (cached per device).
int num_sms_current();

// Launch policy (dv_set_launch_overlap): 1 lets the first kernel of a batch-1
// attention or MLP call start during the kernel before the call (k_misc.cu).
int launch_overlap();
int set_launch_overlap(int level);

// ---- predictor (k_predict.cu) ----------------------------------------------

// Largest unit count a selection CTA stages in shared memory (208 KB).
constexpr int kSelectMaxN = 53248;

struct PredLaunch {
  const void* P1t[2];
  const void* P2t[2];
  int r[2], N[2];
  int mode[2], k[2];
  float t[2];
  int32_t* idx[2];
  int cap[2];
  int32_t* count[2];
  float* h[2];       // [B][r] fp32 scratch
  float* s[2];       // [B][N] fp32 scores (caller buffer or scratch)
  void* h_hi[2];     // tensor-core path: [32][r] storage-type halves of h,
  void* h_lo[2];     // or null (then the CUDA-core path runs)
};

cudaError_t launch_predict(const void* y, int B, int d, dv_dtype dt,
                           const PredLaunch& p, int n_preds, WsHeader* hdr,
                           cudaStream_t stream);

// Both products of the predictor for 2..32 rows on tcgen05 (k_predict_tc.cu):
// scores into p.s; the selection is launched by launch_predict.
bool predict_tc_supported(int B, int d, dv_dtype dt, const PredLaunch& p, int n_preds);
cudaError_t launch_predict_tc(const void* y, int B, int d, dv_dtype dt, const PredLaunch& p, int n_preds,
                              WsHeader* hdr, cudaStream_t stream);

// ---- sparse MLP (k_mlp.cu) ---------------------------------------------------

struct MlpLaunch {
  const void* y; int B, d, N;
  const void* W1n; const void* W2n;
  const int32_t* idx; int cap; const int32_t* count;
  float* out; int accumulate;
  // batch union scratch (B > 1)
  int32_t* U; int32_t* U_count; uint32_t* member;  // member [B][ceil(N/32)]
  // tensor-core path: activations split into two storage-type halves,
  // [32][tc_act_cols(N)] each
  void* act_hi; void* act_lo;
  // CUDA-core path: fp32 activations [B][cap] (B == 1) or [B][mlp_union_cap]
  float* act;
  // batch 1: arrival counters of the one-launch MLP (zero between calls)
  int* ctr;
  // tensor-core path: split-K partial tiles of the up-projection and their
  // arrival counts (tc_part_floats(min(N, B cap)) floats, one count per tile;
  // zero between calls)
  float* tc_part; int* tc_sem;
};

// Room for the batch union of B lists of up to `cap` neurons out of N.
int mlp_union_cap(int B, int N, int cap);

// Batches of at least this many rows use the tcgen05 paths (16-bit types);
// batch 1 has its own kernels.  Four rows on CUDA cores took 814 us per
// OPT-30B-shaped layer at half the units kept, 339 us on the tensor cores.
constexpr int kTcMinBatch = 2;
bool tc_mlp_supported(int B, int d, dv_dtype dt);
int tc_act_cols(int N);
// Floats of split-K partial tiles for up to max_rows rows (32 columns a tile).
size_t tc_part_floats(int max_rows);
cudaError_t launch_sparse_mlp_tc(const MlpLaunch& a, dv_dtype dt, WsHeader* hdr,
                                 cudaStream_t stream);

cudaError_t launch_sparse_mlp(const MlpLaunch& a, dv_dtype dt, WsHeader* hdr,
                              int num_sms, cudaStream_t stream);

// Batched attention on the tensor cores (k_mlp_tc.cu; 2+ rows, 16-bit, d a
// multiple of 128).  Projections of the union heads' Wqkv rows (`rows`,
// `rows_count` on the device, at most max_rows) with the current tokens: q
// of the member rows in fp32, K/V at pos rounded into the cache.
struct TcQkvLaunch {
  const void* y; int B, d, h, d_h, n_max, capQ;
  const void* Wqkv;
  const int32_t* rows; const int32_t* rows_count; int max_rows;
  const uint32_t* member; int words;
  const int32_t* slot_of; const int32_t* pos;
  float* q; void* K; void* V;
  float* part; int* sem;  // split-K partial tiles (tc_part_floats(max_rows)) and counts, zero between calls
};
cudaError_t launch_qkv_tc(const TcQkvLaunch& a, dv_dtype dt, WsHeader* hdr, cudaStream_t stream);
// out[b] += sum_k coef[b][k] W[rows[k]] with the coefficients split into two
// storage-type halves [32][Upad] (fp32 atomics into out).
struct TcRowsLaunch {
  const void* W; int n_rows, d, B;
  int rows_per_unit;  // rows are listed in contiguous runs of this many (a head's d_h rows)
  const int32_t* rows; const int32_t* rows_count; int max_rows;
  void* act_hi; void* act_lo; int Upad;
  float* out;
};
cudaError_t launch_rows_tc(const TcRowsLaunch& a, dv_dtype dt, WsHeader* hdr, cudaStream_t stream);

// Batch 1, streaming pass over the selected rows with bulk copies into a
// shared-memory ring (k_stream.cu); adds into out with atomics.
bool mlp_stream_supported(int d, dv_dtype dt);
// Batch 1: out += sum_u sum_t coef[u][t] W[units[u] * rpu + t] streamed the
// same way (the attention output projection of long rows).
cudaError_t launch_rows_stream(const void* W, const int32_t* units, const int32_t* n_units, int cap,
                               int n_rows_units, int rpu, int d, const float* coef, dv_dtype dt, float* out,
                               WsHeader* hdr, int num_sms, cudaStream_t stream);
cudaError_t launch_mlp_stream(const void* y, int d, int N, const void* W1n, const void* W2n,
                              const int32_t* list, const int32_t* count, int cap, dv_dtype dt, float* out,
                              WsHeader* hdr, int num_sms, int pdl, cudaStream_t stream);

// Weight-row lists of the union's units, written by the union kernel: for
// list q (rows[q] non-null), rows[q][k] = U[k / per[q]] * per[q] + k % per[q]
// for every unit of U, and count[q] = |U| per[q] (the attention's tensor-core
// projections: per = 3 d_h Wqkv rows and d_h W^O rows per head).
struct RowsExpand {
  int32_t* rows[2];
  int32_t* count[2];
  int per[2];
};
// Union of per-row index lists: U ascending, U_count, member bitmaps and
// (optional) slot_of[unit] = position of the unit in U; with `ex`, also its
// row lists (single-CTA path only, i.e. with `clear`).
cudaError_t launch_union(const int32_t* idx, int cap, const int32_t* count, int B,
                         int N, int32_t* U, int32_t* U_count, uint32_t* member,
                         int32_t* slot_of, WsHeader* hdr, cudaStream_t stream,
                         uint32_t* clear = nullptr, const RowsExpand* ex = nullptr);

// ---- attention (k_attn.cu) ---------------------------------------------------

struct AttnLaunch {
  const void* y; int B, d, h, d_h;
  const void* Wqkv; const void* Wo;
  void* K; void* V; void* X; uint8_t* valid; int n_max;
  const int32_t* pos;
  const int32_t* head_idx; int cap; const int32_t* head_count;  // per-row lists
  float scale;
  float* out; int accumulate;
  // scratch
  int32_t* U; int32_t* U_count; uint32_t* member; int32_t* slot_of;  // union (B > 1)
  float* q;                   // [B][capU][d_h]
  float* H;                   // [B][capU][d_h]
  // batches on the tensor-core path (B >= kTcMinBatch), else null
  int32_t* rows; int32_t* rows_count;   // expanded Wqkv rows of the union heads
  int32_t* rows_o; int32_t* rows_o_count;  // expanded W^O rows of the union heads
  uint32_t* need_bits; uint8_t* miss;   // repair plan
  void* act_hi; void* act_lo;           // [32][tc_act_cols(h * d_h)] output-projection coefficients
  float* tc_part; int* tc_sem;          // q/K/V split-K partial tiles and counts (zero between calls)
};


cudaError_t launch_sparse_attn(const AttnLaunch& a, dv_dtype dt, WsHeader* hdr,
                               int num_sms, cudaStream_t stream);
cudaError_t launch_kv_repair(const AttnLaunch& a, dv_dtype dt, WsHeader* hdr,
                             cudaStream_t stream);

// q/K/V of one token with the selected heads' KV repair on the tensor cores
// (k_qkv_tc.cu): batch 1, 16-bit storage, d_h 128, d a multiple of 64, at
// most 4096 cache positions.  Also appends the token (X[p], valid column p).
struct Qkv1Launch {
  const void* y; int d, h;
  const void* Wqkv;
  void* K; void* V; void* X; uint8_t* valid; int n_max;
  const int32_t* pos;
  const int32_t* U; const int32_t* U_count; int capU;  // the row's head list
  float* q;                                            // [capU][128]
  int pdl;                                             // launched with overlap
};
bool qkv1_tc_supported(int B, int d, int d_h, int n_max, dv_dtype dt);
cudaError_t launch_qkv1_tc(const Qkv1Launch& a, dv_dtype dt, WsHeader* hdr, cudaStream_t stream);

// Bulk K/V fill of the missing positions on the tensor cores (k_kv_tc.cu):
// 16-bit storage, d_h 64 or 128.
bool kv_tc_supported(int d, int d_h, dv_dtype dt);
cudaError_t launch_kv_repair_tc(const AttnLaunch& a, dv_dtype dt, WsHeader* hdr,
                                cudaStream_t stream);

// ---- true-sparsity labels (k_label.cu) ----------------------------------------

struct LabelLaunch {
  const void* X; int T, d;          // sequence [T][d], storage type
  const void* W1n; int N;           // neurons: W1n [N][d]
  const void* Wqkv; int h, d_h;     // heads: Wqkv [h][3][d_h][d]
  float scale;
  float* norms;                     // out: [N] or [h]
  // scratch
  float* partial;                   // per-tile sums of squares
  float* Q; void* K; void* V;       // heads: [h][T][d_h]
};
cudaError_t launch_label_neurons(const LabelLaunch& a, dv_dtype dt, WsHeader* hdr, cudaStream_t stream);
cudaError_t launch_label_heads(const LabelLaunch& a, dv_dtype dt, WsHeader* hdr, cudaStream_t stream);

// Top-k / threshold selection of rows of non-negative scores (k_predict.cu).
cudaError_t launch_select(const float* scores, int B, int N, int mode, int k, float t, int32_t* idx, int cap,
                          int32_t* count, WsHeader* hdr, cudaStream_t stream);

// ---- weighted sum of selected rows, column-sliced (k_rows.cu) -----------------

struct CombineLaunch {
  const void* W; int d;                  // rows of d elements, storage type
  const int32_t* units; const int32_t* n_units; int cap_units;
  int rpu;                               // rows per unit: row = units[u] * rpu + t
  int n_rows_units;                      // valid units are < n_rows_units
  const float* coef; size_t coef_stride; // coef[b * coef_stride + u * rpu + t]
  const uint32_t* member; int words;     // optional: unit must be in row b's set
  int B; float* out; int accumulate; WsHeader* hdr;
};
cudaError_t launch_rows_combine(const CombineLaunch& a, dv_dtype dt, cudaStream_t stream);

// ---- misc (k_misc.cu) --------------------------------------------------------

cudaError_t launch_layernorm(const float* x, int B, int d, float eps, void* y,
                             dv_dtype dt, cudaStream_t stream);
cudaError_t launch_positions_advance(int32_t* pos, int B, int lo, int hi,
                                     cudaStream_t stream);

}  // namespace dv

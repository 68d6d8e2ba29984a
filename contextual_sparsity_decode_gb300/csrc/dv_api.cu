// C ABI of libdv: argument validation, workspace layout and kernel launches.
// Every entry point checks its arguments on the host before launching
// anything and never synchronises (except dv_check).

#include <cstdint>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "dv_kernels.h"

using namespace dv;

namespace {

// A named NVTX range around each public call that enqueues work: profilers
// that collect NVTX (ncu --nvtx, nsys) see the library's calls by name;
// without one attached the push and pop are near no-ops.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

}  // namespace

namespace {

thread_local int g_last_cuda_error = 0;

}  // namespace

namespace dv {
dv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return DV_ERR_CUDA;
}
}  // namespace dv

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int vec_of(dv_dtype dt) { return dt == DV_F32 ? 4 : 8; }
bool dtype_ok(dv_dtype dt) { return dt == DV_F32 || dt == DV_F16 || dt == DV_BF16; }

// Sequential carving of 256-byte aligned regions out of a workspace.  With a
// null base it only measures.
struct Carver {
  char* base;
  size_t off = sizeof(WsHeader);
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
  size_t size() const { return (off + 255) & ~size_t(255); }
};

constexpr int kMaxB = 32;

// ---- workspace layouts --------------------------------------------------------

struct PredWs {
  float* h[2];
  float* s[2];
  uint16_t* h_hi[2];
  uint16_t* h_lo[2];
};
PredWs carve_pred(Carver& c, int B, int n_preds, const int* r, const int* N) {
  PredWs w{};
  for (int i = 0; i < n_preds; ++i) {
    w.h[i] = c.take<float>((size_t)B * r[i]);
    w.s[i] = c.take<float>((size_t)B * N[i]);
    if (B >= kTcMinBatch) {  // tensor-core path: h as two 16-bit halves, 32 rows
      w.h_hi[i] = c.take<uint16_t>((size_t)32 * r[i]);
      w.h_lo[i] = c.take<uint16_t>((size_t)32 * r[i]);
    }
  }
  return w;
}

struct MlpWs {
  int32_t* U;
  int32_t* U_count;
  uint32_t* member;
  uint16_t* act_hi;
  uint16_t* act_lo;
  float* act;
  int32_t* ctr;
  float* tc_part;
  int32_t* tc_sem;
};
MlpWs carve_mlp(Carver& c, int B, int N, int cap) {
  MlpWs w{};
  w.act = c.take<float>((size_t)B * (B == 1 ? cap : mlp_union_cap(B, N, cap)));
  w.U = c.take<int32_t>((size_t)N);
  w.U_count = c.take<int32_t>(4);
  w.member = c.take<uint32_t>((size_t)B * ((N + 31) / 32));
  if (B == 1) w.ctr = c.take<int32_t>(8);
  if (B >= kTcMinBatch) {
    w.act_hi = c.take<uint16_t>((size_t)32 * tc_act_cols(N));
    w.act_lo = c.take<uint16_t>((size_t)32 * tc_act_cols(N));
    const int maxU = mlp_union_cap(B, N, cap);
    w.tc_part = c.take<float>(tc_part_floats(maxU));
    w.tc_sem = c.take<int32_t>((size_t)tc_act_cols(maxU) / 128);
  }
  return w;
}

struct AttnWs {
  int32_t* U;
  int32_t* U_count;
  uint32_t* member;
  int32_t* slot_of;
  float* q;
  float* H;
  int32_t* rows;
  int32_t* rows_count;
  int32_t* rows_o;
  int32_t* rows_o_count;
  uint32_t* need_bits;
  uint8_t* miss;
  uint16_t* act_hi;
  uint16_t* act_lo;
  float* tc_part;
  int32_t* tc_sem;
};
AttnWs carve_attn(Carver& c, int B, int h, int d_h, int cap, int n_max) {
  AttnWs w{};
  const int capU = B == 1 ? cap : h;
  w.U = c.take<int32_t>((size_t)h);
  w.U_count = c.take<int32_t>(4);
  w.member = c.take<uint32_t>((size_t)B * ((h + 31) / 32));
  w.slot_of = c.take<int32_t>((size_t)h);
  w.q = c.take<float>((size_t)B * capU * d_h);
  w.H = c.take<float>((size_t)B * capU * d_h);
  if (B >= kTcMinBatch) {  // tensor-core path (16-bit types)
    w.rows = c.take<int32_t>((size_t)h * 3 * d_h);
    w.rows_count = c.take<int32_t>(4);
    w.rows_o = c.take<int32_t>((size_t)h * d_h);
    w.rows_o_count = c.take<int32_t>(4);
    w.need_bits = c.take<uint32_t>((size_t)(h + 31) / 32);
    w.miss = c.take<uint8_t>((size_t)B * h);
    w.act_hi = c.take<uint16_t>((size_t)32 * tc_act_cols(h * d_h));
    w.act_lo = c.take<uint16_t>((size_t)32 * tc_act_cols(h * d_h));
    w.tc_part = c.take<float>(tc_part_floats(h * 3 * d_h));
    w.tc_sem = c.take<int32_t>((size_t)tc_act_cols(h * 3 * d_h) / 128);
  }
  return w;
}

struct LabelWs {
  float* partial;
  float* Q;
  uint16_t* K;
  uint16_t* V;
};
// neurons: per-tile sums [ceil(T/256)][N]; heads: per-block sums
// [h][ceil(T/32)] and Q (fp32), K, V (16-bit) [h][T][d_h]
LabelWs carve_label(Carver& c, int T, int N, int h, int d_h, bool heads) {
  LabelWs w{};
  if (!heads) {
    w.partial = c.take<float>((size_t)((T + 255) / 256) * N);
  } else {
    w.partial = c.take<float>((size_t)h * ((T + 31) / 32));
    w.Q = c.take<float>((size_t)h * T * d_h);
    w.K = c.take<uint16_t>((size_t)h * T * d_h);
    w.V = c.take<uint16_t>((size_t)h * T * d_h);
  }
  return w;
}

// ---- validation ---------------------------------------------------------------------

dv_status check_pred(const void* y, int B, int d, dv_dtype dt, const dv_predictor* preds,
                     int n_preds) {
  if (!dtype_ok(dt)) return DV_ERR_DTYPE;
  if (!y || !aligned16(y) || !preds || n_preds < 1 || n_preds > 2) return DV_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxB || d < 1 || d > 16384 || d % vec_of(dt)) return DV_ERR_INVALID_ARG;
  for (int i = 0; i < n_preds; ++i) {
    const dv_predictor& p = preds[i];
    if (!p.P1t || !p.P2t || !p.idx || !p.count) return DV_ERR_INVALID_ARG;
    if (!aligned16(p.P1t) || !aligned16(p.P2t) || !aligned4(p.idx) || !aligned4(p.count))
      return DV_ERR_INVALID_ARG;
    if (p.scores && !aligned4(p.scores)) return DV_ERR_INVALID_ARG;
    if (p.r < 1 || p.r > 4096 || p.r % vec_of(dt)) return DV_ERR_INVALID_ARG;
    if (p.N < 1 || p.N > kSelectMaxN || p.cap < 1) return DV_ERR_INVALID_ARG;
    if (p.mode != DV_TOPK && p.mode != DV_THRESHOLD) return DV_ERR_INVALID_ARG;
    if (p.mode == DV_TOPK && (p.k < 0 || p.k > p.N || p.k > p.cap)) return DV_ERR_INVALID_ARG;
  }
  return DV_OK;
}

bool ws_ok(void* ws, size_t ws_bytes, size_t need) {
  return ws && aligned16(ws) && ws_bytes >= need;
}

}  // namespace

namespace {
dv_status check_attn(const void* y, int B, int d, int h, int d_h, const void* Wqkv,
                     const void* Wo, const dv_kv* kv, const int32_t* pos,
                     const int32_t* head_idx, int cap, const int32_t* head_count, dv_dtype dt,
                     bool need_y_wo) {
  if (!dtype_ok(dt)) return DV_ERR_DTYPE;
  if (!Wqkv || !kv || !pos || !head_idx || !head_count) return DV_ERR_INVALID_ARG;
  if (need_y_wo && (!y || !Wo || !aligned16(y) || !aligned16(Wo))) return DV_ERR_INVALID_ARG;
  if (!kv->K || !kv->V || !kv->X || !kv->valid) return DV_ERR_INVALID_ARG;
  if (!aligned16(Wqkv) || !aligned16(kv->K) || !aligned16(kv->V) || !aligned16(kv->X) ||
      !aligned16(kv->valid) || !aligned4(pos) || !aligned4(head_idx) || !aligned4(head_count))
    return DV_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxB || d < 1 || d % vec_of(dt) || h < 1 || h > 1024) return DV_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return DV_ERR_UNSUPPORTED;
  // one projection row must fit a 40 KB shared-memory stage of attn_qkv
  if ((size_t)d * (dt == DV_F32 ? 4 : 2) > 40960) return DV_ERR_UNSUPPORTED;
  if (cap < 1 || cap > h) return DV_ERR_INVALID_ARG;
  if (kv->n_max < 16 || kv->n_max > 65536 || kv->n_max % 16) return DV_ERR_INVALID_ARG;
  return DV_OK;
}

AttnLaunch make_attn(const void* y, int B, int d, int h, int d_h, const void* Wqkv, const void* Wo,
                     const dv_kv* kv, const int32_t* pos, const int32_t* head_idx, int cap,
                     const int32_t* head_count, float scale, float* out, int accumulate,
                     const AttnWs& w) {
  AttnLaunch L{};
  L.y = y; L.B = B; L.d = d; L.h = h; L.d_h = d_h; L.Wqkv = Wqkv; L.Wo = Wo;
  L.K = kv->K; L.V = kv->V; L.X = kv->X; L.valid = kv->valid; L.n_max = kv->n_max;
  L.pos = pos; L.head_idx = head_idx; L.cap = cap; L.head_count = head_count;
  L.scale = scale; L.out = out; L.accumulate = accumulate ? 1 : 0;
  L.U = w.U; L.U_count = w.U_count; L.member = w.member; L.slot_of = w.slot_of;
  L.q = w.q; L.H = w.H;
  L.rows = w.rows; L.rows_count = w.rows_count; L.need_bits = w.need_bits; L.miss = w.miss;
  L.rows_o = w.rows_o; L.rows_o_count = w.rows_o_count;
  L.act_hi = w.act_hi; L.act_lo = w.act_lo;
  L.tc_part = w.tc_part; L.tc_sem = w.tc_sem;
  return L;
}
}  // namespace

extern "C" {

const char* dv_status_str(dv_status s) {
  switch (s) {
    case DV_OK: return "ok";
    case DV_ERR_INVALID_ARG: return "invalid argument";
    case DV_ERR_DTYPE: return "unsupported data type";
    case DV_ERR_WORKSPACE: return "workspace missing or too small";
    case DV_ERR_CUDA: return "CUDA error";
    case DV_ERR_INDEX_RANGE: return "index out of range (skipped on the device)";
    case DV_ERR_TIMEOUT: return "device wait timed out";
    case DV_ERR_UNSUPPORTED: return "shape not supported";
    case DV_ERR_CAPACITY: return "list longer than its capacity (truncated)";
    case DV_ERR_POSITION: return "position outside the KV cache";
  }
  return "unknown status";
}

int dv_last_cuda_error(void) { return g_last_cuda_error; }

int dv_version(void) { return 100; }

int dv_set_launch_overlap(int level) { return set_launch_overlap(level); }

long long dv_set_wait_limit_ns(long long ns) { return set_wait_limit_ns(ns); }

long long dv_kernel_launches(void) { return launches_total(); }

dv_status dv_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes < sizeof(WsHeader)) return DV_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_check(void* ws, cudaStream_t stream, int* info) {
  if (!ws) return DV_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int hv[2] = {0, 0};
  e = cudaMemcpy(hv, ws, sizeof(hv), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (info) *info = hv[1];
  if (hv[0] != 0) {
    e = cudaMemset(ws, 0, sizeof(hv));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return (dv_status)hv[0];
}

// ---- predictor ------------------------------------------------------------------------

dv_status dv_predict_workspace_size(int B, int n_preds, int r_max, int N_max, size_t* bytes) {
  if (!bytes || B < 1 || B > kMaxB || n_preds < 1 || n_preds > 2 || r_max < 1 || N_max < 1)
    return DV_ERR_INVALID_ARG;
  Carver c(nullptr);
  const int r[2] = {r_max, r_max}, N[2] = {N_max, N_max};
  carve_pred(c, B, n_preds, r, N);
  *bytes = c.size();
  return DV_OK;
}

dv_status dv_predict(const void* y, int B, int d, dv_dtype dt, const dv_predictor* preds,
                     int n_preds, void* ws, size_t ws_bytes, cudaStream_t stream) {
  Range nvtx_range("dv_predict");
  dv_status st = check_pred(y, B, d, dt, preds, n_preds);
  if (st != DV_OK) return st;
  int r[2] = {0, 0}, N[2] = {0, 0};
  for (int i = 0; i < n_preds; ++i) { r[i] = preds[i].r; N[i] = preds[i].N; }
  Carver meas(nullptr);
  carve_pred(meas, B, n_preds, r, N);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  PredWs w = carve_pred(c, B, n_preds, r, N);
  PredLaunch L{};
  for (int i = 0; i < n_preds; ++i) {
    const dv_predictor& p = preds[i];
    L.P1t[i] = p.P1t; L.P2t[i] = p.P2t; L.r[i] = p.r; L.N[i] = p.N;
    L.mode[i] = (int)p.mode; L.k[i] = p.k; L.t[i] = p.t;
    L.idx[i] = p.idx; L.cap[i] = p.cap; L.count[i] = p.count;
    L.h[i] = w.h[i];
    L.h_hi[i] = w.h_hi[i];
    L.h_lo[i] = w.h_lo[i];
    L.s[i] = p.scores ? p.scores : w.s[i];
  }
  cudaError_t e = launch_predict(y, B, d, dt, L, n_preds, static_cast<WsHeader*>(ws), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_lookahead(const void* y, int B, int d, dv_dtype dt, const dv_predictor* preds,
                       int n_preds, void* ws, size_t ws_bytes, cudaEvent_t input_ready,
                       cudaStream_t side, cudaEvent_t done) {
  Range nvtx_range("dv_lookahead");
  dv_status st = check_pred(y, B, d, dt, preds, n_preds);
  if (st != DV_OK) return st;
  if (input_ready) {
    cudaError_t e = cudaStreamWaitEvent(side, input_ready, 0);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  st = dv_predict(y, B, d, dt, preds, n_preds, ws, ws_bytes, side);
  if (st != DV_OK) return st;
  if (done) {
    cudaError_t e = cudaEventRecord(done, side);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return DV_OK;
}

// ---- sparse MLP -------------------------------------------------------------------------

dv_status dv_sparse_mlp_workspace_size(int B, int d, int N, int cap, size_t* bytes) {
  if (!bytes || B < 1 || B > kMaxB || d < 1 || N < 1 || cap < 1) return DV_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_mlp(c, B, N, cap);
  *bytes = c.size();
  return DV_OK;
}

dv_status dv_sparse_mlp(const void* y, int B, int d, int N, const void* W1n, const void* W2n,
                        const int32_t* idx, int cap, const int32_t* count, dv_dtype dt,
                        float* out, int accumulate, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  Range nvtx_range("dv_sparse_mlp");
  if (!dtype_ok(dt)) return DV_ERR_DTYPE;
  if (!y || !W1n || !W2n || !idx || !count || !out) return DV_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(W1n) || !aligned16(W2n) || !aligned16(out) ||
      !aligned4(idx) || !aligned4(count))
    return DV_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxB || d < 1 || d % vec_of(dt) || N < 1 || N > 65536 || cap < 1)
    return DV_ERR_INVALID_ARG;
  Carver meas(nullptr);
  carve_mlp(meas, B, N, cap);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  MlpWs w = carve_mlp(c, B, N, cap);
  MlpLaunch L{};
  L.y = y; L.B = B; L.d = d; L.N = N; L.W1n = W1n; L.W2n = W2n;
  L.idx = idx; L.cap = cap; L.count = count; L.out = out; L.accumulate = accumulate ? 1 : 0;
  L.U = w.U; L.U_count = w.U_count; L.member = w.member;
  L.act_hi = w.act_hi; L.act_lo = w.act_lo; L.act = w.act; L.ctr = w.ctr;
  L.tc_part = w.tc_part; L.tc_sem = w.tc_sem;
  cudaError_t e = launch_sparse_mlp(L, dt, static_cast<WsHeader*>(ws), num_sms_current(), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

// ---- attention ----------------------------------------------------------------------------

dv_status dv_sparse_attn_workspace_size(int B, int d, int h, int d_h, int cap, int n_max,
                                        size_t* bytes) {
  if (!bytes || B < 1 || B > kMaxB || d < 1 || h < 1 || d_h < 1 || cap < 1 || n_max < 1)
    return DV_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_attn(c, B, h, d_h, cap, n_max);
  *bytes = c.size();
  return DV_OK;
}


dv_status dv_sparse_attn(const void* y, int B, int d, int h, int d_h, const void* Wqkv,
                         const void* Wo, const dv_kv* kv, const int32_t* pos,
                         const int32_t* head_idx, int cap, const int32_t* head_count, float scale,
                         dv_dtype dt, float* out, int accumulate, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  Range nvtx_range("dv_sparse_attn");
  dv_status st = check_attn(y, B, d, h, d_h, Wqkv, Wo, kv, pos, head_idx, cap, head_count, dt, true);
  if (st != DV_OK) return st;
  if (!out || !aligned16(out)) return DV_ERR_INVALID_ARG;
  Carver meas(nullptr);
  carve_attn(meas, B, h, d_h, cap, kv->n_max);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  AttnWs w = carve_attn(c, B, h, d_h, cap, kv->n_max);
  AttnLaunch L = make_attn(y, B, d, h, d_h, Wqkv, Wo, kv, pos, head_idx, cap, head_count, scale,
                           out, accumulate, w);
  cudaError_t e = launch_sparse_attn(L, dt, static_cast<WsHeader*>(ws), num_sms_current(), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_kv_repair(const dv_kv* kv, int B, int d, int h, int d_h, const void* Wqkv,
                       const int32_t* pos, const int32_t* head_idx, int cap,
                       const int32_t* head_count, dv_dtype dt, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  Range nvtx_range("dv_kv_repair");
  dv_status st = check_attn(nullptr, B, d, h, d_h, Wqkv, nullptr, kv, pos, head_idx, cap, head_count,
                            dt, false);
  if (st != DV_OK) return st;
  Carver meas(nullptr);
  carve_attn(meas, B, h, d_h, cap, kv->n_max);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  AttnWs w = carve_attn(c, B, h, d_h, cap, kv->n_max);
  AttnLaunch L = make_attn(nullptr, B, d, h, d_h, Wqkv, nullptr, kv, pos, head_idx, cap, head_count,
                           1.f, nullptr, 0, w);
  cudaError_t e = launch_kv_repair(L, dt, static_cast<WsHeader*>(ws), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

// ---- true-sparsity labels ----------------------------------------------------------------------

dv_status dv_label_workspace_size(int T, int d, int N, int h, int d_h, size_t* bytes) {
  if (!bytes || T < 1 || d < 1 || N < 0 || h < 0 || d_h < 0) return DV_ERR_INVALID_ARG;
  Carver a(nullptr), b(nullptr);
  carve_label(a, T, N, h, d_h, false);
  carve_label(b, T, N, h, d_h, true);
  *bytes = a.size() > b.size() ? a.size() : b.size();
  return DV_OK;
}

namespace {
dv_status check_label(const void* X, int T, int d, dv_dtype dt, const float* norms, void* ws) {
  if (!dtype_ok(dt)) return DV_ERR_DTYPE;
  if (dt == DV_F32) return DV_ERR_DTYPE;  // tensor-core products: 16-bit storage
  if (!X || !norms || !ws || !aligned16(X) || !aligned4(norms) || !aligned16(ws)) return DV_ERR_INVALID_ARG;
  if (T < 1 || T > (1 << 20) || d < 8 || d % 8 || d > 65536) return DV_ERR_INVALID_ARG;
  return DV_OK;
}
}  // namespace

dv_status dv_label_neurons(const void* X, int T, int d, int N, const void* W1n, dv_dtype dt, float* norms,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  Range nvtx_range("dv_label_neurons");
  dv_status st = check_label(X, T, d, dt, norms, ws);
  if (st != DV_OK) return st;
  if (!W1n || !aligned16(W1n) || N < 1) return DV_ERR_INVALID_ARG;
  Carver meas(nullptr);
  carve_label(meas, T, N, 0, 0, false);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  LabelWs w = carve_label(c, T, N, 0, 0, false);
  LabelLaunch L{};
  L.X = X; L.T = T; L.d = d; L.W1n = W1n; L.N = N; L.norms = norms; L.partial = w.partial;
  cudaError_t e = launch_label_neurons(L, dt, static_cast<WsHeader*>(ws), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_label_heads(const void* X, int T, int d, int h, int d_h, const void* Wqkv, float scale,
                         dv_dtype dt, float* norms, void* ws, size_t ws_bytes, cudaStream_t stream) {
  Range nvtx_range("dv_label_heads");
  dv_status st = check_label(X, T, d, dt, norms, ws);
  if (st != DV_OK) return st;
  if (!Wqkv || !aligned16(Wqkv) || h < 1 || h > 1024) return DV_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return DV_ERR_UNSUPPORTED;
  Carver meas(nullptr);
  carve_label(meas, T, 0, h, d_h, true);
  if (!ws_ok(ws, ws_bytes, meas.size())) return DV_ERR_WORKSPACE;
  Carver c(ws);
  LabelWs w = carve_label(c, T, 0, h, d_h, true);
  LabelLaunch L{};
  L.X = X; L.T = T; L.d = d; L.Wqkv = Wqkv; L.h = h; L.d_h = d_h; L.scale = scale; L.norms = norms;
  L.partial = w.partial; L.Q = w.Q; L.K = w.K; L.V = w.V;
  cudaError_t e = launch_label_heads(L, dt, static_cast<WsHeader*>(ws), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_select_scores(const float* scores, int B, int N, dv_select mode, int k, float t, int32_t* idx, int cap,
                    int32_t* count, void* ws, size_t ws_bytes, cudaStream_t stream) {
  Range nvtx_range("dv_select_scores");
  if (!scores || !idx || !count || !aligned4(scores) || !aligned4(idx) || !aligned4(count))
    return DV_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kSelectMaxN || cap < 1) return DV_ERR_INVALID_ARG;
  if (mode != DV_TOPK && mode != DV_THRESHOLD) return DV_ERR_INVALID_ARG;
  if (mode == DV_TOPK && (k < 0 || k > N || k > cap)) return DV_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, sizeof(WsHeader))) return DV_ERR_WORKSPACE;
  cudaError_t e = launch_select(scores, B, N, (int)mode, k, t, idx, cap, count, static_cast<WsHeader*>(ws), stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

// ---- helpers ----------------------------------------------------------------------------------

dv_status dv_layernorm(const float* x, int B, int d, float eps, void* y, dv_dtype dt,
                       cudaStream_t stream) {
  Range nvtx_range("dv_layernorm");
  if (!dtype_ok(dt)) return DV_ERR_DTYPE;
  if (!x || !y || B < 1 || d < 4 || d > 16384 || d % 4 || !(eps >= 0.f)) return DV_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 7u)) return DV_ERR_INVALID_ARG;
  cudaError_t e = launch_layernorm(x, B, d, eps, y, dt, stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

dv_status dv_positions_advance(int32_t* pos, int B, int lo, int hi, cudaStream_t stream) {
  Range nvtx_range("dv_positions_advance");
  if (!pos || B < 1 || lo < 0 || hi <= lo) return DV_ERR_INVALID_ARG;
  cudaError_t e = launch_positions_advance(pos, B, lo, hi, stream);
  return e == cudaSuccess ? DV_OK : cuda_fail(e);
}

}  // extern "C"

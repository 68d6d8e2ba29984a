// dv_predict_static: the sparsity predictor with its scratch space in a
// fixed, library-owned device array instead of a caller workspace, for
// callers that cannot allocate device memory.  Everything else (kernels,
// arithmetic, outputs) is the dv_predict path.

#include <cstdint>
#include <mutex>

#include "dv_kernels.h"

namespace {

using dv::kMaxDevices;
constexpr int kStaticMaxB = 4;
constexpr int kStaticMaxR = 1024;
constexpr int kStaticMaxN = 32768;

// header + two predictors' hidden [B][r] and score [B][N] fp32 rows, each
// region 256-byte aligned
constexpr size_t kStaticBytes =
    sizeof(dv::WsHeader) + 2 * ((size_t)kStaticMaxB * kStaticMaxR * 4 + 256) +
    2 * ((size_t)kStaticMaxB * kStaticMaxN * 4 + 256);

// One copy per device that loads the library; it lives until the process
// exits.  Host code must not use this name as a device address: the device
// address is obtained per device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_predict_scratch[kStaticBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" dv_status dv_predict_static(const void* y, int B, int d, dv_dtype dt,
                                       const dv_predictor* preds, int n_preds,
                                       cudaStream_t stream) {
  // argument checks (the same rules as dv_predict) plus the static limits
  if (dt != DV_F32 && dt != DV_F16 && dt != DV_BF16) return DV_ERR_DTYPE;
  const int vec = dt == DV_F32 ? 4 : 8;
  if (!y || (reinterpret_cast<uintptr_t>(y) & 15u) || !preds || n_preds < 1 || n_preds > 2)
    return DV_ERR_INVALID_ARG;
  if (B < 1 || d < 1 || d > 16384 || d % vec) return DV_ERR_INVALID_ARG;
  for (int i = 0; i < n_preds; ++i) {
    const dv_predictor& p = preds[i];
    if (!p.P1t || !p.P2t || !p.idx || !p.count) return DV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p.P1t) & 15u) || (reinterpret_cast<uintptr_t>(p.P2t) & 15u) ||
        (reinterpret_cast<uintptr_t>(p.idx) & 3u) || (reinterpret_cast<uintptr_t>(p.count) & 3u) ||
        (reinterpret_cast<uintptr_t>(p.scores) & 3u))
      return DV_ERR_INVALID_ARG;
    if (p.r < 1 || p.r % vec || p.N < 1 || p.cap < 1) return DV_ERR_INVALID_ARG;
    if (p.mode != DV_TOPK && p.mode != DV_THRESHOLD) return DV_ERR_INVALID_ARG;
    if (p.mode == DV_TOPK && (p.k < 0 || p.k > p.N || p.k > p.cap)) return DV_ERR_INVALID_ARG;
    if (p.r > kStaticMaxR || p.N > kStaticMaxN) return DV_ERR_WORKSPACE;  // beyond the fixed array
  }
  if (B > kStaticMaxB) return DV_ERR_WORKSPACE;

  // per-device set-up: the array's device address, looked up once with the
  // device current
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dv::cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return dv::cuda_fail(cudaErrorInvalidDevice);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_predict_scratch);
      if (e != cudaSuccess) return dv::cuda_fail(e);
      if (!p) return dv::cuda_fail(cudaErrorInvalidSymbol);
      g_addr[dev] = p;
    }
    base = g_addr[dev];
  }

  // carve the hidden / score rows after the header; clear the error word
  char* cur = static_cast<char*>(base) + sizeof(dv::WsHeader);
  dv::PredLaunch L{};
  for (int i = 0; i < n_preds; ++i) {
    const dv_predictor& p = preds[i];
    L.P1t[i] = p.P1t; L.P2t[i] = p.P2t; L.r[i] = p.r; L.N[i] = p.N;
    L.mode[i] = (int)p.mode; L.k[i] = p.k; L.t[i] = p.t;
    L.idx[i] = p.idx; L.cap[i] = p.cap; L.count[i] = p.count;
    L.h[i] = reinterpret_cast<float*>(cur);
    cur += align256((size_t)B * p.r * sizeof(float));
    float* s_scratch = reinterpret_cast<float*>(cur);
    cur += align256((size_t)B * p.N * sizeof(float));
    L.s[i] = p.scores ? p.scores : s_scratch;
  }
  if ((size_t)(cur - static_cast<char*>(base)) > kStaticBytes) return DV_ERR_WORKSPACE;
  e = cudaMemsetAsync(base, 0, sizeof(dv::WsHeader), stream);
  if (e != cudaSuccess) return dv::cuda_fail(e);
  e = dv::launch_predict(y, B, d, dt, L, n_preds, static_cast<dv::WsHeader*>(base), stream);
  return e == cudaSuccess ? DV_OK : dv::cuda_fail(e);
}

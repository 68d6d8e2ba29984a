// Sparsity predictor: two-layer MLP with a sigmoid per unit, then top-k or
// threshold selection.  Follows "用Deja Vu来提高 LLM 的推理速度" §2 (稀疏性预测)
// and the Deja Vu reading notes, "Sparsity operator for MLP / Attention".
//
// Launch 1 (predict_gemv<ReLU>):    h = ReLU(y P1)       both predictors
// Launch 2 (predict_gemv<Sigmoid>): s = sigmoid(h P2)    both predictors
// Launch 3 (select_kernel):         index lists, one CTA per (predictor, row)
//
// Both GEMVs are HBM-bound row streams: one warp per weight row, 16-byte
// read-only loads, four loads in flight per lane, fp32 accumulation and a
// shuffle reduction.  h and s stay fp32.

#include "dv_kernels.h"

namespace dv {
namespace {

enum Epi { kRelu = 0, kSigmoid = 1 };

struct GemvSeg {
  const void* W;   // [rows][K], storage type T
  const void* x;   // [B][K], XT
  float* out;      // [B][rows]
  int rows, K;
};
struct GemvArgs {
  GemvSeg seg[2];
  int nseg;
  int total_rows;
  int B;
};

template <typename T, typename XT, int EPI, int BT>
__global__ void __launch_bounds__(256) predict_gemv(GemvArgs a, int b0) {
  constexpr int V = Elem<T>::kVec;
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int gr = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gr < a.total_rows;
       gr += warps_total) {
    // pick the segment with selects (no dynamic indexing of the parameter block)
    const bool s1 = a.nseg > 1 && gr >= a.seg[0].rows;
    const int K = s1 ? a.seg[1].K : a.seg[0].K;
    const int rows = s1 ? a.seg[1].rows : a.seg[0].rows;
    const void* Wp = s1 ? a.seg[1].W : a.seg[0].W;
    const void* xp = s1 ? a.seg[1].x : a.seg[0].x;
    float* outp = s1 ? a.seg[1].out : a.seg[0].out;
    const int row = gr - (s1 ? a.seg[0].rows : 0);
    const int C = K / V;
    const T* wrow = static_cast<const T*>(Wp) + (size_t)row * K;
    const XT* xb = static_cast<const XT*>(xp) + (size_t)b0 * K;
    float acc[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) acc[b] = 0.f;
    const int nb = min(BT, a.B - b0);
    for (int c0 = lane; c0 < C; c0 += 32 * U) {
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c < C) w[u] = ld_stream(wrow + (size_t)c * V);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c < C) {
          float wf[V];
          unpack<T>(w[u], wf);
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            if (b < nb) {
              float xf[V];
              const XT* xr = xb + (size_t)b * K + (size_t)c * V;
              if constexpr (sizeof(XT) == sizeof(T)) {
                unpack<T>(ld_cached(xr), xf);
              } else {  // fp32 activations against 16-bit weights: 2 x 16 B
                const uint4 lo = ld_cached(xr), hi = ld_cached(xr + 4);
                unpack<float>(lo, xf);
                unpack<float>(hi, xf + 4);
              }
#pragma unroll
              for (int v = 0; v < V; ++v) acc[b] = fmaf(wf[v], xf[v], acc[b]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float z = warp_sum(acc[b]);
      if (lane == 0 && b < nb) {
        float o = (EPI == kRelu) ? fmaxf(z, 0.f) : 1.f / (1.f + expf(-z));
        outp[(size_t)(b0 + b) * rows + row] = o;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// selection

struct SelArgs {
  const float* s[2];
  int N[2], mode[2], k[2], cap[2];
  float t[2];
  int32_t* idx[2];
  int32_t* count[2];
};

constexpr int kSelThreads = 1024;

// Add 1 to hist[bin] for every active lane, one shared-memory atomic per
// distinct bin in the warp (scores cluster in few bins of the top digits).
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool act) {
  const uint32_t key = act ? bin : 0xffffffffu;
  const unsigned grp = __match_any_sync(0xffffffffu, key);
  const int lane = threadIdx.x & 31;
  if (act && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
}

// One CTA per (predictor, batch row).  The row's scores are staged in shared
// memory; thread t owns the contiguous element range [t*E, (t+1)*E) with E
// odd, so a warp's reads of element t*E+e hit 32 distinct banks.  Because
// ranges are contiguous and in thread order, a block prefix sum of per-thread
// counts gives every selected element its slot in the ascending output.
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a, WsHeader* hdr) {
  extern __shared__ uint32_t keys[];
  __shared__ int tmp[32];
  __shared__ int hist[256];
  __shared__ int sel_digit, sel_greater;
  const int b = blockIdx.x;
  const bool p1 = blockIdx.y != 0;
  const int N = p1 ? a.N[1] : a.N[0];
  const int mode = p1 ? a.mode[1] : a.mode[0];
  const int k = p1 ? a.k[1] : a.k[0];
  const int cap = p1 ? a.cap[1] : a.cap[0];
  const float thr = p1 ? a.t[1] : a.t[0];
  int32_t* count = p1 ? a.count[1] : a.count[0];
  const float* s = (p1 ? a.s[1] : a.s[0]) + (size_t)b * N;
  int32_t* out = (p1 ? a.idx[1] : a.idx[0]) + (size_t)b * cap;
  // Scores are sigmoid outputs in [0, 1]: their IEEE bits order like the values.
  for (int i = threadIdx.x; i < N; i += kSelThreads) keys[i] = __float_as_uint(s[i]);
  __syncthreads();
  const int E = ((N + kSelThreads - 1) / kSelThreads) | 1;
  const int i0 = min(N, threadIdx.x * E);
  const int i1 = min(N, i0 + E);

  int total;
  if (mode == DV_THRESHOLD) {
    const float t = thr;
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += __uint_as_float(keys[i]) > t;
    const int incl = block_inclusive_scan<kSelThreads>(mine, tmp, &total);
    int o = incl - mine;
    for (int i = i0; i < i1; ++i)
      if (__uint_as_float(keys[i]) > t) {
        if (o < cap) out[o] = i;
        ++o;
      }
    if (threadIdx.x == 0) {
      count[b] = min(total, cap);
      if (total > cap) set_error(hdr, DV_ERR_CAPACITY, total);
    }
    return;
  }

  // top-k
  if (k <= 0 || k >= N) {
    if (k >= N)
      for (int i = threadIdx.x; i < N; i += kSelThreads) out[i] = i;
    if (threadIdx.x == 0) count[b] = k >= N ? N : 0;
    return;
  }
  // Radix select (most significant digit first, 8-bit digits) of the k-th
  // largest key T; `remaining` counts how many keys equal to T are taken.
  uint32_t prefix = 0, pmask = 0;
  int remaining = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (threadIdx.x < 256) hist[threadIdx.x] = 0;
    __syncthreads();
    for (int e = 0; e < E; ++e) {  // E is uniform: warps stay converged for match.any
      const int i = i0 + e;
      const uint32_t kv = keys[min(i, N - 1)];
      hist_add(hist, (kv >> shift) & 255u, i < i1 && (kv & pmask) == prefix);
    }
    __syncthreads();
    const int v = threadIdx.x < 256 ? hist[255 - threadIdx.x] : 0;
    const int incl = block_inclusive_scan<kSelThreads>(v, tmp, &total);
    if (threadIdx.x < 256 && incl >= remaining && incl - v < remaining) {
      sel_digit = 255 - threadIdx.x;
      sel_greater = incl - v;
    }
    __syncthreads();
    remaining -= sel_greater;
    prefix |= (uint32_t)sel_digit << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) { gt += keys[i] > T; eq += keys[i] == T; }
  const int eq_incl = block_inclusive_scan<kSelThreads>(eq, tmp, &total);
  const int eq_before = eq_incl - eq;
  const int take_eq = max(0, min(eq, remaining - eq_before));
  const int mine = gt + take_eq;
  const int tk_incl = block_inclusive_scan<kSelThreads>(mine, tmp, &total);
  int o = tk_incl - mine;
  int eq_seen = 0;
  for (int i = i0; i < i1; ++i) {
    bool take = keys[i] > T;
    if (keys[i] == T) { take = eq_seen < take_eq; ++eq_seen; }
    if (take) out[o++] = i;
  }
  if (threadIdx.x == 0) count[b] = k;
}

template <typename T, typename XT, int EPI>
cudaError_t run_gemv(const GemvArgs& a, cudaStream_t stream) {
  const int grid = (a.total_rows + 7) / 8;  // one warp per row, 8 warps per CTA
  for (int b0 = 0; b0 < a.B;) {
    const int nb = a.B - b0;
    const int bt = nb >= 8 ? 8 : (nb >= 4 ? 4 : (nb >= 2 ? 2 : 1));
    switch (bt) {
      case 8: predict_gemv<T, XT, EPI, 8><<<grid, 256, 0, stream>>>(a, b0); break;
      case 4: predict_gemv<T, XT, EPI, 4><<<grid, 256, 0, stream>>>(a, b0); break;
      case 2: predict_gemv<T, XT, EPI, 2><<<grid, 256, 0, stream>>>(a, b0); break;
      default: predict_gemv<T, XT, EPI, 1><<<grid, 256, 0, stream>>>(a, b0); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t predict_t(const void* y, int B, int d, const PredLaunch& p, int n_preds,
                      WsHeader* hdr, cudaStream_t stream) {
  GemvArgs g1{};
  g1.nseg = n_preds;
  g1.B = B;
  g1.total_rows = 0;
  for (int i = 0; i < n_preds; ++i) {
    g1.seg[i] = GemvSeg{p.P1t[i], y, p.h[i], p.r[i], d};
    g1.total_rows += p.r[i];
  }
  cudaError_t e = run_gemv<T, T, kRelu>(g1, stream);
  if (e != cudaSuccess) return e;

  GemvArgs g2{};
  g2.nseg = n_preds;
  g2.B = B;
  g2.total_rows = 0;
  for (int i = 0; i < n_preds; ++i) {
    g2.seg[i] = GemvSeg{p.P2t[i], p.h[i], p.s[i], p.N[i], p.r[i]};
    g2.total_rows += p.N[i];
  }
  e = run_gemv<T, float, kSigmoid>(g2, stream);
  if (e != cudaSuccess) return e;

  SelArgs sa{};
  int nmax = 0;
  for (int i = 0; i < n_preds; ++i) {
    sa.s[i] = p.s[i]; sa.N[i] = p.N[i]; sa.mode[i] = p.mode[i]; sa.k[i] = p.k[i];
    sa.cap[i] = p.cap[i]; sa.t[i] = p.t[i]; sa.idx[i] = p.idx[i]; sa.count[i] = p.count[i];
    nmax = p.N[i] > nmax ? p.N[i] : nmax;
  }
  const size_t smem = (size_t)nmax * sizeof(uint32_t);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t ea = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)(kSelectMaxN * sizeof(uint32_t)));
    if (ea != cudaSuccess) return ea;
    attr_set = true;
  }
  select_kernel<<<dim3(B, n_preds), kSelThreads, smem, stream>>>(sa, hdr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_predict(const void* y, int B, int d, dv_dtype dt, const PredLaunch& p,
                           int n_preds, WsHeader* hdr, cudaStream_t stream) {
  switch (dt) {
    case DV_F32: return predict_t<float>(y, B, d, p, n_preds, hdr, stream);
    case DV_F16: return predict_t<__half>(y, B, d, p, n_preds, hdr, stream);
    case DV_BF16: return predict_t<__nv_bfloat16>(y, B, d, p, n_preds, hdr, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

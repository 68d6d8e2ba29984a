// Sparsity predictor: two-layer MLP with a sigmoid per unit, then top-k or
// threshold selection.  Follows "用Deja Vu来提高 LLM 的推理速度" §2 (稀疏性预测)
// and the Deja Vu reading notes, "Sparsity operator for MLP / Attention".
//
// Launch 1 (rows_dot<ReLU>):    h = ReLU(y P1)       both predictors
// Launch 2 (rows_dot<Sigmoid>): s = sigmoid(h P2)    both predictors
// Launch 3 (select_kernel):     index lists, one CTA per (predictor, row)
// Batches of 2..32 rows in 16-bit types run launches 1 and 2 on the tensor
// cores instead (k_predict_tc.cu).
//
// Both GEMVs are HBM-bound row streams.  A CTA owns a tile of rows; a group
// of TPR threads (32..256) shares one row, each thread holding up to kC
// 16-byte chunks of up to kR rows.  Every weight load of a thread is issued
// before the first one is used, so a CTA keeps kR x kC x 16 B per thread in
// flight (the probe of this design on GB300: ~1.9 us + bytes / 7.1 TB/s per
// launch inside a graph).  Reductions run in a fixed order, so scores are
// reproducible run to run.  h and s stay fp32.

#include "dv_kernels.h"

namespace dv {
namespace {

enum Epi { kRelu = 0, kSigmoid = 1 };

constexpr int kThreads = 256;
constexpr int kC = 4;   // chunks per thread per pass
constexpr int kR = 3;   // rows per thread group

struct RowSeg {
  const void* W;   // [rows][K], storage type T
  const void* x;   // [B][K], XT
  float* out;      // [B][rows]
  int rows, K;
  int tpr_log2;    // threads per row (log2)
  int cta0;        // first CTA of the segment
};
struct RowArgs {
  RowSeg seg[2];
  int nseg;
  int B, b0;
  int pdl;  // launched programmatically: x is the predecessor's output
};

// Threads per row: the smallest power of two in [32, 256] covering the row's
// chunks in one pass of kC chunks per thread (256 when none does).
int tpr_log2_for(int chunks) {
  int l = 5;
  while (l < 8 && (1 << l) * kC < chunks) ++l;
  return l;
}
int rows_per_cta(int tpr_log2) { return (kThreads >> tpr_log2) * kR; }

template <typename T, typename XT, int EPI, int BT>
__global__ void __launch_bounds__(kThreads) rows_dot(RowArgs a) {
  constexpr int V = Elem<T>::kVec;
  __shared__ float red[kThreads / 32][kR][BT];
  // segment fields picked with selects (no dynamic indexing of the parameter block)
  const bool s1 = a.nseg > 1 && (int)blockIdx.x >= a.seg[1].cta0;
  const T* W = static_cast<const T*>(s1 ? a.seg[1].W : a.seg[0].W);
  const XT* x = static_cast<const XT*>(s1 ? a.seg[1].x : a.seg[0].x);
  float* out = s1 ? a.seg[1].out : a.seg[0].out;
  const int rows = s1 ? a.seg[1].rows : a.seg[0].rows;
  const int K = s1 ? a.seg[1].K : a.seg[0].K;
  const int tl = s1 ? a.seg[1].tpr_log2 : a.seg[0].tpr_log2;
  const int cta = (int)blockIdx.x - (s1 ? a.seg[1].cta0 : 0);

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tpr = 1 << tl, RS = kThreads >> tl;
  const int slot = tid >> tl, tt = tid & (tpr - 1);
  const int row0 = (cta * RS + slot) * kR;
  const int C = K / V;
  const int nb = min(BT, a.B - a.b0);

  float acc[kR][BT];
#pragma unroll
  for (int k = 0; k < kR; ++k)
#pragma unroll
    for (int b = 0; b < BT; ++b) acc[k][b] = 0.f;
  if (!a.pdl) grid_dep_launch();

  for (int cb = 0; cb < C; cb += tpr * kC) {
    uint4 w[kR][kC];
#pragma unroll
    for (int k = 0; k < kR; ++k)
#pragma unroll
      for (int j = 0; j < kC; ++j) {
        const int c = cb + tt + j * tpr;
        if (row0 + k < rows && c < C) w[k][j] = ld_stream(W + (size_t)(row0 + k) * K + (size_t)c * V);
      }
    if (a.pdl && cb == 0) {  // the weights are in flight; x comes from the predecessor
      grid_dep_wait();
      grid_dep_launch();
    }
#pragma unroll
    for (int j = 0; j < kC; ++j) {
      const int c = cb + tt + j * tpr;
      if (c >= C) break;
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (b >= nb) break;
        float xf[V];
        const XT* xr = x + (size_t)(a.b0 + b) * K + (size_t)c * V;
        if constexpr (sizeof(XT) == sizeof(T)) {
          unpack<T>(ld_cached(xr), xf);
        } else {  // fp32 activations against 16-bit weights: 2 x 16 B
          unpack<float>(ld_cached(xr), xf);
          unpack<float>(ld_cached(xr + 4), xf + 4);
        }
#pragma unroll
        for (int k = 0; k < kR; ++k) {
          if (row0 + k >= rows) break;
          float wf[V];
          unpack<T>(w[k][j], wf);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[k][b] = fmaf(wf[v], xf[v], acc[k][b]);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kR; ++k)
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const float z = warp_sum(acc[k][b]);
      if (lane == 0) red[wid][k][b] = z;
    }
  __syncthreads();
  const int nw = tpr >> 5;  // warps per row group
  for (int e = tid; e < RS * kR * BT; e += kThreads) {
    const int sl = e / (kR * BT), k = (e / BT) % kR, b = e % BT;
    const int row = (cta * RS + sl) * kR + k;
    if (row >= rows || b >= nb) continue;
    float z = 0.f;
    for (int q = 0; q < nw; ++q) z += red[sl * nw + q][k][b];
    const float o = (EPI == kRelu) ? fmaxf(z, 0.f) : 1.f / (1.f + expf(-z));
    out[(size_t)(a.b0 + b) * rows + row] = o;
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
constexpr int kBins = 4096;  // histogram bins per refinement level (12 bits)
constexpr int kSelLoads = 24;  // score loads in flight per thread (one round for N <= 24576)
constexpr int kCand = 256;     // keys ranked directly in the cut's bin, at most

// One CTA per (predictor, batch row).  The row's scores are staged in shared
// memory as their IEEE bits (sigmoid outputs are >= 0, so the bits order like
// the values).
//
// Top-k orders the elements by (key descending, index ascending) and finds
// the k-th one, the cut (T, T_idx): element i is selected iff key_i > T, or
// key_i == T and i <= T_idx.  One level bins the keys of [min, max] into
// <= 4096 equal-width bins (width a power of two) and finds the bin holding
// the cut.  When at most kCand keys share that bin they are ranked against
// each other directly; otherwise further levels narrow the range to one key
// value (32-bit keys need at most three levels, and only keys inside the
// range touch the histogram) and the cut is the right count of lowest-index
// keys equal to it.  Output ascending: thread t owns the contiguous element
// range [t*E, (t+1)*E) with E odd (conflict-free bank access; E <= 53 for
// N <= 53248, so its selections fit a 64-bit mask), and a block prefix sum
// of per-thread counts gives every selected element its output slot.
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a, WsHeader* hdr) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ int tmp[32];
  __shared__ uint32_t rlo[32], rhi[32];
  __shared__ int sel_bin, sel_above, sel_count;
  __shared__ uint32_t cand_k[kCand];
  __shared__ int cand_i[kCand];
  __shared__ int n_cand;
  __shared__ uint32_t cut_k;
  __shared__ int cut_i;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
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
  grid_dep_wait();  // the scores are the predecessor's output

  // stage the scores: kSelLoads independent loads per thread per round trip
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int ib = tid; ib < N; ib += kSelThreads * kSelLoads) {
    float v[kSelLoads];
#pragma unroll
    for (int q = 0; q < kSelLoads; ++q) {
      const int i = ib + q * kSelThreads;
      v[q] = i < N ? __ldcg(s + i) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kSelLoads; ++q) {
      const int i = ib + q * kSelThreads;
      if (i < N) {
        const uint32_t kv = __float_as_uint(v[q]);
        keys[i] = kv;
        lo = min(lo, kv);
        hi = max(hi, kv);
      }
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) { rlo[wid] = lo; rhi[wid] = hi; }
  __syncthreads();
  const int E = ((N + kSelThreads - 1) / kSelThreads) | 1;
  const int i0 = min(N, tid * E);
  const int i1 = min(N, i0 + E);

  int total;
  if (mode == DV_THRESHOLD) {
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += __uint_as_float(keys[i]) > thr;
    const int incl = block_inclusive_scan<kSelThreads>(mine, tmp, &total);
    int o = incl - mine;
    for (int i = i0; i < i1; ++i)
      if (__uint_as_float(keys[i]) > thr) {
        if (o < cap) out[o] = i;
        ++o;
      }
    if (tid == 0) {
      count[b] = min(total, cap);
      if (total > cap) set_error(hdr, DV_ERR_CAPACITY, total);
    }
    return;
  }

  if (k <= 0 || k >= N) {
    if (k >= N)
      for (int i = tid; i < N; i += kSelThreads) out[i] = i;
    if (tid == 0) count[b] = k >= N ? N : 0;
    return;
  }
  lo = rlo[lane];
  hi = rhi[lane];
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);

  // Level over the keys inside [base, top]: bins them into <= 4096 bins of
  // width 2^shift, finds the bin holding the need-th largest key and
  // narrows [base, top] to it.  Returns that bin's key count.
  uint32_t base = lo, top = hi;
  int need = k;
  auto level = [&]() -> int {
    const uint32_t span = top - base;
    const int shift = max(0, 32 - __clz((int)span) - 12);
    const int nbins = (int)(span >> shift) + 1;
    for (int j = tid; j < nbins; j += kSelThreads) hist[j] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const uint32_t kv = keys[i];
      if (kv >= base && kv <= top) atomicAdd(&hist[(kv - base) >> shift], 1);
    }
    __syncthreads();
    // bins from the top: thread t sums bins nbins-1-4t .. nbins-4-4t
    int v4[4], v = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = nbins - 1 - (4 * tid + q);
      v4[q] = j >= 0 ? hist[j] : 0;
      v += v4[q];
    }
    int tot;
    const int incl = block_inclusive_scan<kSelThreads>(v, tmp, &tot);
    if (incl >= need && incl - v < need) {
      int above = incl - v;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (above + v4[q] >= need) {
          sel_bin = nbins - 1 - (4 * tid + q);
          sel_above = above;
          sel_count = v4[q];
          break;
        }
        above += v4[q];
      }
    }
    __syncthreads();
    need -= sel_above;
    const uint64_t nb = (uint64_t)base + ((uint64_t)sel_bin << shift);
    const uint64_t nt = nb + ((1ull << shift) - 1);
    base = (uint32_t)nb;
    top = (uint32_t)(nt < (uint64_t)top ? nt : (uint64_t)top);
    const int c = sel_count;
    __syncthreads();  // sel_* and hist are rewritten by the next level
    return c;
  };

  // The k-th largest (key, lowest index first) element is the cut (T, T_idx):
  // element i is selected iff keys[i] > T, or keys[i] == T and i <= T_idx.
  int c = level();
  if (c <= kCand) {
    // Few keys share the cut's bin: rank them directly.  Candidate c is
    // ranked by the candidates with a larger key or an equal key and a
    // lower index; the one of rank need-1 is the cut.
    if (tid == 0) n_cand = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const uint32_t kv = keys[i];
      if (kv >= base && kv <= top) {
        const int slot = atomicAdd(&n_cand, 1);
        cand_k[slot] = kv;
        cand_i[slot] = i;
      }
    }
    __syncthreads();
    if (tid < c) {
      const uint32_t kc = cand_k[tid];
      const int ic = cand_i[tid];
      int rank = 0;
      for (int j = 0; j < c; ++j) {
        const uint32_t kj = cand_k[j];
        rank += kj > kc || (kj == kc && cand_i[j] < ic);
      }
      if (rank == need - 1) {
        cut_k = kc;
        cut_i = ic;
      }
    }
  } else {
    // many keys in the bin: refine until one key value remains, then take
    // the need-th lowest index among the keys equal to it
#pragma unroll 1
    while (top > base) c = level();
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += keys[i] == base;
    int tot;
    const int eq_incl = block_inclusive_scan<kSelThreads>(eq, tmp, &tot);
    if (eq_incl >= need && eq_incl - eq < need) {
      int left = need - (eq_incl - eq);
      for (int i = i0; i < i1; ++i)
        if (keys[i] == base && --left == 0) {
          cut_k = base;
          cut_i = i;
          break;
        }
    }
  }
  __syncthreads();
  const uint32_t T = cut_k;
  const int Ti = cut_i;
  // this thread's selected elements (at most 64: E <= 64 for N <= 65536)
  uint64_t mask = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t kv = keys[i];
    if (kv > T || (kv == T && i <= Ti)) mask |= 1ull << (i - i0);
  }
  const int mine = __popcll(mask);
  int total_sel;
  const int sel_incl = block_inclusive_scan<kSelThreads>(mine, tmp, &total_sel);
  int o = sel_incl - mine;
  while (mask) {
    const int bit = __ffsll((long long)mask) - 1;
    out[o++] = i0 + bit;
    mask &= mask - 1;
  }
  if (tid == 0) count[b] = k;
}

template <typename T, typename XT, int EPI, int BT>
cudaError_t launch_rows(RowArgs a, int grid, cudaStream_t stream) {
  return launch_k(rows_dot<T, XT, EPI, BT>, dim3(grid), dim3(kThreads), 0, stream, a.pdl != 0, 1, a);
}

// One launch per batch tile of up to 8 rows; the two segments' CTAs are laid
// out back to back.
template <typename T, typename XT, int EPI>
cudaError_t run_rows(RowArgs a, cudaStream_t stream) {
  int grid = 0;
  for (int i = 0; i < a.nseg; ++i) {
    RowSeg& s = a.seg[i];
    s.tpr_log2 = tpr_log2_for(s.K / Elem<T>::kVec);
    s.cta0 = grid;
    const int rpc = rows_per_cta(s.tpr_log2);
    grid += (s.rows + rpc - 1) / rpc;
  }
  for (int b0 = 0; b0 < a.B;) {
    const int nb = a.B - b0;
    const int bt = nb >= 8 ? 8 : (nb >= 4 ? 4 : (nb >= 2 ? 2 : 1));
    a.b0 = b0;
    cudaError_t e;
    switch (bt) {
      case 8: e = launch_rows<T, XT, EPI, 8>(a, grid, stream); break;
      case 4: e = launch_rows<T, XT, EPI, 4>(a, grid, stream); break;
      case 2: e = launch_rows<T, XT, EPI, 2>(a, grid, stream); break;
      default: e = launch_rows<T, XT, EPI, 1>(a, grid, stream); break;
    }
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

// One CTA per (row, predictor): top-k or threshold over the fp32 scores.
cudaError_t select_all(int B, const PredLaunch& p, int n_preds, WsHeader* hdr, cudaStream_t stream) {
  SelArgs sa{};
  int nmax = 0;
  for (int i = 0; i < n_preds; ++i) {
    sa.s[i] = p.s[i]; sa.N[i] = p.N[i]; sa.mode[i] = p.mode[i]; sa.k[i] = p.k[i];
    sa.cap[i] = p.cap[i]; sa.t[i] = p.t[i]; sa.idx[i] = p.idx[i]; sa.count[i] = p.count[i];
    nmax = p.N[i] > nmax ? p.N[i] : nmax;
  }
  const size_t smem = (size_t)nmax * sizeof(uint32_t);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [] {
    return (int)cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kSelectMaxN * sizeof(uint32_t)));
  });
  if (ea != cudaSuccess) return ea;
  return launch_k(select_kernel, dim3(B, n_preds), dim3(kSelThreads), smem, stream, true, 1, sa, hdr);
}

template <typename T>
cudaError_t predict_t(const void* y, int B, int d, const PredLaunch& p, int n_preds,
                      WsHeader* hdr, cudaStream_t stream) {
  RowArgs g1{};
  g1.nseg = n_preds;
  g1.B = B;
  for (int i = 0; i < n_preds; ++i) g1.seg[i] = RowSeg{p.P1t[i], y, p.h[i], p.r[i], d, 0, 0};
  cudaError_t e = run_rows<T, T, kRelu>(g1, stream);
  if (e != cudaSuccess) return e;

  RowArgs g2{};
  g2.nseg = n_preds;
  g2.B = B;
  g2.pdl = 1;
  for (int i = 0; i < n_preds; ++i) g2.seg[i] = RowSeg{p.P2t[i], p.h[i], p.s[i], p.N[i], p.r[i], 0, 0};
  e = run_rows<T, float, kSigmoid>(g2, stream);
  if (e != cudaSuccess) return e;
  return select_all(B, p, n_preds, hdr, stream);
}

}  // namespace

cudaError_t launch_select(const float* scores, int B, int N, int mode, int k, float t, int32_t* idx, int cap,
                          int32_t* count, WsHeader* hdr, cudaStream_t stream) {
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [] {
    return (int)cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kSelectMaxN * sizeof(uint32_t)));
  });
  if (ea != cudaSuccess) return ea;
  SelArgs sa{};
  sa.s[0] = scores; sa.N[0] = N; sa.mode[0] = mode; sa.k[0] = k; sa.cap[0] = cap; sa.t[0] = t;
  sa.idx[0] = idx; sa.count[0] = count;
  return launch_k(select_kernel, dim3(B, 1), dim3(kSelThreads), (size_t)N * sizeof(uint32_t), stream, true, 1, sa,
                  hdr);
}

cudaError_t launch_predict(const void* y, int B, int d, dv_dtype dt, const PredLaunch& p,
                           int n_preds, WsHeader* hdr, cudaStream_t stream) {
  if (predict_tc_supported(B, d, dt, p, n_preds)) {
    const cudaError_t e = launch_predict_tc(y, B, d, dt, p, n_preds, hdr, stream);
    return e != cudaSuccess ? e : select_all(B, p, n_preds, hdr, stream);
  }
  switch (dt) {
    case DV_F32: return predict_t<float>(y, B, d, p, n_preds, hdr, stream);
    case DV_F16: return predict_t<__half>(y, B, d, p, n_preds, hdr, stream);
    case DV_BF16: return predict_t<__nv_bfloat16>(y, B, d, p, n_preds, hdr, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

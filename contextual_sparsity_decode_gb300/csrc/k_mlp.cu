// Sparsified MLP, one pass over the selected weight rows:
//     out_b += sum_{j in S_b} ReLU(y_b . W^1[:, j]) * W^2[:, j]
// (Deja Vu reading notes, "Sparsified MLP"; the fused index-select + matmul
// of "用Deja Vu来提高 LLM 的推理速度" §3.2, which reads each selected weight
// byte once and never writes a gathered sub-matrix.)
//
// GB300 design.  W^1 and W^2 are stored neuron-major (row j = neuron j's d
// weights, 16-byte aligned), so every gathered neuron is two contiguous rows
// ("Memory coalescing", §3.3).  A thread-block cluster of CS CTAs splits the
// d columns; cluster g owns a contiguous share of the selected neurons:
//   phase 1  each CTA dots its column slice of W^1[j] with its slice of y
//            (every load of a warp's batch of rows issued before any use) and
//            pushes the partial into every peer's shared memory;
//   barrier  one cluster barrier per sub-chunk, after which every CTA sums
//            the CS partials locally in a fixed rank order (all CTAs agree)
//            and applies ReLU (and the row's membership mask when B > 1);
//   phase 2  each CTA accumulates a_j * W^2[j] over its column slice in
//            registers; the W^2 rows were prefetched into L2 when the
//            sub-chunk started and the first loads are in flight across the
//            barrier.
// Clusters add their column slices into out with 16-byte fp32 atomics.  The
// grid holds only as many clusters as fit on the GPU at once (no second
// wave).  Selected neurons are processed in sub-chunks of 64 with
// double-buffered partials.
#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kThreads = 256;
constexpr int kJS = 64;  // neurons per sub-chunk
constexpr int kMaxCS = 8;  // largest cluster

struct MlpArgs {
  const void* y;
  const void* W1n;
  const void* W2n;
  const int32_t* list;        // neuron ids (ascending)
  const int32_t* list_count;  // device count
  const uint32_t* member;     // [B][words] or nullptr
  int words;
  int B, b0, d, N, cap;
  int CS, CPR;                // cluster size, 16-byte chunks per CTA row slice
  float* out;
  WsHeader* hdr;
};

constexpr int kL1 = 12;  // phase-1 loads in flight per lane
constexpr int kL2 = 10;  // phase-2 loads in flight per thread

// CPLT: 16-byte chunks per lane of a row slice (>= ceil(CPR / 32)).
template <typename T, int BT, int CPLT>
__global__ void __launch_bounds__(kThreads, 2) sparse_mlp_kernel(MlpArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int RB = kL1 / CPLT;  // rows per warp per phase-1 batch
  extern __shared__ float ys[];   // [BT][w]
  __shared__ float pd[2][kMaxCS][kJS][BT];  // partials pushed by each rank
  __shared__ float as[kJS][BT];
  __shared__ int rows_s[kJS];

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int CS = a.CS, CPR = a.CPR, w = CPR * V;
  const int rank = (int)cluster_ctarank();
  const int g = blockIdx.x / CS, G = gridDim.x / CS;
  const int col0 = rank * w;
  const int nb = min(BT, a.B - a.b0);

  // every CTA of the cluster must be running before a peer stores into its
  // shared memory: arrive now, wait before the first push
  cluster_arrive();

  // Batch 1 splits the list by its capacity, so list entries are read in
  // parallel with the count and the y slice; the batch union splits by the
  // count.
  int cnt = *a.list_count;
  const int span = a.member ? max(0, min(cnt, a.cap)) : a.cap;
  const int n_c = (span + G - 1) / G;
  const int j_begin = min(span, g * n_c), j_end = min(span, j_begin + n_c);
  const int row_pre = tid < min(kJS, j_end - j_begin) ? a.list[j_begin + tid] : -1;

  // stage this CTA's slice of y (fp32), 16-byte loads
  for (int e = tid; e < BT * CPR; e += kThreads) {
    const int b = e / CPR, c = e - b * CPR;
    float f[V];
    if (b < nb) {
      unpack<T>(ld_cached(static_cast<const T*>(a.y) + (size_t)(a.b0 + b) * a.d + col0 + (size_t)c * V), f);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) f[v] = 0.f;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) ys[b * w + c * V + v] = f[v];
  }
  if (cnt > a.cap) {
    if (tid == 0 && rank == 0 && g == 0) set_error(a.hdr, DV_ERR_CAPACITY, cnt);
    cnt = a.cap;
  }

  const T* W1 = static_cast<const T*>(a.W1n);
  const T* W2 = static_cast<const T*>(a.W2n);
  const int NG = kThreads / CPR;          // phase-2 thread groups over neurons
  const int cc = tid % CPR, gi = tid / CPR;
  float acc2[BT][V];
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int v = 0; v < V; ++v) acc2[b][v] = 0.f;

  const int nsub = (j_end - j_begin + kJS - 1) / kJS;
  cluster_wait();
  for (int sc = 0; sc < nsub; ++sc) {
    const int jj0 = j_begin + sc * kJS;
    const int jn = min(kJS, j_end - jj0);
    const int buf = sc & 1;
    __syncthreads();  // previous sub-chunk done with rows_s / as; ys staged
    if (tid < jn) {
      const int j = jj0 + tid;
      int row = sc == 0 ? row_pre : a.list[j];
      if (j >= cnt) {
        row = -1;
      } else if (row < 0 || row >= a.N) {
        if (rank == 0) set_error(a.hdr, DV_ERR_INDEX_RANGE, row);
        row = -1;
      } else {
        prefetch_l2(W2 + (size_t)row * a.d + col0, (uint32_t)(w * sizeof(T)));
      }
      rows_s[tid] = row;
    }
    __syncthreads();

    // phase 1: partial dots over this CTA's column slice; a warp issues all
    // loads of a batch of RB rows before using them
    for (int rb0 = wid; rb0 < jn; rb0 += 8 * RB) {
      uint4 wv[RB][CPLT];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int jj = rb0 + 8 * r;
        const int row = jj < jn ? rows_s[jj] : -1;
#pragma unroll
        for (int c = 0; c < CPLT; ++c) {
          const int ch = lane + 32 * c;
          if (row >= 0 && ch < CPR) wv[r][c] = ld_stream(W1 + (size_t)row * a.d + col0 + (size_t)ch * V);
        }
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int jj = rb0 + 8 * r;
        if (jj >= jn) break;
        const int row = rows_s[jj];
        float acc[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[b] = 0.f;
        if (row >= 0) {
#pragma unroll
          for (int c = 0; c < CPLT; ++c) {
            const int ch = lane + 32 * c;
            if (ch < CPR) {
              float wf[V];
              unpack<T>(wv[r][c], wf);
#pragma unroll
              for (int b = 0; b < BT; ++b) {
                const float4* yb = reinterpret_cast<const float4*>(ys + b * w + ch * V);
#pragma unroll
                for (int v4 = 0; v4 < V / 4; ++v4) {
                  const float4 yv = yb[v4];
                  acc[b] = fmaf(wf[4 * v4 + 0], yv.x, acc[b]);
                  acc[b] = fmaf(wf[4 * v4 + 1], yv.y, acc[b]);
                  acc[b] = fmaf(wf[4 * v4 + 2], yv.z, acc[b]);
                  acc[b] = fmaf(wf[4 * v4 + 3], yv.w, acc[b]);
                }
              }
            }
          }
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const float sm = warp_sum(acc[b]);  // every lane holds the sum
          if (lane < CS) st_dsmem_f32(&pd[buf][rank][jj][b], (uint32_t)lane, sm);
        }
      }
    }

    // first batch of phase-2 loads, in flight across the cluster barrier
    uint4 w2[kL2];
    const int q_end = gi < NG ? (jn - gi + NG - 1) / NG : 0;  // rows gi, gi + NG, ...
#pragma unroll
    for (int q = 0; q < kL2; ++q) {
      const int jj = gi + q * NG;
      if (q < q_end && rows_s[jj] >= 0)
        w2[q] = ld_stream(W2 + (size_t)rows_s[jj] * a.d + col0 + (size_t)cc * V);
    }
    cluster_arrive();
    cluster_wait();

    // cluster-wide sum of the partials, ReLU, batch-row mask
    for (int e = tid; e < jn * BT; e += kThreads) {
      const int jj = e / BT, b = e - jj * BT;
      float sum = 0.f;
      for (int q = 0; q < CS; ++q) sum += pd[buf][q][jj][b];
      float act = fmaxf(sum, 0.f);
      const int row = rows_s[jj];
      if (row < 0 || b >= nb) act = 0.f;
      else if (a.member && !bit_test(a.member + (size_t)(a.b0 + b) * a.words, row)) act = 0.f;
      as[jj][b] = act;
    }
    __syncthreads();

    // phase 2: out slice += a_j * W^2[j] (slice)
    for (int q0 = 0; q0 < q_end; q0 += kL2) {
      if (q0 > 0) {
#pragma unroll
        for (int q = 0; q < kL2; ++q) {
          const int jj = gi + (q0 + q) * NG;
          if (q0 + q < q_end && rows_s[jj] >= 0)
            w2[q] = ld_stream(W2 + (size_t)rows_s[jj] * a.d + col0 + (size_t)cc * V);
        }
      }
#pragma unroll
      for (int q = 0; q < kL2; ++q) {
        const int jj = gi + (q0 + q) * NG;
        if (q0 + q < q_end && rows_s[jj] >= 0) {
          float wf[V];
          unpack<T>(w2[q], wf);
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            const float ab = as[jj][b];
#pragma unroll
            for (int v = 0; v < V; ++v) acc2[b][v] = fmaf(ab, wf[v], acc2[b][v]);
          }
        }
      }
    }
  }
  // No final cluster barrier: peers write into this CTA's shared memory only
  // before the barrier of the same sub-chunk, which this CTA has passed.

  if (gi < NG && j_end > j_begin) {
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      if (b >= nb) break;
      float* o = a.out + (size_t)(a.b0 + b) * a.d + col0 + (size_t)cc * V;
#pragma unroll
      for (int v = 0; v < V; v += 4)
        atomic_add_f32x4(o + v, acc2[b][v], acc2[b][v + 1], acc2[b][v + 2], acc2[b][v + 3]);
    }
  }
}

// Union of the rows' lists: ascending U, |U|, and per-row membership bitmaps.
__global__ void __launch_bounds__(1024) union_kernel(const int32_t* idx, int cap, const int32_t* count,
                                                     int B, int N, int32_t* U, int32_t* U_count,
                                                     uint32_t* member, int32_t* slot_of,
                                                     WsHeader* hdr) {
  extern __shared__ uint32_t bm[];
  __shared__ int tmp[32];
  const int words = (N + 31) / 32;
  for (int i = threadIdx.x; i < words; i += blockDim.x) bm[i] = 0u;
  for (int i = threadIdx.x; i < B * words; i += blockDim.x) member[i] = 0u;
  __syncthreads();
  for (int b = 0; b < B; ++b) {
    int cnt = count[b];
    if (cnt > cap) {
      if (threadIdx.x == 0) set_error(hdr, DV_ERR_CAPACITY, cnt);
      cnt = cap;
    }
    for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
      const int j = idx[(size_t)b * cap + e];
      if (j < 0 || j >= N) {
        set_error(hdr, DV_ERR_INDEX_RANGE, j);
        continue;
      }
      const uint32_t bit = 1u << (j & 31);
      atomicOr(&bm[j >> 5], bit);
      atomicOr(&member[(size_t)b * words + (j >> 5)], bit);
    }
  }
  __syncthreads();
  const int WW = (words + 1023) / 1024;
  const int w0 = min(words, (int)threadIdx.x * WW), w1 = min(words, w0 + WW);
  int mine = 0;
  for (int i = w0; i < w1; ++i) mine += __popc(bm[i]);
  int total;
  const int incl = block_inclusive_scan<1024>(mine, tmp, &total);
  int o = incl - mine;
  for (int i = w0; i < w1; ++i) {
    uint32_t m = bm[i];
    while (m) {
      const int bit = __ffs(m) - 1;
      if (slot_of) slot_of[i * 32 + bit] = o;
      U[o++] = i * 32 + bit;
      m &= m - 1;
    }
  }
  if (threadIdx.x == 0) *U_count = total;
}

struct ClusterPlan {
  int CS = 0, CPR = 0;
};

// Largest cluster size (<= 8) that splits the d/V chunks evenly into slices
// of at most 256 chunks, preferring slices that are whole warps wide.
ClusterPlan plan_cluster(int chunks) {
  ClusterPlan best;
  for (int pass = 0; pass < 2 && best.CS == 0; ++pass)
    for (int cs = 8; cs >= 1; --cs) {
      if (chunks % cs) continue;
      const int cpr = chunks / cs;
      if (cpr > kThreads) continue;
      if (pass == 0 && cpr % 32) continue;
      best.CS = cs;
      best.CPR = cpr;
      break;
    }
  return best;
}

template <typename T, int BT, int CPLT>
cudaError_t run_mlp(MlpArgs a, int num_sms, cudaStream_t stream) {
  const size_t smem = (size_t)BT * a.CPR * Elem<T>::kVec * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sparse_mlp_kernel<T, BT, CPLT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(BT * 256 * Elem<T>::kVec * sizeof(float)));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sparse_mlp_kernel<T, BT, CPLT>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // As many clusters as are co-resident (cached per cluster size and shared
  // memory), never more than 16-neuron shares of the work.
  static int cached_cs[kMaxCS + 1] = {0};
  static size_t cached_smem[kMaxCS + 1] = {0};
  if (cached_cs[a.CS] == 0 || cached_smem[a.CS] != smem) {
    cfg.gridDim = dim3(a.CS * num_sms);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mlp_kernel<T, BT, CPLT>, &cfg) != cudaSuccess || n < 1)
      n = (2 * num_sms) / a.CS;
    cached_cs[a.CS] = n;
    cached_smem[a.CS] = smem;
  }
  int G = cached_cs[a.CS];
  const int by_work = (a.cap + 15) / 16;
  G = G < by_work ? G : by_work;
  G = G < 1 ? 1 : G;
  cfg.gridDim = dim3(G * a.CS);
  return cudaLaunchKernelEx(&cfg, sparse_mlp_kernel<T, BT, CPLT>, a);
}

template <typename T, int BT>
cudaError_t run_mlp_cpl(MlpArgs a, int num_sms, cudaStream_t stream) {
  const int cpl = (a.CPR + 31) / 32;
  if (cpl <= 2) return run_mlp<T, BT, 2>(a, num_sms, stream);
  if (cpl <= 4) return run_mlp<T, BT, 4>(a, num_sms, stream);
  return run_mlp<T, BT, 8>(a, num_sms, stream);
}

template <typename T>
cudaError_t mlp_t(const MlpLaunch& L, WsHeader* hdr, int num_sms, cudaStream_t stream) {
  const ClusterPlan cp = plan_cluster(L.d / Elem<T>::kVec);
  if (cp.CS == 0) return cudaErrorInvalidValue;
  MlpArgs a{};
  a.y = L.y; a.W1n = L.W1n; a.W2n = L.W2n;
  a.B = L.B; a.d = L.d; a.N = L.N;
  a.CS = cp.CS; a.CPR = cp.CPR;
  a.out = L.out; a.hdr = hdr;
  a.words = (L.N + 31) / 32;
  if (L.B == 1) {
    a.list = L.idx; a.list_count = L.count; a.member = nullptr; a.cap = L.cap;
  } else {
    a.list = L.U; a.list_count = L.U_count; a.member = L.member; a.cap = L.N;
  }
  for (int b0 = 0; b0 < L.B;) {
    const int nb = L.B - b0;
    const int bt = nb >= 8 ? 8 : (nb >= 4 ? 4 : (nb >= 2 ? 2 : 1));
    a.b0 = b0;
    cudaError_t e;
    switch (bt) {
      case 8: e = run_mlp_cpl<T, 8>(a, num_sms, stream); break;
      case 4: e = run_mlp_cpl<T, 4>(a, num_sms, stream); break;
      case 2: e = run_mlp_cpl<T, 2>(a, num_sms, stream); break;
      default: e = run_mlp_cpl<T, 1>(a, num_sms, stream); break;
    }
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_union(const int32_t* idx, int cap, const int32_t* count, int B, int N,
                         int32_t* U, int32_t* U_count, uint32_t* member, int32_t* slot_of,
                         WsHeader* hdr, cudaStream_t stream) {
  const size_t smem = (size_t)((N + 31) / 32) * sizeof(uint32_t);
  union_kernel<<<1, 1024, smem, stream>>>(idx, cap, count, B, N, U, U_count, member, slot_of, hdr);
  return cudaGetLastError();
}

cudaError_t launch_sparse_mlp(const MlpLaunch& L, dv_dtype dt, WsHeader* hdr, int num_sms,
                              cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (!L.accumulate) {
    e = cudaMemsetAsync(L.out, 0, (size_t)L.B * L.d * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  if (L.B > 1) {
    e = launch_union(L.idx, L.cap, L.count, L.B, L.N, L.U, L.U_count, L.member, nullptr, hdr,
                     stream);
    if (e != cudaSuccess) return e;
  }
  if (L.B > 1 && tc_mlp_supported(L.B, L.d, dt)) return launch_sparse_mlp_tc(L, dt, hdr, stream);
  switch (dt) {
    case DV_F32: return mlp_t<float>(L, hdr, num_sms, stream);
    case DV_F16: return mlp_t<__half>(L, hdr, num_sms, stream);
    case DV_BF16: return mlp_t<__nv_bfloat16>(L, hdr, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

// Sparsified MLP, out_b += sum_{j in S_b} ReLU(y_b . W^1[:, j]) * W^2[:, j]
// (Deja Vu reading notes, "Sparsified MLP"), as the fused index-select +
// matmul of "用Deja Vu来提高 LLM 的推理速度" §3.2: each selected weight byte is
// read once and no gathered sub-matrix is ever written.
//
// W^1 and W^2 are stored neuron-major (row j = neuron j's d weights,
// 16-byte aligned), so every selected neuron is two contiguous rows
// ("Memory coalescing", §3.3).  Two steps:
//   up            a_b[u] = ReLU(W^1[list[u]] . y_b) (x the row's membership
//                 mask when B > 1), a gathered row-dot: a CTA holds a tile of
//                 selected rows and every thread issues all of its row loads
//                 before using any (same tiling as the predictor GEMV);
//   combine       out_b (+)= sum_u a_b[u] W^2[list[u]], column-sliced with one
//                 writer per output element (rows_combine.cuh).
// At batch 1 both run in one launch (mlp_fused_kernel) when its grid fits
// on the GPU at once; otherwise as mlp_up_kernel + rows_combine_kernel.
// Batches of 2+ rows in a 16-bit type use the tcgen05 path (k_mlp_tc.cu).

#include <cstdlib>

#include "rows_combine.cuh"

namespace dv {
namespace {

constexpr int kThreads = 256;
constexpr int kUpC = 4;   // 16-byte chunks per thread per pass over a row
constexpr int kUpR = 3;   // rows per thread group

struct UpArgs {
  const void* y;
  const void* W1n;
  const int32_t* list;        // selected neurons (ascending)
  const int32_t* list_count;  // device count
  int cap;                    // room in list and in each act row
  const uint32_t* member;     // [B][words] or nullptr (batch 1)
  int words;
  int B, b0, d, N;
  int tl;                     // threads per row (log2)
  float* act;                 // [B][cap]
  WsHeader* hdr;
  int pdl;                    // launched with overlap: y is read after grid_dep_wait()
};

int up_tpr_log2(int chunks, int kC) {
  int l = 5;
  while (l < 8 && (1 << l) * kC < chunks) ++l;
  return l;
}

// One CTA (row tile bx) of the up-projection.
template <typename T, int BT, int kC, int kR>
__device__ __forceinline__ void mlp_up_block(const UpArgs& a, int bx) {
  constexpr int V = Elem<T>::kVec;
  __shared__ float red[kThreads / 32][kR][BT];
  __shared__ int nid_s[kThreads / 32 * kR];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tpr = 1 << a.tl, RS = kThreads >> a.tl;
  const int slot = tid >> a.tl, tt = tid & (tpr - 1);
  const int row0 = (bx * RS + slot) * kR;  // positions in the list
  const int C = a.d / V;
  if (!a.pdl) grid_dep_launch();  // the down-projection may start loading its rows
  const int nb = min(BT, a.B - a.b0);
  // list entries are read in parallel with the count (positions < cap are in bounds)
  int nid[kR];
#pragma unroll
  for (int k = 0; k < kR; ++k) nid[k] = row0 + k < a.cap ? a.list[row0 + k] : -1;
  const int cnt = max(0, min(*a.list_count, a.cap));
#pragma unroll
  for (int k = 0; k < kR; ++k) {
    if (row0 + k >= cnt) {
      nid[k] = -1;
    } else if (nid[k] < 0 || nid[k] >= a.N) {
      if (tt == 0) set_error(a.hdr, DV_ERR_INDEX_RANGE, nid[k]);
      nid[k] = -1;
    }
  }
  if (tt == 0)
#pragma unroll
    for (int k = 0; k < kR; ++k) nid_s[slot * kR + k] = nid[k];
  const T* W = static_cast<const T*>(a.W1n);
  const T* y = static_cast<const T*>(a.y);

  float acc[kR][BT];
#pragma unroll
  for (int k = 0; k < kR; ++k)
#pragma unroll
    for (int b = 0; b < BT; ++b) acc[k][b] = 0.f;
  for (int cb = 0; cb < C; cb += tpr * kC) {
    uint4 w[kR][kC];
#pragma unroll
    for (int k = 0; k < kR; ++k)
#pragma unroll
      for (int j = 0; j < kC; ++j) {
        const int c = cb + tt + j * tpr;
        if (nid[k] >= 0 && c < C) w[k][j] = ld_stream(W + (size_t)nid[k] * a.d + (size_t)c * V);
      }
    if (a.pdl && cb == 0) {  // rows in flight; y comes from the kernel before the call
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
        unpack<T>(ld_cached(y + (size_t)(a.b0 + b) * a.d + (size_t)c * V), xf);
#pragma unroll
        for (int k = 0; k < kR; ++k) {
          if (nid[k] < 0) continue;
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
  const int nw = tpr >> 5;
  for (int e = tid; e < RS * kR * BT; e += kThreads) {
    const int sl = e / (kR * BT), k = (e / BT) % kR, b = e % BT;
    const int pos = (bx * RS + sl) * kR + k;
    if (pos >= a.cap || b >= nb) continue;
    const int j = nid_s[sl * kR + k];
    float z = 0.f;
    for (int q = 0; q < nw; ++q) z += red[sl * nw + q][k][b];
    float act = fmaxf(z, 0.f);
    if (j < 0) act = 0.f;
    else if (a.member && !bit_test(a.member + (size_t)(a.b0 + b) * a.words, j)) act = 0.f;
    a.act[(size_t)(a.b0 + b) * a.cap + pos] = act;
  }
}

template <typename T, int BT>
__global__ void __launch_bounds__(kThreads) mlp_up_kernel(UpArgs a) {
  mlp_up_block<T, BT, kUpC, kUpR>(a, (int)blockIdx.x);
}

// Batch 1, one launch for both products: CTAs [0, nA) compute activations
// (mlp_up_block, 5 chunks x 4 rows per thread so that few CTAs hold all
// selected rows), CTAs [nA, nA + nB) are the column blocks of the second
// product (rows_combine_block).  A down-projection CTA requests its W^2 rows
// first and then waits for the nA arrivals on ctr[0].  The host launches
// this kernel only when the whole grid fits on the GPU at once, so every CTA
// can be resident together and a waiting CTA never keeps an up-projection
// CTA from starting (CTAs of other kernels on the SMs finish without waiting
// for this one); up-projection CTAs also have the lower indices.
//
// The wait is bounded (wait_ns of the global timer) and reports
// DV_ERR_TIMEOUT.  ctr[1] counts the down-projection CTAs past the wait; the
// last one takes nA back off ctr[0] and nB off ctr[1] (subtraction, not a
// reset, so an up-projection CTA that arrives after a timed-out wait still
// brings ctr[0] back to zero for the next call).  Counts above nA cannot
// occur in a zero-filled workspace and are reported as DV_ERR_WORKSPACE.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    mlp_fused_kernel(UpArgs u, CombineLaunch c, int nA, int* ctr, long long wait_ns) {
  if ((int)blockIdx.x < nA) {
    mlp_up_block<T, 1, 5, 4>(u, (int)blockIdx.x);
    __syncthreads();  // this CTA's activations are written
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(ctr, 1);
    }
    return;
  }
  const int nB = (int)gridDim.x - nA;
  rows_combine_block<T, 1>(c, 0, (int)blockIdx.x - nA, [&] {
    grid_dep_wait();  // out was written by kernels before this one
    grid_dep_launch();
    if (threadIdx.x == 0) {
      const unsigned long long t0 = globaltimer_ns();
      int seen = 0;
      while ((seen = ld_acquire_gpu(ctr)) < nA) {
        if ((long long)(globaltimer_ns() - t0) > wait_ns) {
          set_error(c.hdr, DV_ERR_TIMEOUT, seen);
          break;
        }
      }
      if (seen > nA) set_error(c.hdr, DV_ERR_WORKSPACE, seen);
      if (atomicAdd(ctr + 1, 1) == nB - 1) {  // every down-projection CTA is past the wait
        atomicSub(ctr, nA);
        atomicSub(ctr + 1, nB);
      }
    }
    __syncthreads();
  });
}

// Union of the rows' lists: ascending U, |U|, and per-row membership bitmaps.
// `clear` (optional, `words` long) is zeroed for a later kernel.
__global__ void __launch_bounds__(1024) union_kernel(const int32_t* idx, int cap, const int32_t* count,
                                                     int B, int N, int32_t* U, int32_t* U_count,
                                                     uint32_t* member, int32_t* slot_of,
                                                     WsHeader* hdr, uint32_t* clear, RowsExpand ex) {
  extern __shared__ uint32_t bm[];
  __shared__ int tmp[32];
  const int words = (N + 31) / 32;
  for (int i = threadIdx.x; i < words; i += blockDim.x) bm[i] = 0u;
  for (int i = threadIdx.x; i < B * words; i += blockDim.x) member[i] = 0u;
  if (clear)
    for (int i = threadIdx.x; i < words; i += blockDim.x) clear[i] = 0u;
  __syncthreads();
  __shared__ int cnt_s[32];
  if ((int)threadIdx.x < B) {  // every row's count in one round trip
    int cnt = count[threadIdx.x];
    if (cnt > cap) {
      set_error(hdr, DV_ERR_CAPACITY, cnt);
      cnt = cap;
    }
    cnt_s[threadIdx.x] = max(cnt, 0);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < B * cap; t += blockDim.x) {  // all rows' entries at once
    const int b = t / cap, e = t - b * cap;
    if (e >= cnt_s[b]) continue;
    const int j = idx[(size_t)b * cap + e];
    if (j < 0 || j >= N) {
      set_error(hdr, DV_ERR_INDEX_RANGE, j);
      continue;
    }
    const uint32_t bit = 1u << (j & 31);
    atomicOr(&bm[j >> 5], bit);
    atomicOr(&member[(size_t)b * words + (j >> 5)], bit);
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
  // the row lists of the union's units (U as written above by this CTA)
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    if (!ex.rows[q]) continue;
    const int per = ex.per[q];
    if (threadIdx.x == 0) *ex.count[q] = total * per;
    for (int k = threadIdx.x; k < total * per; k += blockDim.x) {
      const int u = k / per;
      ex.rows[q][k] = U[u] * per + (k - u * per);
    }
  }
}


// Large unions (many rows x long lists) in two passes.  One CTA per row
// builds the row's membership bitmap in shared memory from its list and
// writes it out whole (no global atomics, nothing to clear first); then one
// CTA ORs the rows' bitmaps word by word and lists the union.  (The version
// that marked every entry with two global atomicOr took 30 + 18 us for 32
// rows of 14336 entries.)
__global__ void __launch_bounds__(1024) union_rows_kernel(const int32_t* idx, int cap, const int32_t* count, int N,
                                                          uint32_t* member, WsHeader* hdr) {
  extern __shared__ uint32_t bm[];
  const int b = blockIdx.x;
  const int words = (N + 31) / 32;
  for (int i = threadIdx.x; i < words; i += blockDim.x) bm[i] = 0u;
  int cnt = count[b];
  if (cnt > cap) {
    if (threadIdx.x == 0) set_error(hdr, DV_ERR_CAPACITY, cnt);
    cnt = cap;
  }
  cnt = max(cnt, 0);
  __syncthreads();
  const int32_t* row = idx + (size_t)b * cap;
  for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
    const int j = row[e];
    if (j < 0 || j >= N) {
      set_error(hdr, DV_ERR_INDEX_RANGE, j);
      continue;
    }
    atomicOr(&bm[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < words; i += blockDim.x) member[(size_t)b * words + i] = bm[i];
}

constexpr int kUnionMaxB = 32;      // rows of a batch, at most
constexpr int kUnionMaxWW = 2;      // words per thread: N <= 65536 is 2048 words over 1024 threads

// OR of word i over the B rows' bitmaps: every row's load is issued at once
__device__ __forceinline__ uint32_t union_word(const uint32_t* member, int B, int words, int i) {
  uint32_t v[kUnionMaxB];
#pragma unroll
  for (int b = 0; b < kUnionMaxB; ++b) v[b] = b < B ? __ldcg(member + (size_t)b * words + i) : 0u;
  uint32_t m = 0u;
#pragma unroll
  for (int b = 0; b < kUnionMaxB; ++b) m |= v[b];
  return m;
}

__global__ void __launch_bounds__(1024) union_list_kernel(const uint32_t* member, int B, int N, int32_t* U,
                                                          int32_t* U_count, int32_t* slot_of) {
  __shared__ int tmp[32];
  const int words = (N + 31) / 32;
  const int WW = (words + 1023) / 1024;  // <= kUnionMaxWW
  const int w0 = min(words, (int)threadIdx.x * WW), w1 = min(words, w0 + WW);
  uint32_t mw[kUnionMaxWW];
  int mine = 0;
#pragma unroll
  for (int q = 0; q < kUnionMaxWW; ++q) {
    mw[q] = w0 + q < w1 ? union_word(member, B, words, w0 + q) : 0u;
    mine += __popc(mw[q]);
  }
  int total;
  const int incl = block_inclusive_scan<1024>(mine, tmp, &total);
  int o = incl - mine;
#pragma unroll
  for (int q = 0; q < kUnionMaxWW; ++q) {
    const int i = w0 + q;
    uint32_t m = mw[q];
    while (m) {
      const int bit = __ffs(m) - 1;
      if (slot_of) slot_of[i * 32 + bit] = o;
      U[o++] = i * 32 + bit;
      m &= m - 1;
    }
  }
  if (threadIdx.x == 0) *U_count = total;
}

template <typename T, int BT>
cudaError_t launch_up(const UpArgs& a, int grid, cudaStream_t stream) {
  return launch_k(mlp_up_kernel<T, BT>, dim3(grid), dim3(kThreads), 0, stream, a.pdl != 0, 1, a);
}

// Does the one-launch MLP's grid fit on the GPU at once?  (CTAs per SM are
// a property of the device, so the answer is cached per device.)
template <typename T>
bool fused_fits(int grid, int num_sms) {
  static PerDevice per_sm;
  const int n_sm = per_sm.get(current_device(), [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mlp_fused_kernel<T>, kThreads, 0) != cudaSuccess)
      n = 0;
    (void)cudaGetLastError();
    return n;
  });
  return (long long)n_sm * num_sms >= grid;
}

// Batch-1 path choice: the streaming pass when the selected rows amount to
// at least 96 MB (measured on GB300: OPT-175B-shaped, 121 MB: 36.9 against
// 48.2 us; OPT-30B-shaped at 50 %, 411 MB: 85.1 against 120.9 us; at 41 MB
// and below the one-launch kernel wins: OPT-13B-shaped, 21 MB: 15.0
// against 19.0 us).  DV_MLP_STREAM=1 or 0 in the environment forces it on
// or off.
bool use_stream(int d, int cap, dv_dtype dt) {
  static const int forced = [] {
    const char* e = getenv("DV_MLP_STREAM");
    return e ? atoi(e) : -1;
  }();
  if (!mlp_stream_supported(d, dt)) return false;
  if (forced >= 0) return forced != 0;
  return 2.0 * cap * d * (dt == DV_F32 ? 4 : 2) >= 96.0 * (1 << 20);
}

template <typename T>
cudaError_t mlp_t(const MlpLaunch& L, dv_dtype dt, WsHeader* hdr, int num_sms, cudaStream_t stream) {
  UpArgs u{};
  u.y = L.y; u.W1n = L.W1n;
  u.B = L.B; u.d = L.d; u.N = L.N;
  u.words = (L.N + 31) / 32;
  u.act = L.act; u.hdr = hdr;
  if (L.B == 1) {
    u.list = L.idx; u.list_count = L.count; u.member = nullptr; u.cap = L.cap;
  } else {
    u.list = L.U; u.list_count = L.U_count; u.member = L.member; u.cap = mlp_union_cap(L.B, L.N, L.cap);
  }
  u.pdl = (launch_overlap() > 0 && L.B == 1) ? 1 : 0;
  CombineLaunch c{};
  c.W = L.W2n; c.d = L.d;
  c.units = u.list; c.n_units = u.list_count; c.cap_units = u.cap; c.rpu = 1; c.n_rows_units = L.N;
  c.coef = L.act; c.coef_stride = (size_t)u.cap;
  c.member = nullptr; c.words = 0;  // the activations already carry the masks
  c.B = L.B; c.out = L.out; c.accumulate = L.accumulate; c.hdr = hdr;
  const int C = L.d / Elem<T>::kVec;
  if (L.B == 1 && use_stream(L.d, L.cap, dt)) {
    if (!L.accumulate) {  // the streaming pass adds into out
      cudaError_t e = cudaMemsetAsync(L.out, 0, (size_t)L.d * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
    return launch_mlp_stream(L.y, L.d, L.N, L.W1n, L.W2n, L.idx, L.count, L.cap, dt, L.out, hdr, num_sms,
                             u.pdl, stream);
  }
  if (L.B == 1 && L.ctr) {  // one launch for both products when its grid fits at once
    UpArgs f = u;
    f.tl = up_tpr_log2(C, 5);
    const int rpcf = (kThreads >> f.tl) * 4;
    const int nA = (f.cap + rpcf - 1) / rpcf;
    const int nB = (C + kRcCW - 1) / kRcCW;
    if (fused_fits<T>(nA + nB, num_sms))
      return launch_k(mlp_fused_kernel<T>, dim3(nA + nB), dim3(kThreads), 0, stream, f.pdl != 0, 1, f, c,
                      nA, L.ctr, wait_limit_ns());
  }
  u.tl = up_tpr_log2(C, kUpC);
  const int rpc = (kThreads >> u.tl) * kUpR;
  const int grid = (u.cap + rpc - 1) / rpc;
  for (int b0 = 0; b0 < L.B;) {
    const int nb = L.B - b0;
    const int bt = nb >= 4 ? 4 : (nb >= 2 ? 2 : 1);
    u.b0 = b0;
    cudaError_t e;
    switch (bt) {
      case 4: e = launch_up<T, 4>(u, grid, stream); break;
      case 2: e = launch_up<T, 2>(u, grid, stream); break;
      default: e = launch_up<T, 1>(u, grid, stream); break;
    }
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return launch_rows_combine(c, dt, stream);
}

}  // namespace

int mlp_union_cap(int B, int N, int cap) {
  const long long m = (long long)B * cap;
  return m < N ? (int)m : N;
}

cudaError_t launch_union(const int32_t* idx, int cap, const int32_t* count, int B, int N,
                         int32_t* U, int32_t* U_count, uint32_t* member, int32_t* slot_of,
                         WsHeader* hdr, cudaStream_t stream, uint32_t* clear, const RowsExpand* ex) {
  const size_t words = (size_t)((N + 31) / 32);
  if ((long long)B * cap > 8192 && !clear) {  // two passes: a CTA per row, then the list
    if (B > kUnionMaxB || words > (size_t)1024 * kUnionMaxWW) return cudaErrorInvalidValue;
    union_rows_kernel<<<B, 1024, words * sizeof(uint32_t), stream>>>(idx, cap, count, N, member, hdr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    union_list_kernel<<<1, 1024, 0, stream>>>(member, B, N, U, U_count, slot_of);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(2);
    return e;
  }
  const size_t smem = words * sizeof(uint32_t);
  const RowsExpand none{};
  union_kernel<<<1, 1024, smem, stream>>>(idx, cap, count, B, N, U, U_count, member, slot_of, hdr, clear,
                                          ex ? *ex : none);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

cudaError_t launch_sparse_mlp(const MlpLaunch& L, dv_dtype dt, WsHeader* hdr, int num_sms,
                              cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  const bool tc = L.B > 1 && tc_mlp_supported(L.B, L.d, dt);
  if (!L.accumulate && tc) {  // the tensor-core path adds into out with atomics
    e = cudaMemsetAsync(L.out, 0, (size_t)L.B * L.d * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  if (L.B > 1) {
    e = launch_union(L.idx, L.cap, L.count, L.B, L.N, L.U, L.U_count, L.member, nullptr, hdr, stream);
    if (e != cudaSuccess) return e;
  }
  if (tc) return launch_sparse_mlp_tc(L, dt, hdr, stream);
  switch (dt) {
    case DV_F32: return mlp_t<float>(L, dt, hdr, num_sms, stream);
    case DV_F16: return mlp_t<__half>(L, dt, hdr, num_sms, stream);
    case DV_BF16: return mlp_t<__nv_bfloat16>(L, dt, hdr, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

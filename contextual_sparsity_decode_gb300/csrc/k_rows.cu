// Weighted sum of selected weight rows, column-sliced:
//     out_b[c] (+)= sum_u sum_{t < rpu} coef_b[u * rpu + t] * W[units[u] * rpu + t][c]
// Both sparse blocks end with this contraction over the rows their set
// selects: the output projection sum_{i in S_A} H_i W_i^O (Deja Vu reading
// notes, "Sparsified Attention"; rpu = d_h rows per head) and the second MLP
// product sum_{j in S_M} a_j W^2[:, j] ("Sparsified MLP"; rpu = 1).
//
// A CTA owns kCW 16-byte column chunks of out and walks every selected row,
// so each output element is produced by exactly one CTA: no atomics, and the
// summation order is fixed.  Memory round trips are the cost that matters,
// so a batch of rows takes two: the unit ids (staged in shared memory) and
// the thread's coefficients are loaded together, then all kPL row loads of
// the thread are issued before any is used.

#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kThreads = 256;
constexpr int kCW = 4;                   // 16-byte column chunks per CTA
constexpr int kNRG = kThreads / kCW;     // row groups
constexpr int kPL = 16;                  // rows per thread per batch
constexpr int kUnitsMax = 1024;          // unit ids staged per batch

template <typename T, int BT>
__global__ void __launch_bounds__(kThreads) rows_combine_kernel(CombineLaunch a, int b0) {
  constexpr int V = Elem<T>::kVec;
  __shared__ float red[kThreads / 32][kCW][BT][V];
  __shared__ int unit_s[kUnitsMax];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int c = tid % kCW, rg = tid / kCW;
  const int C = a.d / V;
  const int chunk = blockIdx.x * kCW + c;
  const int nb = min(BT, a.B - b0);
  const int n_units = max(0, min(*a.n_units, a.cap_units));
  const int R = n_units * a.rpu;
  const T* W = static_cast<const T*>(a.W);

  float acc[BT][V];
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[b][v] = 0.f;

  // a batch covers kPL * kNRG rows and at most kUnitsMax units
  const int rows_per_batch = min(kPL * kNRG, kUnitsMax * a.rpu);
  for (int rb = 0; rb < R; rb += rows_per_batch) {
    const int re = min(R, rb + rows_per_batch);
    const int u0 = rb / a.rpu, u1 = (re - 1) / a.rpu + 1;
    __syncthreads();  // unit_s of the previous batch is no longer read
    for (int e = tid; e < u1 - u0; e += kThreads) {
      int j = a.units[u0 + e];
      if (j < 0 || j >= a.n_rows_units) {
        set_error(a.hdr, DV_ERR_INDEX_RANGE, j);
        j = -1;
      }
      unit_s[e] = j;
    }
    __syncthreads();
    uint4 wv[kPL];
    int jr[kPL];
#pragma unroll
    for (int q = 0; q < kPL; ++q) {
      const int r = rb + rg + q * kNRG;
      jr[q] = -1;
      if (r < re && chunk < C) {
        const int u = r / a.rpu;
        const int j = unit_s[u - u0];
        if (j >= 0) {
          jr[q] = j;
          wv[q] = ld_stream(W + ((size_t)j * a.rpu + (r - u * a.rpu)) * a.d + (size_t)chunk * V);
        }
      }
    }
    // The unit ids and rows above do not depend on the predecessor kernel
    // (it produces only the coefficients), so they were requested before
    // waiting for it.
    if (rb == 0) {
      grid_dep_wait();
      grid_dep_launch();  // a following layernorm may be scheduled; it waits for this kernel
    }
    float cf[kPL][BT];
#pragma unroll
    for (int q = 0; q < kPL; ++q) {
      const int r = rb + rg + q * kNRG;
#pragma unroll
      for (int b = 0; b < BT; ++b)
        cf[q][b] = (r < re && b < nb) ? a.coef[(size_t)(b0 + b) * a.coef_stride + r] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kPL; ++q) {
      if (jr[q] < 0) continue;
      float wf[V];
      unpack<T>(wv[q], wf);
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (b >= nb) break;
        if (a.member && !bit_test(a.member + (size_t)(b0 + b) * a.words, jr[q])) continue;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[b][v] = fmaf(cf[q][b], wf[v], acc[b][v]);
      }
    }
  }
  // lanes with the same column chunk: lane bits 2..4
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float x = acc[b][v];
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      if (lane < kCW) red[wid][lane][b][v] = x;
    }
  __syncthreads();
  for (int e = tid; e < kCW * BT * V; e += kThreads) {
    const int cc = e / (BT * V), b = (e / V) % BT, v = e % V;
    const int ch = blockIdx.x * kCW + cc;
    if (b >= nb || ch >= C) continue;
    float sm = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) sm += red[w][cc][b][v];
    float* o = a.out + (size_t)(b0 + b) * a.d + (size_t)ch * V + v;
    *o = a.accumulate ? *o + sm : sm;
  }
}

template <typename T>
cudaError_t combine_t(const CombineLaunch& a, cudaStream_t stream) {
  const int grid = (a.d / Elem<T>::kVec + kCW - 1) / kCW;
  for (int b0 = 0; b0 < a.B;) {
    const int nb = a.B - b0;
    const int bt = nb >= 4 ? 4 : (nb >= 2 ? 2 : 1);
    cudaError_t e;
    switch (bt) {
      case 4: e = launch_k(rows_combine_kernel<T, 4>, dim3(grid), dim3(kThreads), 0, stream, true, 1, a, b0); break;
      case 2: e = launch_k(rows_combine_kernel<T, 2>, dim3(grid), dim3(kThreads), 0, stream, true, 1, a, b0); break;
      default: e = launch_k(rows_combine_kernel<T, 1>, dim3(grid), dim3(kThreads), 0, stream, true, 1, a, b0); break;
    }
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_rows_combine(const CombineLaunch& a, dv_dtype dt, cudaStream_t stream) {
  switch (dt) {
    case DV_F32: return combine_t<float>(a, stream);
    case DV_F16: return combine_t<__half>(a, stream);
    case DV_BF16: return combine_t<__nv_bfloat16>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

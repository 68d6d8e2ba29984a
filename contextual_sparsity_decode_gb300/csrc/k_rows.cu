// Weighted sum of selected weight rows, column-sliced:
//     out_b[c] (+)= sum_u sum_{t < rpu} coef_b[u * rpu + t] * W[units[u] * rpu + t][c]
// Both sparse blocks end with this contraction over the rows their set
// selects: the output projection sum_{i in S_A} H_i W_i^O (Deja Vu reading
// notes, "Sparsified Attention"; rpu = d_h rows per head) and the second MLP
// product sum_{j in S_M} a_j W^2[:, j] ("Sparsified MLP"; rpu = 1).
//
// A CTA owns kCW 16-byte column chunks of out and walks every selected row,
// so each output element is produced by exactly one CTA: no atomics, and the
// summation order is fixed.  Threads split the rows (NRG row groups x kCW
// chunks); each issues kPL row loads before using any.  The partial sums are
// reduced across lanes with shuffles and across warps in shared memory.

#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kThreads = 256;
constexpr int kCW = 4;                   // 16-byte column chunks per CTA
constexpr int kNRG = kThreads / kCW;     // row groups
constexpr int kPL = 16;                  // row loads in flight per thread

template <typename T, int BT>
__global__ void __launch_bounds__(kThreads) rows_combine_kernel(CombineLaunch a, int b0) {
  constexpr int V = Elem<T>::kVec;
  __shared__ float red[kThreads / 32][kCW][BT][V];
  __shared__ int unit_s[1024];
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

  // units staged in shared memory, 1024 at a time
  for (int ub = 0; ub < n_units; ub += 1024) {
    const int un = min(1024, n_units - ub);
    __syncthreads();
    for (int e = tid; e < un; e += kThreads) {
      int j = a.units[ub + e];
      if (j < 0 || j >= a.n_rows_units) {
        set_error(a.hdr, DV_ERR_INDEX_RANGE, j);
        j = -1;
      }
      unit_s[e] = j;
    }
    __syncthreads();
    const int r_lo = ub * a.rpu, r_hi = min(R, (ub + un) * a.rpu);
    for (int r0 = r_lo + rg; r0 < r_hi; r0 += kPL * kNRG) {
      uint4 wv[kPL];
      int wrow[kPL];
#pragma unroll
      for (int q = 0; q < kPL; ++q) {
        const int r = r0 + q * kNRG;
        wrow[q] = -1;
        if (r < r_hi && chunk < C) {
          const int u = r / a.rpu, t = r - u * a.rpu;
          const int j = unit_s[u - ub];
          if (j >= 0) {
            wrow[q] = r;
            wv[q] = ld_stream(W + ((size_t)j * a.rpu + t) * a.d + (size_t)chunk * V);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kPL; ++q) {
        if (wrow[q] < 0) continue;
        const int r = wrow[q];
        float wf[V];
        unpack<T>(wv[q], wf);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          if (b >= nb) break;
          const int bb = b0 + b;
          if (a.member) {
            const int u = r / a.rpu;
            if (!bit_test(a.member + (size_t)bb * a.words, unit_s[u - ub])) continue;
          }
          const float cf = a.coef[(size_t)bb * a.coef_stride + r];
#pragma unroll
          for (int v = 0; v < V; ++v) acc[b][v] = fmaf(cf, wf[v], acc[b][v]);
        }
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
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w][cc][b][v];
    float* o = a.out + (size_t)(b0 + b) * a.d + (size_t)ch * V + v;
    *o = a.accumulate ? *o + s : s;
  }
}

}  // namespace

cudaError_t launch_rows_combine(const CombineLaunch& a, dv_dtype dt, cudaStream_t stream) {
  const int V = dt == DV_F32 ? 4 : 8;
  const int grid = (a.d / V + kCW - 1) / kCW;
  for (int b0 = 0; b0 < a.B;) {
    const int nb = a.B - b0;
    const int bt = nb >= 4 ? 4 : (nb >= 2 ? 2 : 1);
    switch (dt * 8 + bt) {
      case DV_F32 * 8 + 4: rows_combine_kernel<float, 4><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_F32 * 8 + 2: rows_combine_kernel<float, 2><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_F32 * 8 + 1: rows_combine_kernel<float, 1><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_F16 * 8 + 4: rows_combine_kernel<__half, 4><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_F16 * 8 + 2: rows_combine_kernel<__half, 2><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_F16 * 8 + 1: rows_combine_kernel<__half, 1><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_BF16 * 8 + 4: rows_combine_kernel<__nv_bfloat16, 4><<<grid, kThreads, 0, stream>>>(a, b0); break;
      case DV_BF16 * 8 + 2: rows_combine_kernel<__nv_bfloat16, 2><<<grid, kThreads, 0, stream>>>(a, b0); break;
      default: rows_combine_kernel<__nv_bfloat16, 1><<<grid, kThreads, 0, stream>>>(a, b0); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

}  // namespace dv

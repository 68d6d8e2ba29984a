// Weighted sum of selected weight rows, column-sliced:
//     out_b[c] (+)= sum_u sum_{t < rpu} coef_b[u * rpu + t] * W[units[u] * rpu + t][c]
// Both sparse blocks end with this contraction over the rows their set
// selects: the output projection sum_{i in S_A} H_i W_i^O (Deja Vu reading
// notes, "Sparsified Attention"; rpu = d_h rows per head) and the second MLP
// product sum_{j in S_M} a_j W^2[:, j] ("Sparsified MLP"; rpu = 1).
//
// A CTA owns kRcCW 16-byte column chunks of out and walks every selected row,
// so each output element is produced by exactly one CTA: no atomics, and the
// summation order is fixed.  Memory round trips are the cost that matters,
// so a batch of rows takes two: the unit ids (staged in shared memory) and
// the thread's coefficients are loaded together, then all kRcPL row loads of
// the thread are issued before any is used.  Coefficients are read from L2
// (they may have been written by other CTAs of the same grid).
#pragma once

#include "dv_kernels.h"

namespace dv {


constexpr int kRcThreads = 256;
constexpr int kRcCW = 4;                    // 16-byte column chunks per CTA
constexpr int kRcNRG = kRcThreads / kRcCW;  // row groups
constexpr int kRcPL = 16;                   // rows per thread per batch
constexpr int kRcUnitsMax = 1024;           // unit ids staged per batch

// One CTA (column block bx) of the combine.  `wait` runs exactly once, by all
// threads: after the first batch's unit ids and rows are requested and
// before any coefficient is read.  It waits for the producer of the
// coefficients (and of out).
template <typename T, int BT, typename Wait>
__device__ __forceinline__ void rows_combine_block(const CombineLaunch& a, int b0, int bx, Wait wait) {
  constexpr int V = Elem<T>::kVec;
  __shared__ float red[kRcThreads / 32][kRcCW][BT][V];
  __shared__ int unit_s[kRcUnitsMax];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int c = tid % kRcCW, rg = tid / kRcCW;
  const int C = a.d / V;
  const int chunk = bx * kRcCW + c;
  const int nb = min(BT, a.B - b0);
  const int n_units = max(0, min(*a.n_units, a.cap_units));
  const int R = n_units * a.rpu;
  const T* W = static_cast<const T*>(a.W);

  float acc[BT][V];
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[b][v] = 0.f;

  // a batch covers kRcPL * kRcNRG rows and at most kRcUnitsMax units
  const int rows_per_batch = min(kRcPL * kRcNRG, kRcUnitsMax * a.rpu);
  if (R == 0) wait();  // no rows: still ordered after the producer of out
  for (int rb = 0; rb < R; rb += rows_per_batch) {
    const int re = min(R, rb + rows_per_batch);
    const int u0 = rb / a.rpu, u1 = (re - 1) / a.rpu + 1;
    __syncthreads();  // unit_s of the previous batch is no longer read
    for (int e = tid; e < u1 - u0; e += kRcThreads) {
      int j = a.units[u0 + e];
      if (j < 0 || j >= a.n_rows_units) {
        set_error(a.hdr, DV_ERR_INDEX_RANGE, j);
        j = -1;
      }
      unit_s[e] = j;
    }
    __syncthreads();
    uint4 wv[kRcPL];
    int jr[kRcPL];
#pragma unroll
    for (int q = 0; q < kRcPL; ++q) {
      const int r = rb + rg + q * kRcNRG;
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
    // The unit ids and rows above do not depend on the producer of the
    // coefficients, so they were requested before waiting for it.
    if (rb == 0) wait();
    float cf[kRcPL][BT];
#pragma unroll
    for (int q = 0; q < kRcPL; ++q) {
      const int r = rb + rg + q * kRcNRG;
#pragma unroll
      for (int b = 0; b < BT; ++b)
        cf[q][b] = (r < re && b < nb) ? __ldcg(a.coef + (size_t)(b0 + b) * a.coef_stride + r) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kRcPL; ++q) {
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
      if (lane < kRcCW) red[wid][lane][b][v] = x;
    }
  __syncthreads();
  for (int e = tid; e < kRcCW * BT * V; e += kRcThreads) {
    const int cc = e / (BT * V), b = (e / V) % BT, v = e % V;
    const int ch = bx * kRcCW + cc;
    if (b >= nb || ch >= C) continue;
    float sm = 0.f;
#pragma unroll
    for (int w = 0; w < kRcThreads / 32; ++w) sm += red[w][cc][b][v];
    float* o = a.out + (size_t)(b0 + b) * a.d + (size_t)ch * V + v;
    *o = a.accumulate ? *o + sm : sm;
  }
}


}  // namespace dv

// Batch-1 sparsified MLP as one streaming pass over the selected rows
// (Deja Vu reading notes, "Sparsified MLP"; the fused gather of
// "用Deja Vu来提高 LLM 的推理速度" §3.2 with the rows of §3.3 contiguous).
//
//     out (+)= sum_{j in S} ReLU(W^1[j] . y) W^2[j]
//
// Each selected neuron owns two contiguous rows, W1n[j] and W2n[j], and
// neither depends on anything computed in this call, so both can be in
// flight from the start: the only dependency inside a neuron is that its
// W^2 row is scaled by the activation computed from its W^1 row.  Persistent
// CTAs (two per SM) each take a contiguous share of the neuron list.  One
// elected thread streams the share's rows into a ring of shared-memory
// stages with bulk copies (cp.async.bulk, completing on an mbarrier); all
// threads take a stage as it lands: the row dots with y (y held in
// registers, one 16-byte chunk slice per thread), one block reduction per
// stage, ReLU, then the W^2 rows scaled into the thread's slice of a
// private output accumulator.  At the end every CTA adds its accumulator to
// out with 16-byte vector atomics (so out must hold 0 or the residual
// before the call, and the summation order across CTAs is not fixed).  The
// path pays off for long lists of long rows, where each CTA streams several
// hundred KB; a stage is one or more whole neurons (measured on GB300:
// stages of one row each, with a block barrier per row, were 1.1-1.4x
// slower).
//
// Every wait is bounded (dv_set_wait_limit_ns) and reports DV_ERR_TIMEOUT;
// a CTA that gives up still waits (at least two seconds) for the copies it
// issued before it exits.

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kSThreads = 256;
constexpr int kMaxSt = 6;       // ring stages
constexpr int kMaxR = 8;        // neurons per stage
constexpr int kMaxItems = 512;  // neurons per CTA
constexpr long long kUnwindNs = 2000000000LL;
constexpr int kMaxRing = 160 * 1024;  // shared-memory ring, at most

struct StreamMlpArgs {
  const void* y;
  const void* W1n;
  const void* W2n;
  const int32_t* list;
  const int32_t* list_count;
  int cap, N, d;
  int R, S;             // neurons per stage, stages
  uint32_t row_bytes;   // d * sizeof(T)
  float* out;
  WsHeader* hdr;
  long long wait_ns;
  int pdl;              // launched with overlap: list and rows are read before the wait for y
};

template <typename T, int kCh>
__global__ void __launch_bounds__(kSThreads) mlp_stream_kernel(StreamMlpArgs a) {
  constexpr int V = Elem<T>::kVec;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxSt];
  __shared__ float red[kSThreads / 32][kMaxR];
  __shared__ int nid_s[kMaxItems];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int C = a.d / V;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;

  // Launched with overlap (pdl), the kernel may start while the producer of
  // y still runs: the list, its count and the weight rows are read (and the
  // first stages requested) before grid_dep_wait(), y only after it.
  if (!a.pdl) grid_dep_wait();
  const int cnt = max(0, min(*a.list_count, a.cap));
  const int G = (int)gridDim.x, g = (int)blockIdx.x;
  const int r0 = (int)((long long)cnt * g / G), r1 = (int)((long long)cnt * (g + 1) / G);
  const int n = min(r1 - r0, kMaxItems);
  if (n == 0) return;  // uniform: nothing to add
  for (int e = tid; e < n; e += kSThreads) {
    int j = a.list[r0 + e];
    if (j < 0 || j >= a.N) {
      set_error(a.hdr, DV_ERR_INDEX_RANGE, j);
      j = -1;
    }
    nid_s[e] = j;
  }
  if (tid == 0) {
    for (int s = 0; s < a.S; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  const int nst = (n + a.R - 1) / a.R;
  const size_t stage_bytes = (size_t)a.R * 2 * a.row_bytes;
  const T* W1 = static_cast<const T*>(a.W1n);
  const T* W2 = static_cast<const T*>(a.W2n);
  int issued = 0;  // thread 0 only
  auto issue = [&](int q) {
    uint8_t* buf = ring + (size_t)(q % a.S) * stage_bytes;
    const int i0 = q * a.R, i1 = min(n, i0 + a.R);
    uint32_t bytes = 0;
    for (int it = i0; it < i1; ++it)
      if (nid_s[it] >= 0) bytes += 2 * a.row_bytes;
    tc::mbar_arrive_expect_tx(&full[q % a.S], bytes);
    for (int it = i0; it < i1; ++it) {
      const int j = nid_s[it];
      if (j < 0) continue;
      uint8_t* dst = buf + (size_t)(it - i0) * 2 * a.row_bytes;
      tc::bulk_g2s(dst, W1 + (size_t)j * a.d, a.row_bytes, &full[q % a.S]);
      tc::bulk_g2s(dst + a.row_bytes, W2 + (size_t)j * a.d, a.row_bytes, &full[q % a.S]);
    }
    issued = q + 1;
  };
  if (tid == 0)
    for (int q = 0; q < min(a.S - 1, nst); ++q) issue(q);
  if (a.pdl) grid_dep_wait();  // y (and out) come from the kernels before this one
  grid_dep_launch();
  const T* y = static_cast<const T*>(a.y);
  uint4 yr[kCh];
#pragma unroll
  for (int k = 0; k < kCh; ++k) {
    const int c = tid + k * kSThreads;
    yr[k] = c < C ? ld_cached(y + (size_t)c * V) : make_uint4(0u, 0u, 0u, 0u);
  }

  float acc[kCh][V];
#pragma unroll
  for (int k = 0; k < kCh; ++k)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[k][v] = 0.f;

  int q = 0;
  for (; q < nst; ++q) {
    // the stage issued now was last read in iteration q - 1, which every
    // thread has left (barrier at the end of each iteration)
    if (tid == 0 && q + a.S - 1 < nst) issue(q + a.S - 1);
    const bool landed = tc::mbar_wait(&full[q % a.S], (q / a.S) & 1, a.wait_ns);
    if (!__syncthreads_and(landed)) {
      if (tid == 0) set_error(a.hdr, DV_ERR_TIMEOUT, q);
      break;
    }
    const uint8_t* buf = ring + (size_t)(q % a.S) * stage_bytes;
    const int nit = min(a.R, n - q * a.R);
    float part[kMaxR];
#pragma unroll
    for (int it = 0; it < kMaxR; ++it) {
      part[it] = 0.f;
      if (it < nit) {
        const uint4* w1 = reinterpret_cast<const uint4*>(buf + (size_t)it * 2 * a.row_bytes);
#pragma unroll
        for (int k = 0; k < kCh; ++k) {
          const int c = tid + k * kSThreads;
          if (c < C) {
            float wf[V], xf[V];
            unpack<T>(w1[c], wf);
            unpack<T>(yr[k], xf);
#pragma unroll
            for (int v = 0; v < V; ++v) part[it] = fmaf(wf[v], xf[v], part[it]);
          }
        }
        part[it] = warp_sum(part[it]);
      }
    }
    if (lane == 0)
#pragma unroll
      for (int it = 0; it < kMaxR; ++it)
        if (it < nit) red[wid][it] = part[it];
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kMaxR; ++it) {
      if (it >= nit) break;
      if (nid_s[q * a.R + it] < 0) continue;  // skipped (out of range): no rows were copied
      float z = 0.f;
#pragma unroll
      for (int w = 0; w < kSThreads / 32; ++w) z += red[w][it];
      const float act = fmaxf(z, 0.f);
      const uint4* w2 = reinterpret_cast<const uint4*>(buf + (size_t)it * 2 * a.row_bytes + a.row_bytes);
#pragma unroll
      for (int k = 0; k < kCh; ++k) {
        const int c = tid + k * kSThreads;
        if (c < C) {
          float wf[V];
          unpack<T>(w2[c], wf);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[k][v] = fmaf(act, wf[v], acc[k][v]);
        }
      }
    }
    __syncthreads();  // the stage and red are rewritten next
  }
  // a CTA that gave up waits for the copies it issued before it exits
  if (tid == 0)
    for (int qq = q; qq < issued; ++qq)
      if (!tc::mbar_wait(&full[qq % a.S], (qq / a.S) & 1, unwind_ns)) break;
  if (q < nst) return;  // timed out: out is left as it is
#pragma unroll
  for (int k = 0; k < kCh; ++k) {
    const int c = tid + k * kSThreads;
    if (c < C) {
      float* o = a.out + (size_t)c * V;
#pragma unroll
      for (int v = 0; v < V; v += 4) atomic_add_f32x4(o + v, acc[k][v], acc[k][v + 1], acc[k][v + 2], acc[k][v + 3]);
    }
  }
}

// The attention output projection at batch 1 as a streaming pass:
//     out (+)= sum_{u < |S_A|} sum_{t < d_h} H[u][t] W^O[head_u][t]
// (Deja Vu reading notes, "Sparsified Attention"), column-sliced: CTA
// (c, s) owns the 512-byte column slice c of out and the s-th share of the
// selected heads' W^O rows (a head's d_h rows are contiguous), and streams
// its rows' slices as 16-row TMA tiles (plain row-major boxes) through an
// 8-stage ring.  The first stages are requested before the wait for the
// kernel that writes H, so they arrive while the softmax runs.  Each thread
// owns 4 bytes of the slice; at the end it adds its columns into out, so
// every output element takes one atomic per row share (~6) instead of one
// per CTA (a CTA per share of rows over all d columns added 304 x d floats
// into the same d addresses).
constexpr int kTRows = 16;                   // rows per tile
constexpr int kTSlice = 512;                 // bytes of a row per tile (the column slice)
constexpr int kTSt = 8;                      // ring stages
constexpr int kTThreads = kTSlice / 4;       // 4 bytes of the slice per thread
constexpr int kTStage = kTRows * kTSlice;    // 8 KB

struct TileRowsArgs {
  const int32_t* units;     // selected heads
  const int32_t* n_units;   // device count
  int cap, n_rows_units, rpu, d;
  int rs;                   // row shares (grid y)
  const float* coef;        // [cap][rpu]
  float* out;
  WsHeader* hdr;
  long long wait_ns;
};

template <typename T>
__global__ void __launch_bounds__(kTThreads)
    rows_stream_kernel(const __grid_constant__ CUtensorMap mapW, TileRowsArgs a) {
  constexpr int EPT = 4 / (int)sizeof(T);          // elements of the slice per thread
  constexpr int CWe = kTSlice / (int)sizeof(T);    // slice width in elements
  extern __shared__ __align__(128) uint8_t ring[];  // [kTSt][kTRows][kTSlice], then the coefficients
  __shared__ uint64_t full[kTSt];
  const int tid = threadIdx.x;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int cs = (int)blockIdx.x, share = (int)blockIdx.y;
  // unit list and weight rows do not depend on the kernel before this one
  const int cnt = max(0, min(*a.n_units, a.cap));
  const int tpu = a.rpu / kTRows;  // tiles per head
  const int tot = cnt * tpu;
  const int t0 = (int)((long long)tot * share / a.rs), t1 = (int)((long long)tot * (share + 1) / a.rs);
  const int nt = t1 - t0;
  if (nt <= 0) {
    grid_dep_wait();
    grid_dep_launch();
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kTSt; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  auto head_of = [&](int tt) { return a.units[tt / tpu]; };
  int issued = 0;  // thread 0 only
  auto issue = [&](int q) {
    const int tt = t0 + q, j = head_of(tt);
    uint64_t* bar = &full[q % kTSt];
    if (j < 0 || j >= a.n_rows_units) {  // reported below; the stage completes empty
      tc::mbar_arrive(bar);
    } else {
      tc::mbar_arrive_expect_tx(bar, kTStage);
      tc::tma_load_2d(ring + (size_t)(q % kTSt) * kTStage, &mapW, cs * CWe, j * a.rpu + (tt % tpu) * kTRows, bar);
    }
    issued = q + 1;
  };
  if (tid == 0)
    for (int q = 0; q < min(kTSt, nt); ++q) issue(q);
  grid_dep_wait();  // H (and out) come from the kernels before this one
  grid_dep_launch();
  float* cf = reinterpret_cast<float*>(ring + (size_t)kTSt * kTStage);
  for (int e = tid; e < nt * kTRows; e += kTThreads) cf[e] = __ldcg(a.coef + (size_t)t0 * kTRows + e);
  __syncthreads();
  float acc[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
  int q = 0;
  for (; q < nt; ++q) {
    const bool landed = tc::mbar_wait(&full[q % kTSt], (q / kTSt) & 1, a.wait_ns);
    if (!__syncthreads_and(landed)) {
      if (tid == 0) set_error(a.hdr, DV_ERR_TIMEOUT, q);
      break;
    }
    const int j = head_of(t0 + q);
    if (j >= 0 && j < a.n_rows_units) {
      const uint8_t* buf = ring + (size_t)(q % kTSt) * kTStage + tid * 4;
#pragma unroll
      for (int r = 0; r < kTRows; ++r) {
        const float c = cf[q * kTRows + r];
        const uint32_t w = *reinterpret_cast<const uint32_t*>(buf + r * kTSlice);
        if (EPT == 2) {
          float lo, hi;
          if (sizeof(T) == 2 && std::is_same<T, __half>::value) {
            const __half2 h2 = *reinterpret_cast<const __half2*>(&w);
            lo = __low2float(h2); hi = __high2float(h2);
          } else {
            lo = __uint_as_float(w << 16); hi = __uint_as_float(w & 0xffff0000u);
          }
          acc[0] = fmaf(c, lo, acc[0]);
          acc[EPT - 1] = fmaf(c, hi, acc[EPT - 1]);
        } else {
          acc[0] = fmaf(c, __uint_as_float(w), acc[0]);
        }
      }
    } else if (tid == 0 && (t0 + q) % tpu == 0) {
      set_error(a.hdr, DV_ERR_INDEX_RANGE, j);
    }
    __syncthreads();  // the stage is rewritten next
    if (tid == 0 && q + kTSt < nt) issue(q + kTSt);
  }
  if (tid == 0)
    for (int qq = q; qq < issued; ++qq)
      if (!tc::mbar_wait(&full[qq % kTSt], (qq / kTSt) & 1, unwind_ns)) break;
  if (q < nt) return;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int c = cs * CWe + tid * EPT + e;
    if (c < a.d) atomicAdd(a.out + c, acc[e]);
  }
}

template <typename T>
cudaError_t rows_stream_t(const TileRowsArgs& a0, const void* W, int num_sms, cudaStream_t stream) {
  TileRowsArgs a = a0;
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int CWe = kTSlice / (int)sizeof(T);
  CUtensorMap mW;
  if (!make_map_rows(&mW, W, (int)sizeof(T), bf16, a.d, (uint64_t)a.n_rows_units * a.rpu, CWe, kTRows))
    return cudaErrorInvalidValue;
  const int ncs = (a.d + CWe - 1) / CWe;
  a.rs = max(1, min(a.cap * (a.rpu / kTRows), (2 * num_sms + ncs - 1) / ncs));
  const int max_tiles = (a.cap * (a.rpu / kTRows) + a.rs - 1) / a.rs;
  const size_t smem = (size_t)kTSt * kTStage + (size_t)max_tiles * kTRows * sizeof(float);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [] {
    return (int)cudaFuncSetAttribute(rows_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxRing);
  });
  if (ea != cudaSuccess) return ea;
  if (smem > (size_t)kMaxRing) return cudaErrorInvalidValue;
  return launch_k(rows_stream_kernel<T>, dim3(ncs, a.rs), dim3(kTThreads), smem, stream, true, 1, mW, a);
}

template <typename T, int kCh>
cudaError_t launch_stream_ch(const StreamMlpArgs& a, int grid, size_t smem, cudaStream_t stream) {
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [] {
    return (int)cudaFuncSetAttribute(mlp_stream_kernel<T, kCh>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxRing);
  });
  if (ea != cudaSuccess) return ea;
  return launch_k(mlp_stream_kernel<T, kCh>, dim3(grid), dim3(kSThreads), smem, stream, a.pdl != 0, 1, a);
}

template <typename T>
cudaError_t stream_t(const StreamMlpArgs& a0, int num_sms, cudaStream_t stream) {
  StreamMlpArgs a = a0;
  constexpr int V = Elem<T>::kVec;
  const int C = a.d / V;
  a.row_bytes = (uint32_t)(a.d * sizeof(T));
  // stages of ~32 KB (at least one neuron: two rows), ~100 KB of ring per CTA
  a.R = max(1, min(kMaxR, (int)(32768 / (2 * a.row_bytes))));
  const size_t stage = (size_t)a.R * 2 * a.row_bytes;
  a.S = max(2, min(kMaxSt, (int)((100 * 1024) / stage)));
  const size_t smem = stage * a.S;
  // two CTAs per SM, each with at most kMaxItems neurons
  const int grid = max(2 * num_sms, (a.cap + kMaxItems - 1) / kMaxItems);
  const int ch = (C + kSThreads - 1) / kSThreads;
  if (ch <= 1) return launch_stream_ch<T, 1>(a, grid, smem, stream);
  if (ch <= 2) return launch_stream_ch<T, 2>(a, grid, smem, stream);
  if (ch <= 3) return launch_stream_ch<T, 3>(a, grid, smem, stream);
  if (ch <= 4) return launch_stream_ch<T, 4>(a, grid, smem, stream);
  if (ch <= 6) return launch_stream_ch<T, 6>(a, grid, smem, stream);
  return launch_stream_ch<T, 8>(a, grid, smem, stream);
}

}  // namespace

bool mlp_stream_supported(int d, dv_dtype dt) {
  const int V = dt == DV_F32 ? 4 : 8;
  const size_t row = (size_t)d * (dt == DV_F32 ? 4 : 2);
  // two stages of one neuron (two rows) fit the ring; the thread slices
  // cover a row in at most 8 chunks
  return d / V <= 8 * kSThreads && 2 * (2 * row) <= (size_t)kMaxRing;
}

cudaError_t launch_mlp_stream(const void* y, int d, int N, const void* W1n, const void* W2n,
                              const int32_t* list, const int32_t* count, int cap, dv_dtype dt, float* out,
                              WsHeader* hdr, int num_sms, int pdl, cudaStream_t stream) {
  StreamMlpArgs a{};
  a.pdl = pdl;
  a.y = y; a.W1n = W1n; a.W2n = W2n; a.list = list; a.list_count = count; a.cap = cap; a.N = N; a.d = d;
  a.out = out; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  switch (dt) {
    case DV_F32: return stream_t<float>(a, num_sms, stream);
    case DV_F16: return stream_t<__half>(a, num_sms, stream);
    case DV_BF16: return stream_t<__nv_bfloat16>(a, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_rows_stream(const void* W, const int32_t* units, const int32_t* n_units, int cap,
                               int n_rows_units, int rpu, int d, const float* coef, dv_dtype dt, float* out,
                               WsHeader* hdr, int num_sms, cudaStream_t stream) {
  if (rpu % kTRows) return cudaErrorInvalidValue;
  TileRowsArgs a{};
  a.units = units; a.n_units = n_units; a.cap = cap; a.n_rows_units = n_rows_units; a.rpu = rpu;
  a.d = d; a.coef = coef; a.out = out; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  switch (dt) {
    case DV_F32: return rows_stream_t<float>(a, W, num_sms, stream);
    case DV_F16: return rows_stream_t<__half>(a, W, num_sms, stream);
    case DV_BF16: return rows_stream_t<__nv_bfloat16>(a, W, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

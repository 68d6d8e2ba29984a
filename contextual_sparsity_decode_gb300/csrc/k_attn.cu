// Sparsified attention with KV repair (Deja Vu reading notes, "Sparsified
// Attention": MHA_{S_A}(y) = sum_{i in S_A} H_i(y) W_i^O with
// H_i(y) = D_i(y)^-1 exp(y W_i^Q (W_i^K)^T X^T) X W_i^V; and "Sparsity operator
// for Attention": skipped heads keep the token embedding and have their K/V
// recomputed when selected later).
//
// One decode step is three kernels:
//   attn_qkv     a CTA holds a few rows of W_i^{Q,K,V} of one selected head
//                in registers (head rows are contiguous: Wqkv[i][m][t][:]) and
//                dots them with every vector that needs them: the current
//                token(s) and, for K/V rows, the stored embeddings X[j] of
//                positions whose K/V were skipped (fused repair, so a repair
//                costs no extra weight traffic).  Its last CTA also appends
//                X[pos] and writes the valid column of pos.
//   attn_decode  split-KV softmax: one thread-block cluster per (row, head),
//                each CTA a share of the positions with every K/V load of a
//                batch issued before the first use; partials are pushed into
//                rank 0's shared memory and combined after one cluster barrier.
//                Marks the repaired positions valid.
//   rows_combine out += sum_i H_i W_i^O as a weighted sum of the selected
//                heads' W^O rows, column-sliced so every output element has
//                one writer (k_rows.cu).
// The standalone repair (dv_kv_repair, e.g. a dense prefill) is a GEMM over
// the missing positions: on the tensor cores for 16-bit storage
// (k_kv_tc.cu), else the tiled CUDA-core GEMM below.

#include <cstdlib>

#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kCur = 1 << 30;      // entry flag: the current token (vector = y_b)

struct AttnArgs {
  const void* y;
  const void* Wqkv;
  const void* Wo;
  void* K;
  void* V;
  void* X;
  uint8_t* valid;
  const int32_t* pos;
  const int32_t* head_idx;
  const int32_t* head_count;
  int cap;
  const int32_t* U;
  const int32_t* U_count;
  int capU;
  const uint32_t* member;   // [B][hwords], nullptr when B == 1
  int hwords;
  const int32_t* slot_of;   // head -> union slot, nullptr when B == 1
  int B, d, h, d_h, n_max;
  float scale;
  float* q;
  float* H;
  float* out;
  WsHeader* hdr;
  // batches on the tensor-core path: attn_qkv only repairs, for the
  // (row, head) pairs the planning kernel marked
  int repair_only;
  const uint32_t* need_bits;  // [ceil(h / 32)]: heads with a skipped position in some row
  const uint8_t* miss;        // [B][h]: row b's selected head i has a skipped position
};

__device__ __forceinline__ bool member_of(const AttnArgs& a, int b, int i) {
  return a.member ? bit_test(a.member + (size_t)b * a.hwords, i) : true;
}
__device__ __forceinline__ int row_pos(const AttnArgs& a, int b) {
  const int p = a.pos[b];
  return (p >= 0 && p < a.n_max) ? p : -1;
}

// ---------------------------------------------------------------------------
// attn_qkv
//
// A CTA owns rpc = (256 / TPR) * kQR consecutive rows of one selected head's
// W^{Q,K,V} block (rpc divides d_h, so a CTA never straddles Q/K/V); a group
// of TPR threads shares kQR rows, each thread holding kQC 16-byte chunks of
// each.  All weight loads are issued before any entry is processed, and the
// registers are reused for every vector the rows are dotted with: the
// current token of every batch row that selected the head, and (K/V rows)
// the stored embedding X[j] of every position j < pos whose K/V were skipped.

constexpr int kQCMax = 4;   // chunks per thread per pass over a row that fits 1024 chunks
constexpr int kQR = 4;      // rows per thread group (divides d_h) with 3 chunks; else 2
constexpr int kNE = 2;      // vectors per group of entries
constexpr int kWin = 4096;  // positions scanned per repair window (256 x 16)

int qkv_tpr_log2(int chunks) {
  int l = 5;
  while (l < 8 && (1 << l) * kQCMax < chunks) ++l;
  return l;
}

template <typename T, int kQC, int QR>
__device__ __forceinline__ void qkv_load_w(const T* wbase, int d, int C, int cb, int tt, int tpr,
                                           uint4 (&w)[QR][kQC]) {
  constexpr int V = Elem<T>::kVec;
#pragma unroll
  for (int k = 0; k < QR; ++k)
#pragma unroll
    for (int j = 0; j < kQC; ++j) {
      const int c = cb + tt + j * tpr;
      if (c < C) w[k][j] = ld_stream(wbase + (size_t)k * d + (size_t)c * V);
    }
}

// Dots the CTA's rows with entries ent[0..n) and stores the results (q in
// fp32, K/V rounded to the storage type).  Called by all threads.  After the
// multiply-adds of the last group, `after_last_fma()` runs (all threads) while
// the partial sums wait in registers: the persistent kernel uses it to issue
// the next tile's weight loads into `w`.
template <typename T, int kQC, int QR, typename F>
__device__ void qkv_entries(const AttnArgs& a, const int* ent, int n, uint4 (&w)[QR][kQC],
                            bool one_pass, const T* wbase, int tl, int m, int tbase, int i, int u,
                            float (&red)[8][QR][kNE], const uint4 (&ycur)[kQC], bool ycur_ok,
                            F&& after_last_fma) {
  constexpr int V = Elem<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tpr = 1 << tl, RS = 256 >> tl, tt = tid & (tpr - 1);
  const int C = a.d / V;
  const T* y = static_cast<const T*>(a.y);
  const T* X = static_cast<const T*>(a.X);
  for (int g0 = 0; g0 < n; g0 += kNE) {
    const int ne = min(kNE, n - g0);
    float acc[QR][kNE];
#pragma unroll
    for (int k = 0; k < QR; ++k)
#pragma unroll
      for (int e = 0; e < kNE; ++e) acc[k][e] = 0.f;
    for (int cb = 0; cb < C; cb += tpr * kQC) {
      if (!one_pass) qkv_load_w<T, kQC, QR>(wbase, a.d, C, cb, tt, tpr, w);
#pragma unroll
      for (int j = 0; j < kQC; ++j) {
        const int c = cb + tt + j * tpr;
        if (c >= C) break;
#pragma unroll
        for (int e = 0; e < kNE; ++e) {
          if (e >= ne) break;
          const int en = ent[g0 + e];
          const int b = (en >> 20) & 1023, jp = en & 0xfffff;
          const T* vec = (en & kCur) ? y + (size_t)b * a.d : X + ((size_t)b * a.n_max + jp) * a.d;
          float xf[V];
          if ((en & kCur) && ycur_ok) unpack<T>(ycur[j], xf);  // preloaded (batch 1, one pass)
          else unpack<T>(ld_cached(vec + (size_t)c * V), xf);
#pragma unroll
          for (int k = 0; k < QR; ++k) {
            float wf[V];
            unpack<T>(w[k][j], wf);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[k][e] = fmaf(wf[v], xf[v], acc[k][e]);
          }
        }
      }
    }
    if (g0 + kNE >= n) after_last_fma();
#pragma unroll
    for (int k = 0; k < QR; ++k)
#pragma unroll
      for (int e = 0; e < kNE; ++e) {
        if (e >= ne) break;
        const float z = warp_sum(acc[k][e]);
        if (lane == 0) red[wid][k][e] = z;
      }
    __syncthreads();
    const int nw = tpr >> 5;
    for (int q = tid; q < RS * QR * ne; q += 256) {
      const int sl = q / (QR * ne), k = (q / ne) % QR, e = q % ne;
      float z = 0.f;
      for (int x = 0; x < nw; ++x) z += red[sl * nw + x][k][e];
      const int en = ent[g0 + e];
      const int b = (en >> 20) & 1023, jp = en & 0xfffff;
      const int t = tbase + sl * QR + k;
      if (m == 0) {
        a.q[((size_t)b * a.capU + u) * a.d_h + t] = z;
      } else {
        T* dst = static_cast<T*>(m == 1 ? a.K : a.V);
        dst[(((size_t)b * a.h + i) * a.n_max + jp) * a.d_h + t] = Elem<T>::from_f(z);
      }
    }
    __syncthreads();  // red is rewritten by the next group
  }
  if (n == 0) after_last_fma();
}

// Single-pass rows (every thread holds all of its chunks of the CTA's rows):
// the same products as qkv_entries, pipelined for long entry lists (KV
// repair of a head skipped for many steps).  Each thread copies its own
// chunks of the vectors of the next `stages - 1` groups into shared memory
// (cp.async, no registers held), so those loads are in flight while the
// current group is multiplied; the cross-warp sums run once per kGB groups
// (one barrier pair per 2 x kGB vectors instead of per 2).  The current
// token of a batch-1 call comes from registers (ycur) as before.
constexpr int kGB = 8;  // groups per cross-warp reduction

// Staging depth of qkv_entries_pipe (used with 3 chunks per thread): 3
// groups, 72 KB of shared memory, so two CTAs still fit on an SM.
__host__ __device__ constexpr int qkv_stages(int qc) { return qc == 3 ? 3 : 2; }
__host__ __device__ constexpr int qkv_stage_bytes(int qc) { return qkv_stages(qc) * kNE * qc * 256 * 16; }

template <int S>
__device__ __forceinline__ void cp_async_wait_stages() {
  cp_async_wait<S - 1>();
}

template <typename T, int kQC, int QR, int kStages, typename F>
__device__ void qkv_entries_pipe(const AttnArgs& a, const int* ent, int n, uint4 (&w)[QR][kQC], int tl,
                                 int m, int tbase, int i, int u, float (&redb)[8][kGB][QR][kNE],
                                 uint4* xs, const uint4 (&ycur)[kQC], bool ycur_ok, F&& after_last_fma) {
  constexpr int V = Elem<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tpr = 1 << tl, RS = 256 >> tl, tt = tid & (tpr - 1);
  const int C = a.d / V;
  const T* y = static_cast<const T*>(a.y);
  const T* X = static_cast<const T*>(a.X);
  const int ng = (n + kNE - 1) / kNE;
  // slot of (stage, entry, chunk) for this thread: consecutive threads take
  // consecutive 16-byte words (no bank conflicts)
  auto slot = [&](int st, int e, int j) { return xs + ((st * kNE + e) * kQC + j) * 256 + tid; };
  auto issue = [&](int g) {
    if (g < ng) {
      const int st = g % kStages;
#pragma unroll
      for (int e = 0; e < kNE; ++e) {
        const int idx = g * kNE + e;
        if (idx >= n) break;
        const int en = ent[idx];
        if ((en & kCur) && ycur_ok) continue;
        const int b = (en >> 20) & 1023, jp = en & 0xfffff;
        const T* vec = (en & kCur) ? y + (size_t)b * a.d : X + ((size_t)b * a.n_max + jp) * a.d;
#pragma unroll
        for (int j = 0; j < kQC; ++j) {
          const int c = tt + j * tpr;
          if (c < C) cp_async16(slot(st, e, j), vec + (size_t)c * V);
        }
      }
    }
    cp_async_commit();  // one group per call, empty or not, so the counting stays uniform
  };
#pragma unroll
  for (int g = 0; g < kStages - 1; ++g) issue(g);
  for (int gb0 = 0; gb0 < ng; gb0 += kGB) {
    const int gbn = min(kGB, ng - gb0);
    for (int q = 0; q < gbn; ++q) {
      const int g = gb0 + q;
      issue(g + kStages - 1);
      cp_async_wait_stages<kStages>();  // group g has landed (for this thread)
      const int st = g % kStages;
      float acc[QR][kNE];
#pragma unroll
      for (int k = 0; k < QR; ++k)
#pragma unroll
        for (int e = 0; e < kNE; ++e) acc[k][e] = 0.f;
#pragma unroll
      for (int j = 0; j < kQC; ++j) {
        const int c = tt + j * tpr;
        if (c >= C) break;
#pragma unroll
        for (int e = 0; e < kNE; ++e) {
          const int idx = g * kNE + e;
          if (idx >= n) break;
          float xf[V];
          if ((ent[idx] & kCur) && ycur_ok) unpack<T>(ycur[j], xf);
          else unpack<T>(*slot(st, e, j), xf);
#pragma unroll
          for (int k = 0; k < QR; ++k) {
            float wf[V];
            unpack<T>(w[k][j], wf);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[k][e] = fmaf(wf[v], xf[v], acc[k][e]);
          }
        }
      }
      if (g == ng - 1) after_last_fma();
#pragma unroll
      for (int k = 0; k < QR; ++k)
#pragma unroll
        for (int e = 0; e < kNE; ++e) {
          const float z = warp_sum(acc[k][e]);
          if (lane == 0) redb[wid][q][k][e] = z;
        }
    }
    __syncthreads();
    const int nw = tpr >> 5;
    const int per_g = RS * QR * kNE;
    for (int o = tid; o < per_g * gbn; o += 256) {
      const int q = o / per_g, r = o - q * per_g;
      const int sl = r / (QR * kNE), k = (r / kNE) % QR, e = r % kNE;
      const int idx = (gb0 + q) * kNE + e;
      if (idx >= n) continue;
      float z = 0.f;
      for (int x = 0; x < nw; ++x) z += redb[sl * nw + x][q][k][e];
      const int en = ent[idx];
      const int b = (en >> 20) & 1023, jp = en & 0xfffff;
      const int t = tbase + sl * QR + k;
      if (m == 0) {
        a.q[((size_t)b * a.capU + u) * a.d_h + t] = z;
      } else {
        T* dst = static_cast<T*>(m == 1 ? a.K : a.V);
        dst[(((size_t)b * a.h + i) * a.n_max + jp) * a.d_h + t] = Elem<T>::from_f(z);
      }
    }
    __syncthreads();  // redb is rewritten by the next batch
  }
  if (n == 0) after_last_fma();
  cp_async_wait<0>();  // nothing of this call is left in flight
}

// Persistent over tiles: CTA b takes tiles b, b + G, ... (a tile = rpc rows of
// one selected head's W^Q, W^K or W^V block).  The next tile's weights (and,
// batch 1, its valid flags) are requested right after the current tile's
// multiply-adds, so they are in flight during its reduction and stores.
template <typename T, int kQC, int QR>
__global__ void __launch_bounds__(256, 2) attn_qkv_kernel(AttnArgs a, int RG, int tl, int pdl) {
  constexpr int V = Elem<T>::kVec;
  __shared__ int ent[kWin];
  __shared__ int n_ent;
  __shared__ float red[8][QR][kNE];
  __shared__ float redb[8][kGB][QR][kNE];
  __shared__ int U_s[1024];
  extern __shared__ uint4 xs_dyn[];  // single-pass rows: staged vector chunks (qkv_entries_pipe)
  constexpr int kStg = qkv_stages(kQC);
  constexpr bool kPipe = kQC == 3;   // with 4 chunks the staging loop would spill
  const int tid = threadIdx.x;
  const int tpr = 1 << tl, RS = 256 >> tl, slot = tid >> tl, tt = tid & (tpr - 1);
  const int rpc = RS * QR;
  const int G = (int)gridDim.x;
  const int C = a.d / V;
  const bool one_pass = C <= tpr * kQC;
  // Launched with overlap (pdl), the kernel may start while the producer of
  // y still runs: head list, count, position, valid flags and weights are
  // read before grid_dep_wait(), y only after it.
  if (!pdl) grid_dep_launch();  // the decode kernel may start reading its head lists
  // round trip 1: count, head list, position and (batch 1) this thread's
  // chunks of the current token
  const int cnt_raw = *a.U_count;
  for (int e = tid; e < a.capU; e += 256) U_s[e] = a.U[e];
  const int p0 = a.B == 1 ? row_pos(a, 0) : -1;
  const bool ycur_ok = a.B == 1 && one_pass;
  uint4 ycur[kQC];
  auto load_ycur = [&]() {
    if (ycur_ok) {
#pragma unroll
      for (int j = 0; j < kQC; ++j) {
        const int c = tt + j * tpr;
        if (c < C) ycur[j] = ld_cached(static_cast<const T*>(a.y) + (size_t)c * V);
      }
    }
  };
  if (!pdl) load_ycur();
  const int nU = max(0, min(cnt_raw, a.capU));
  const int ntiles = nU * RG;
  // Bookkeeping of this call's token (after the wait for y):
  // X[b][p] = y_b and valid[b][.][p] = (head selected).  Nothing in this
  // call reads X[p] or the valid column p (repairs and the decode kernel
  // read positions < p only).
  auto append = [&]() {
    for (int b = 0; b < a.B; ++b) {
      const int p = row_pos(a, b);
      if (p < 0) {  // uniform in the CTA
        if (tid == 0) set_error(a.hdr, DV_ERR_POSITION, a.pos[b]);
        continue;
      }
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.y) + (size_t)b * a.d);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.X) + ((size_t)b * a.n_max + p) * a.d);
      for (int k0 = tid; k0 < C; k0 += 8 * 256) {  // 8 loads in flight, then 8 stores
        uint4 t8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (k0 + q * 256 < C) t8[q] = ld_cached(src + k0 + q * 256);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (k0 + q * 256 < C) dst[k0 + q * 256] = t8[q];
      }
      for (int i = tid; i < a.h; i += 256) a.valid[((size_t)b * a.h + i) * a.n_max + p] = 0;
      __syncthreads();
      const int cnt = max(0, min(a.head_count[b], a.cap));
      for (int e = tid; e < cnt; e += 256) {
        const int i = a.head_idx[(size_t)b * a.cap + e];
        if (i >= 0 && i < a.h) a.valid[((size_t)b * a.h + i) * a.n_max + p] = 1;
      }
      __syncthreads();
    }
  };
  // The last CTA has the fewest tiles (tiles are dealt round-robin), so it
  // waits for y and appends before loading its first tile; nothing else is
  // live in its registers then.
  if ((int)blockIdx.x == G - 1 && !a.repair_only) {  // repairs-only: the planning kernel appends
    grid_dep_wait();
    append();
  }
  if (a.repair_only) {
    // The current tokens' projections run on the tensor cores; this kernel
    // recomputes only the K/V rows of skipped positions, for the heads whose
    // need bit the planning kernel set (U_s is reused for their list).
    __syncthreads();  // every thread is done with U_s
    if (tid < 32) {  // one warp compacts the bitmap (h <= 1024: 32 words)
      const int lane = tid;
      const uint32_t wv = lane < (a.h + 31) / 32 ? a.need_bits[lane] : 0u;
      const int nb = __popc(wv);
      int incl = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int off = incl - nb;
      uint32_t mw = wv;
      while (mw) {
        U_s[off++] = lane * 32 + __ffs(mw) - 1;
        mw &= mw - 1;
      }
      if (lane == 31) n_ent = incl;
    }
    __syncthreads();
    const int n_need = n_ent;
    const int rg_kv = 2 * a.d_h / rpc;  // K and V rows of a head
    const int nt = n_need * rg_kv;
    __syncthreads();  // n_ent is reused below
    uint4 wr[QR][kQC];
    for (int t = blockIdx.x; t < nt; t += G) {
      const int nh = t / rg_kv;
      const int r0 = a.d_h + (t - nh * rg_kv) * rpc;
      const int i = U_s[nh];
      const int m = r0 / a.d_h, tbase = r0 - m * a.d_h;
      const T* wbase = static_cast<const T*>(a.Wqkv) + ((size_t)(i * 3 + m) * a.d_h + tbase + slot * QR) * a.d;
      bool loaded = false;
      for (int b = 0; b < a.B; ++b) {
        const int p = row_pos(a, b);
        if (p < 0 || !member_of(a, b, i) || !a.miss[(size_t)b * a.h + i]) continue;  // uniform
        const uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
        for (int base = 0; base < p; base += kWin) {
          const int j0 = base + tid * 16;
          const uint4 v4 = j0 < p ? *reinterpret_cast<const uint4*>(vr + j0)
                                  : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
          const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
          int mine = 0;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            mine += (j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
          if (!__syncthreads_or(mine)) continue;
          if (tid == 0) n_ent = 0;
          __syncthreads();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int j = j0 + k;
            if (j < p && ((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0) ent[atomicAdd(&n_ent, 1)] = (b << 20) | j;
          }
          __syncthreads();
          if (one_pass && !loaded) {
            qkv_load_w<T, kQC, QR>(wbase, a.d, C, 0, tt, tpr, wr);
            loaded = true;
          }
          uint4 ynone[kQC];
          if (kPipe && one_pass)
            qkv_entries_pipe<T, kQC, QR, kStg>(a, ent, n_ent, wr, tl, m, tbase, i, 0, redb, xs_dyn, ynone, false,
                                           []() {});
          else
            qkv_entries<T, kQC, QR>(a, ent, n_ent, wr, one_pass, wbase, tl, m, tbase, i, 0, red, ynone, false, []() {});
        }
      }
      __syncthreads();  // ent / n_ent are rebuilt for the next tile
    }
    return;
  }
  if ((int)blockIdx.x >= ntiles) return;  // uniform, before any barrier
  __syncthreads();

  uint4 w[QR][kQC];
  uint4 vflags = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
  auto meta = [&](int t, int& i, int& m, int& tbase, int& u) {
    u = t / RG;
    const int r0 = (t - u * RG) * rpc;
    i = U_s[u];
    m = r0 / a.d_h;
    tbase = r0 - m * a.d_h;
  };
  auto fetch = [&](int t) {  // weights (one pass) and batch-1 valid flags of tile t
    int i, m, tbase, u;
    meta(t, i, m, tbase, u);
    if (i < 0 || i >= a.h) return;
    const T* wb = static_cast<const T*>(a.Wqkv) + ((size_t)(i * 3 + m) * a.d_h + tbase + slot * QR) * a.d;
    if (one_pass) qkv_load_w<T, kQC, QR>(wb, a.d, C, 0, tt, tpr, w);
    vflags = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
    if (a.B == 1 && m > 0 && p0 >= 0 && p0 <= kWin && tid * 16 < p0)
      vflags = *reinterpret_cast<const uint4*>(a.valid + (size_t)i * a.n_max + tid * 16);
  };
  fetch(blockIdx.x);
  if (pdl) {
    grid_dep_wait();
    grid_dep_launch();
    load_ycur();
  }

  for (int t = blockIdx.x; t < ntiles; t += G) {
    int i, m, tbase, u;
    meta(t, i, m, tbase, u);
    const int tn = t + G;
    if (i < 0 || i >= a.h) {
      if (tid == 0 && tbase == 0 && m == 0) set_error(a.hdr, DV_ERR_INDEX_RANGE, i);
      if (tn < ntiles) fetch(tn);
      continue;
    }
    const T* wbase = static_cast<const T*>(a.Wqkv) + ((size_t)(i * 3 + m) * a.d_h + tbase + slot * QR) * a.d;
    const bool fast_scan = a.B == 1 && m > 0 && p0 >= 0 && p0 <= kWin;
    const uint4 vf = vflags;
    // entries: the current token of every row that selected head i, then
    // (K/V rows) the positions whose K/V were skipped; the batch-1 fast path
    // uses the prefetched flags (one window)
    if (tid == 0) n_ent = 0;
    __syncthreads();
    for (int b = tid; b < a.B; b += blockDim.x) {
      const int p = row_pos(a, b);
      if (p >= 0 && member_of(a, b, i)) ent[atomicAdd(&n_ent, 1)] = kCur | (b << 20) | p;
    }
    if (fast_scan) {
      const int j0 = tid * 16;
      const uint32_t w4[4] = {vf.x, vf.y, vf.z, vf.w};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int j = j0 + k;
        if (j < p0 && ((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0) ent[atomicAdd(&n_ent, 1)] = j;
      }
    }
    __syncthreads();
    const int n_first = n_ent;
    auto hook = [&]() {
      if (!(m > 0 && !fast_scan) && tn < ntiles) fetch(tn);
    };
    if (kPipe && one_pass)
      qkv_entries_pipe<T, kQC, QR, kStg>(a, ent, n_first, w, tl, m, tbase, i, u, redb, xs_dyn, ycur, ycur_ok, hook);
    else
      qkv_entries<T, kQC, QR>(a, ent, n_first, w, one_pass, wbase, tl, m, tbase, i, u, red, ycur, ycur_ok, hook);
    if (m > 0 && !fast_scan) {
      // general path (batch > 1 or pos > 4096): windows of 4096 positions
      for (int b = 0; b < a.B; ++b) {
        const int p = row_pos(a, b);
        if (p < 0 || !member_of(a, b, i)) continue;
        const uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
        for (int base = 0; base < p; base += kWin) {
          const int j0 = base + tid * 16;
          const uint4 v4 = j0 < p ? *reinterpret_cast<const uint4*>(vr + j0)
                                  : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
          const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
          int mine = 0;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            mine += (j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
          if (!__syncthreads_or(mine)) continue;
          if (tid == 0) n_ent = 0;
          __syncthreads();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int j = j0 + k;
            if (j < p && ((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0) ent[atomicAdd(&n_ent, 1)] = (b << 20) | j;
          }
          __syncthreads();
          if (kPipe && one_pass)
            qkv_entries_pipe<T, kQC, QR, kStg>(a, ent, n_ent, w, tl, m, tbase, i, u, redb, xs_dyn, ycur, false,
                                           []() {});
          else
            qkv_entries<T, kQC, QR>(a, ent, n_ent, w, one_pass, wbase, tl, m, tbase, i, u, red, ycur, false, []() {});
        }
      }
      if (tn < ntiles) fetch(tn);
    }
    __syncthreads();  // ent / n_ent are rebuilt for the next tile
  }
}

// ---------------------------------------------------------------------------
// batches on the tensor-core path: planning, row lists, coefficient split

// Which selected (row, head) pairs have a skipped position before the
// current one: miss[b][i], and need_bits (zeroed by the union kernel) for
// the heads with any such row.
// CTA (0, b) also appends row b's token: X[b][pos] = y_b and the valid
// column of pos (1 for the row's selected heads, else 0); the planning reads
// positions before pos only.
template <typename T>
__global__ void __launch_bounds__(256) repair_plan_kernel(AttnArgs a, uint32_t* need_bits, uint8_t* miss) {
  const int s = blockIdx.x, b = blockIdx.y;
  const int cnt = max(0, min(a.head_count[b], a.cap));
  if (s == 0) {
    const int p = row_pos(a, b);
    if (p < 0) {
      if (threadIdx.x == 0) set_error(a.hdr, DV_ERR_POSITION, a.pos[b]);
    } else {
      const int C = a.d / Elem<T>::kVec;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.y) + (size_t)b * a.d);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.X) + ((size_t)b * a.n_max + p) * a.d);
      for (int k = threadIdx.x; k < C; k += 256) dst[k] = ld_cached(src + k);
      for (int i = threadIdx.x; i < a.h; i += 256) a.valid[((size_t)b * a.h + i) * a.n_max + p] = 0;
      __syncthreads();
      for (int e = threadIdx.x; e < cnt; e += 256) {
        const int i = a.head_idx[(size_t)b * a.cap + e];
        if (i >= 0 && i < a.h) a.valid[((size_t)b * a.h + i) * a.n_max + p] = 1;
      }
    }
  }
  if (s >= cnt) return;
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int p = row_pos(a, b);
  if (i < 0 || i >= a.h || p < 0) return;  // reported by the other kernels
  const uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
  int any = 0;
  for (int j0 = threadIdx.x * 16; j0 < p; j0 += 256 * 16) {
    const uint4 v4 = *reinterpret_cast<const uint4*>(vr + j0);
    const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) any |= (j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
  }
  any = __syncthreads_or(any);
  if (threadIdx.x == 0) {
    miss[(size_t)b * a.h + i] = any ? 1 : 0;
    if (any) atomicOr(need_bits + (i >> 5), 1u << (i & 31));
  }
}

// The output projection's coefficients for the tensor cores: H[b][u][t] of
// the heads row b selected (0 elsewhere, and for the padding rows), split
// into two storage-type halves hi + lo, laid out [BP][Upad].
template <typename T>
__global__ void coef_split_kernel(const float* H, int B, int capU, int d_h, const int32_t* U,
                                  const int32_t* U_count, int h, const uint32_t* member, int words, T* hi, T* lo,
                                  int Upad) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x, b = blockIdx.y;
  if (k >= Upad) return;
  const int cnt = max(0, min(*U_count, h));
  float x = 0.f;
  if (b < B && k < cnt * d_h) {
    const int u = k / d_h;
    const int i = U[u];
    if (i >= 0 && i < h && bit_test(member + (size_t)b * words, i)) x = H[((size_t)b * capU + u) * d_h + (k - u * d_h)];
  }
  const T vh = Elem<T>::from_f(x);
  hi[(size_t)b * Upad + k] = vh;
  lo[(size_t)b * Upad + k] = Elem<T>::from_f(x - Elem<T>::to_f(vh));
}

// ---------------------------------------------------------------------------
// attn_decode

// E consecutive elements of a K or V row for one lane, loaded raw (one
// 4..16-byte load) and converted to floats at use.
template <typename T, int E> struct KvRaw;
template <> struct KvRaw<float, 4> {
  using type = float4;
  static __device__ __forceinline__ type load(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  static __device__ __forceinline__ void to_f(const type& v, float* f) { f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w; }
};
template <> struct KvRaw<float, 2> {
  using type = float2;
  static __device__ __forceinline__ type load(const float* p) { return __ldg(reinterpret_cast<const float2*>(p)); }
  static __device__ __forceinline__ void to_f(const type& v, float* f) { f[0] = v.x; f[1] = v.y; }
};
template <typename H16> struct KvRaw16x4 {
  using type = uint2;
  static __device__ __forceinline__ type load(const H16* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
  static __device__ __forceinline__ void to_f(const type& v, float* f) {
    float t[8];
    unpack<H16>(make_uint4(v.x, v.y, 0u, 0u), t);
    f[0] = t[0]; f[1] = t[1]; f[2] = t[2]; f[3] = t[3];
  }
};
template <typename H16> struct KvRaw16x2 {
  using type = uint32_t;
  static __device__ __forceinline__ type load(const H16* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }
  static __device__ __forceinline__ void to_f(const type& v, float* f) {
    float t[8];
    unpack<H16>(make_uint4(v, 0u, 0u, 0u), t);
    f[0] = t[0]; f[1] = t[1];
  }
};
template <> struct KvRaw<__half, 4> : KvRaw16x4<__half> {};
template <> struct KvRaw<__half, 2> : KvRaw16x2<__half> {};
template <> struct KvRaw<__nv_bfloat16, 4> : KvRaw16x4<__nv_bfloat16> {};
template <> struct KvRaw<__nv_bfloat16, 2> : KvRaw16x2<__nv_bfloat16> {};

// One thread-block cluster of CSd CTAs per (row, selected head): CTA `rank`
// takes a contiguous share of the positions 0..pos, runs the softmax over it
// in batches of 8 warps x kPW positions (every K/V load of a batch issued
// before the first use, online max/sum across batches), and pushes its
// (max, sum, numerator[d_h]) into rank 0's shared memory; after one cluster
// barrier rank 0 combines the CSd partials in rank order and writes H.
// Butterfly sums of NV values per lane over the warp (NV a power of two,
// 2 <= NV <= 16): at the step with lane bit m (16, 8, ...) each lane keeps
// the half of its values that its bit selects and adds the partner's copy of
// that half.  Afterwards lane l holds the full sum of value butterfly_pos(l);
// every value's sum sits in 32 / NV lanes.
template <int NV>
__device__ __forceinline__ float butterfly_sums(float (&v)[NV], int lane) {
  int n = NV;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool up = (lane & m) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < h) {
          const float send = up ? v[i] : v[i + h];
          const float keep = up ? v[i + h] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}
// The value index a lane holds after butterfly_sums<NV> (bits taken from the
// lane's high bits, one per halving step), and the first lane holding value j.
template <int NV>
__device__ __forceinline__ int butterfly_pos(int lane) {
  int j = 0, n = NV;
#pragma unroll
  for (int m = 16; m >= 1 && n > 1; m >>= 1, n >>= 1) j = 2 * j + ((lane & m) ? 1 : 0);
  return j;
}
template <int NV>
__device__ __forceinline__ int butterfly_lane(int j) {
  int lane = 0, n = NV, m = 16;
#pragma unroll
  for (int b = NV >> 1; b >= 1; b >>= 1, m >>= 1) lane |= (j & b) ? m : 0;
  (void)n;
  return lane;
}

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxCSd = 16;  // CTAs per decode cluster, at most

template <typename T, int DH>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(AttnArgs a) {
  constexpr int E = DH / 32;
  constexpr int kPW = 16;                              // positions per warp per batch
  constexpr int kPB = sizeof(T) == 2 ? kPW : kPW / 2;  // loads issued together
  using Raw = typename KvRaw<T, E>::type;
  __shared__ float sm[kDecWarps], sl[kDecWarps];
  __shared__ float sacc[kDecWarps][DH];
  __shared__ float cm[kMaxCSd], cl[kMaxCSd];
  __shared__ float cacc[kMaxCSd][DH];
  const int s = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int CSd = (int)gridDim.x;  // the grid is one cluster wide
  const int rank = (int)cluster_ctarank();
  const int p = row_pos(a, b);
  // count and head index are independent loads (s < cap keeps the index in bounds)
  const int cnt_raw = a.head_count[b];
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int cnt = max(0, min(cnt_raw, a.cap));
  if (s >= cnt) return;  // the whole cluster agrees
  const bool head_ok = i >= 0 && i < a.h;
  const int n_pos = p + 1;
  const int per = (n_pos + CSd - 1) / CSd;
  const int j_lo = min(n_pos, rank * per), j_hi = min(n_pos, j_lo + per);
  const T* Kr = static_cast<const T*>(a.K) + ((size_t)b * a.h + (head_ok ? i : 0)) * a.n_max * DH + lane * E;
  const T* Vr = static_cast<const T*>(a.V) + ((size_t)b * a.h + (head_ok ? i : 0)) * a.n_max * DH + lane * E;

  // Before waiting for attn_qkv: the K/V of positions it will not write.  It
  // writes only position p and the positions whose valid flag is 0 (repairs),
  // so the warp's first batch is loaded now for every position < p that is
  // valid; the others are loaded after the wait.  (The valid flags of this
  // CTA's positions are written only by this CTA, after the wait.)
  Raw kraw[kPB], vraw[kPB];
  uint32_t pre = 0;  // bit s2: position jw_first + s2 loaded before the wait
  const int jw_first = j_lo + wid * kPW;
  const int jw1_first = min(j_hi, jw_first + kPW);
  if (head_ok && p >= 0) {
    const uint8_t* vrow0 = a.valid + ((size_t)b * a.h + i) * a.n_max;
    uint8_t fl[kPB];
#pragma unroll
    for (int s2 = 0; s2 < kPB; ++s2) {
      const int j = jw_first + s2;
      fl[s2] = (j < jw1_first && j < p) ? vrow0[j] : 0;
    }
#pragma unroll
    for (int s2 = 0; s2 < kPB; ++s2) {
      if (fl[s2] == 1) {
        const int j = jw_first + s2;
        kraw[s2] = KvRaw<T, E>::load(Kr + (size_t)j * DH);
        vraw[s2] = KvRaw<T, E>::load(Vr + (size_t)j * DH);
        pre |= 1u << s2;
      }
    }
  }
  // q and the rest of K/V come from attn_qkv: everything below waits for it
  grid_dep_wait();
  grid_dep_launch();
  if (!head_ok) {
    if (tid == 0 && rank == 0) set_error(a.hdr, DV_ERR_INDEX_RANGE, i);
    return;
  }
  const int u = a.slot_of ? a.slot_of[i] : s;
  float* Hrow = a.H + ((size_t)b * a.capU + u) * DH;
  if (p < 0) {  // nothing to attend: H = 0 (attn_qkv reports the position error)
    if (rank == 0)
      for (int t = tid; t < DH; t += kDecThreads) Hrow[t] = 0.f;
    return;
  }
  cluster_arrive();  // every CTA must be running before peers push into rank 0

  float qr[E];
  const float* qg = a.q + ((size_t)b * a.capU + u) * DH + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) qr[e] = qg[e];  // the scale goes on the logits: no use of q
                                               // before the K/V loads below are issued

  float mw = -INFINITY, lw = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 1
  for (int jw0 = jw_first; jw0 < j_hi; jw0 += kDecWarps * kPW) {
    const int jw1 = min(j_hi, jw0 + kPW);
#pragma unroll 1
    for (int jb = jw0; jb < jw1; jb += kPB) {
      const uint32_t have = jb == jw_first ? pre : 0u;
#pragma unroll
      for (int s2 = 0; s2 < kPB; ++s2) {
        const int j = jb + s2;
        if (j < jw1 && !((have >> s2) & 1u)) {
          kraw[s2] = KvRaw<T, E>::load(Kr + (size_t)j * DH);
          vraw[s2] = KvRaw<T, E>::load(Vr + (size_t)j * DH);
        }
      }
      // the batch's kPB logits: per-lane partial dots, then one butterfly
      // over the warp that halves the values each lane keeps at every step
      // (kPB - 1 shuffles for the sums instead of kPB x 5) and leaves the sum
      // for position bfly_pos(lane) in lanes 2i and 2i + 1; a broadcast per
      // position gives every lane all of them
      float lg[kPB];
#pragma unroll
      for (int s2 = 0; s2 < kPB; ++s2) {
        lg[s2] = 0.f;
        if (jb + s2 < jw1) {
          float kf[E];
          KvRaw<T, E>::to_f(kraw[s2], kf);
#pragma unroll
          for (int e = 0; e < E; ++e) lg[s2] = fmaf(qr[e], kf[e], lg[s2]);
        }
      }
      const float mine = butterfly_sums<kPB>(lg, lane) * a.scale;
      float mb = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < kPB; ++s2) {
        const float v = __shfl_sync(0xffffffffu, mine, butterfly_lane<kPB>(s2));
        lg[s2] = jb + s2 < jw1 ? v : -INFINITY;
        mb = fmaxf(mb, lg[s2]);
      }
      const float mn = fmaxf(mw, mb);
      const float corr = expf(mw - mn);  // 0 on the first batch (mw = -inf)
      lw *= corr;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
      for (int s2 = 0; s2 < kPB; ++s2) {
        if (jb + s2 < jw1) {
          const float pj = expf(lg[s2] - mn);
          float vf[E];
          KvRaw<T, E>::to_f(vraw[s2], vf);
          lw += pj;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, vf[e], acc[e]);
        }
      }
      mw = mn;
    }
  }
  if (lane == 0) { sm[wid] = mw; sl[wid] = lw; }
#pragma unroll
  for (int e = 0; e < E; ++e) sacc[wid][lane * E + e] = acc[e];
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm[w]);
  cluster_wait();
  // push this CTA's partial into rank 0
  for (int t = tid; t < DH; t += kDecThreads) {
    float A = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (sm[w] != -INFINITY) A += sacc[w][t] * expf(sm[w] - M);
    st_dsmem_f32(&cacc[rank][t], 0u, A);
  }
  if (tid == 0) {
    float Lsum = 0.f;
    for (int w = 0; w < kDecWarps; ++w)
      if (sm[w] != -INFINITY) Lsum += sl[w] * expf(sm[w] - M);
    st_dsmem_f32(&cm[rank], 0u, M);
    st_dsmem_f32(&cl[rank], 0u, Lsum);
  }
  cluster_arrive();
  cluster_wait();
  // every position before p of a selected head is now present (repaired by
  // attn_qkv); marked after the barrier, whose release would otherwise wait
  // for these stores (only the next call reads the flags)
  uint8_t* vrow = a.valid + ((size_t)b * a.h + i) * a.n_max;
  for (int j = j_lo + tid; j < min(j_hi, p); j += kDecThreads) vrow[j] = 1;
  if (rank != 0) return;
  float Mg = -INFINITY;
  for (int r = 0; r < CSd; ++r) Mg = fmaxf(Mg, cm[r]);
  float den = 0.f;
  for (int r = 0; r < CSd; ++r)
    if (cm[r] != -INFINITY) den += cl[r] * expf(cm[r] - Mg);
  for (int t = tid; t < DH; t += kDecThreads) {
    float num = 0.f;
    for (int r = 0; r < CSd; ++r)
      if (cm[r] != -INFINITY) num += cacc[r][t] * expf(cm[r] - Mg);
    Hrow[t] = num / den;
  }
}

// ---------------------------------------------------------------------------
// standalone KV repair: tiled GEMM over the missing positions of a head

template <typename T>
__global__ void __launch_bounds__(256) kv_repair_gemm_kernel(AttnArgs a, int n_ct) {
  constexpr int V = Elem<T>::kVec;
  constexpr int TP = 64, TC = 64, KT = 32;
  __shared__ float Xs[KT][TP + 4];
  __shared__ float Ws[KT][TC + 4];
  __shared__ int pos_s[TP];
  __shared__ int tmp[32];
  const int tid = threadIdx.x;
  const int pt = blockIdx.x, s = blockIdx.y;
  const int b = blockIdx.z / n_ct, ct = blockIdx.z % n_ct;
  const int per_m = a.d_h / TC;
  const int m = 1 + ct / per_m, t0 = (ct % per_m) * TC;
  const int cnt = max(0, min(a.head_count[b], a.cap));
  if (s >= cnt) return;
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int p = row_pos(a, b);
  if (i < 0 || i >= a.h || p < 0) {
    if (tid == 0 && pt == 0 && ct == 0) set_error(a.hdr, p < 0 ? DV_ERR_POSITION : DV_ERR_INDEX_RANGE, p < 0 ? a.pos[b] : i);
    return;
  }
  // ranks [pt*TP, pt*TP + TP) of the ascending list of missing positions
  const uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
  int seen = 0;
  for (int base = 0; base < p; base += 256 * 16) {
    const int j0 = base + tid * 16;
    uint32_t w4[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    if (j0 < p) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(vr + j0);
      w4[0] = v4.x; w4[1] = v4.y; w4[2] = v4.z; w4[3] = v4.w;
    }
    int mine = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      mine += (j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
    int total;
    const int incl = block_inclusive_scan<256>(mine, tmp, &total);
    int rank = seen + incl - mine;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if ((j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0)) {
        const int slot = rank - pt * TP;
        if (slot >= 0 && slot < TP) pos_s[slot] = j0 + k;
        ++rank;
      }
    }
    seen += total;
  }
  const int np = min(TP, seen - pt * TP);
  __syncthreads();
  if (np <= 0) return;

  const T* X = static_cast<const T*>(a.X) + (size_t)b * a.n_max * a.d;
  const T* W = static_cast<const T*>(a.Wqkv) + ((size_t)(i * 3 + m) * a.d_h + t0) * a.d;
  const int tp = tid / 16, tc = tid % 16;
  float acc[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
  constexpr int CPRow = KT / V;  // 16-byte chunks per row per K step
  for (int k0 = 0; k0 < a.d; k0 += KT) {
    for (int e = tid; e < TP * CPRow; e += 256) {
      const int row = e / CPRow, ch = e % CPRow;
      float f[V];
      if (row < np && k0 + ch * V < a.d) {
        unpack<T>(ld_cached(X + (size_t)pos_s[row] * a.d + k0 + ch * V), f);
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) f[v] = 0.f;
      }
#pragma unroll
      for (int v = 0; v < V; ++v) Xs[ch * V + v][row] = f[v];
    }
    for (int e = tid; e < TC * CPRow; e += 256) {
      const int row = e / CPRow, ch = e % CPRow;
      float f[V];
      if (k0 + ch * V < a.d) {
        unpack<T>(ld_stream(W + (size_t)row * a.d + k0 + ch * V), f);
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) f[v] = 0.f;
      }
#pragma unroll
      for (int v = 0; v < V; ++v) Ws[ch * V + v][row] = f[v];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < KT; ++kk) {
      const float4 xa = *reinterpret_cast<const float4*>(&Xs[kk][tp * 4]);
      const float4 wb = *reinterpret_cast<const float4*>(&Ws[kk][tc * 4]);
      const float xv[4] = {xa.x, xa.y, xa.z, xa.w}, wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(xv[x], wv[y], acc[x][y]);
    }
    __syncthreads();
  }
  T* dst = static_cast<T*>(m == 1 ? a.K : a.V) + ((size_t)b * a.h + i) * a.n_max * a.d_h;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int row = tp * 4 + x;
    if (row >= np) continue;
    T* d = dst + (size_t)pos_s[row] * a.d_h + t0 + tc * 4;
#pragma unroll
    for (int y = 0; y < 4; ++y) d[y] = Elem<T>::from_f(acc[x][y]);
  }
}

__global__ void mark_valid_kernel(AttnArgs a) {
  const int s = blockIdx.x, b = blockIdx.y;
  const int cnt = max(0, min(a.head_count[b], a.cap));
  if (s >= cnt) return;
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int p = row_pos(a, b);
  if (i < 0 || i >= a.h || p < 0) return;
  uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
  for (int j = threadIdx.x; j < p; j += blockDim.x) vr[j] = 1;
}

// ---------------------------------------------------------------------------

AttnArgs make_args(const AttnLaunch& L, WsHeader* hdr) {
  AttnArgs a{};
  a.y = L.y; a.Wqkv = L.Wqkv; a.Wo = L.Wo;
  a.K = L.K; a.V = L.V; a.X = L.X; a.valid = L.valid;
  a.pos = L.pos; a.head_idx = L.head_idx; a.head_count = L.head_count; a.cap = L.cap;
  a.B = L.B; a.d = L.d; a.h = L.h; a.d_h = L.d_h; a.n_max = L.n_max;
  a.scale = L.scale;
  a.q = L.q; a.H = L.H;
  a.out = L.out; a.hdr = hdr;
  a.hwords = (L.h + 31) / 32;
  a.repair_only = 0;
  a.need_bits = L.need_bits;
  a.miss = L.miss;
  if (L.B == 1) {
    a.U = L.head_idx; a.U_count = L.head_count; a.capU = L.cap;
    a.member = nullptr; a.slot_of = nullptr;
  } else {
    a.U = L.U; a.U_count = L.U_count; a.capU = L.h;
    a.member = L.member; a.slot_of = L.slot_of;
  }
  return a;
}

template <typename T> dv_dtype dtype_of();
template <> dv_dtype dtype_of<float>() { return DV_F32; }
template <> dv_dtype dtype_of<__half>() { return DV_F16; }
template <> dv_dtype dtype_of<__nv_bfloat16>() { return DV_BF16; }

// Cluster width of the decode kernel: enough CTAs that every warp's share
// of the positions fits one batch of kPW at the cache's largest position
// (ceil(n_max / 128)), at least 8 and at most 16, as the GPU can hold such
// clusters (else 8, else 4).  Measured on the 40-layer OPT-13B-shaped step
// (n_max 1152): 9 CTAs 44.6 us per layer, 8 45.1, 10 44.9, 16 45.9, 4 48.1.
// A CTA with one batch per warp needs no second dependent round of K/V
// loads; wider clusters wait longer for room in one GPC.
template <typename T, int DH>
bool decode_width_fits(int w) {
  // per device and width: 1 yes, 2 no (the attribute and the answer belong to the device)
  static PerDevice fits[kMaxCSd + 1];
  if (w < 1 || w > kMaxCSd) return false;
  return fits[w].get(current_device(), [w] {
    if (w > 8) (void)cudaFuncSetAttribute(attn_decode_kernel<T, DH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(w, 1, 1);
    cfg.blockDim = dim3(kDecThreads);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = w;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    const int r = cudaOccupancyMaxActiveClusters(&n, attn_decode_kernel<T, DH>, &cfg) == cudaSuccess && n >= 1 ? 1 : 2;
    (void)cudaGetLastError();
    return r;
  }) == 1;
}

// With many (row, head) pairs the GPU is full anyway, and wider clusters
// only add cluster barriers, co-scheduling constraints and partial sums to
// combine: from 32 pairs on the cluster is 4 CTAs wide, from 64 pairs 2,
// from 640 pairs one CTA per pair (each warp then takes several batches of
// positions).  Measured on GB300 at OPT-30B width, ~2050 positions, whole
// layers: 896 pairs 555 / 528 / 521 us per layer at 4 / 2 / 1 wide; 448
// pairs 417 / 399 / 411 at 4 / 2 / 1; 96-112 pairs 275 / 271 and 313 / 302
// at 8 / 2 (1 wide: 286, 316); 48 pairs 211 / 201 / 208 at 16 / 4 / 2; 12
// pairs 121 / 120 / 124 at 16 / 8 / 4.
// DV_DECODE_WIDTH in the environment forces a width (1..16).
template <typename T, int DH>
int decode_cluster_width(int n_max, int pairs) {
  static const int forced = [] {
    const char* e = getenv("DV_DECODE_WIDTH");
    return e ? atoi(e) : 0;
  }();
  if (forced >= 1 && forced <= kMaxCSd && decode_width_fits<T, DH>(forced)) return forced;
  constexpr int kPos = kDecWarps * 16;  // positions per CTA in one batch (kPW = 16)
  int want = min(kMaxCSd, max(8, (n_max + kPos - 1) / kPos));
  if (pairs >= 32) want = 4;
  if (pairs >= 64) want = 2;
  if (pairs >= 640) want = 1;
  if (decode_width_fits<T, DH>(want)) return want;
  return decode_width_fits<T, DH>(8) ? 8 : 4;
}

template <typename T, int DH>
cudaError_t launch_decode_dh(const AttnArgs& a, cudaStream_t stream) {
  const int cw = decode_cluster_width<T, DH>(a.n_max, a.B * a.cap);
  return launch_k(attn_decode_kernel<T, DH>, dim3(cw, a.cap, a.B), dim3(kDecThreads), 0, stream, true, cw, a);
}

template <typename T>
cudaError_t launch_decode(const AttnArgs& a, cudaStream_t stream) {
  return a.d_h == 128 ? launch_decode_dh<T, 128>(a, stream) : launch_decode_dh<T, 64>(a, stream);
}

// Batch-1 output projection as a streaming pass when the selected W^O rows
// amount to at least 48 MB (OPT-175B-shaped: 63 MB; the column-sliced
// combine reached ~2 TB/s there).  DV_ATTN_STREAM=1 or 0 in the environment
// forces it on or off.
bool use_rows_stream(size_t bytes) {
  static const int forced = [] {
    const char* e = getenv("DV_ATTN_STREAM");
    return e ? atoi(e) : -1;
  }();
  if (forced >= 0) return forced != 0;
  return bytes >= (size_t)48 << 20;
}

template <typename T>
cudaError_t attn_t(const AttnLaunch& L, WsHeader* hdr, int num_sms, cudaStream_t stream) {
  AttnArgs a = make_args(L, hdr);
  // 1. projections + fused repair.  Rows of up to 768 16-byte chunks: 4 rows
  // of 3 chunks per thread; up to 1024 chunks: 2 rows of 4; longer rows
  // (d > 8192 for 16-bit types): 2 rows of 6 or 1 row of 8 or 10 chunks per
  // thread, so that a row is one pass of loads and the next tile's rows are
  // requested during the current tile's sums (4 rows of 4 chunks spilled
  // registers, and longer rows then took two dependent passes per tile)
  const int C = a.d / Elem<T>::kVec;
  const bool wide = C > 256 * kQCMax;
  const int tl = wide ? 8 : qkv_tpr_log2(C);
  // three chunks per thread with four rows when a row fits (fewer registers,
  // staged vectors); otherwise two rows per thread (four rows of four
  // chunks spilled registers)
  const bool three = !wide && C <= (1 << tl) * 3;
  const int qc_wide = (C + 255) / 256;  // chunks per thread of a wide row (one pass)
  const int QR = three ? kQR : (wide && qc_wide > 6 ? 1 : 2);
  const int RG = 3 * a.d_h / ((256 >> tl) * QR);
  if (a.capU > 1024) return cudaErrorInvalidValue;
  const int tiles = a.capU * RG;
  // two resident CTAs per SM at most; no more CTAs than the largest number
  // of tiles per CTA needs (768 tiles on 304 slots take 3 rounds either way,
  // and 256 CTAs leave slots for the decode kernel's CTAs to start early),
  // plus one so that the last CTA, which also appends the token, has a tile
  // fewer than the most loaded ones
  const int slots = 2 * num_sms;
  const int rounds = (tiles + slots - 1) / slots;
  const int grid = min(slots, (tiles + rounds - 1) / rounds + 1);
  // three chunks per thread when a row fits (fewer registers), else four
  const int pdl = (launch_overlap() > 0 && a.B == 1) ? 1 : 0;
  cudaError_t e;
  // batches of 2+ rows in a 16-bit type: the projections of the current
  // tokens and the output projection are dense contractions over the union
  // of the rows' heads and run on the tensor cores; attn_qkv only repairs
  const bool tc = a.B > 1 && L.rows && tc_mlp_supported(a.B, a.d, dtype_of<T>());
  if (tc) {
    repair_plan_kernel<T><<<dim3(a.cap, a.B), 256, 0, stream>>>(a, L.need_bits, L.miss);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    a.repair_only = 1;
  }
  // single-pass rows of 3 chunks stage their vectors in dynamic shared memory
  if (!tc && qkv1_tc_supported(a.B, a.d, a.d_h, a.n_max, dtype_of<T>())) {
    // batch 1: weight tiles on the tensor cores, repairs as extra columns
    Qkv1Launch q{};
    q.y = L.y; q.d = a.d; q.h = a.h; q.Wqkv = L.Wqkv;
    q.K = L.K; q.V = L.V; q.X = L.X; q.valid = L.valid; q.n_max = a.n_max; q.pos = L.pos;
    q.U = a.U; q.U_count = a.U_count; q.capU = a.capU; q.q = a.q; q.pdl = pdl;
    e = launch_qkv1_tc(q, dtype_of<T>(), hdr, stream);
  } else if (wide) {
    if (qc_wide <= 6)
      e = launch_k(attn_qkv_kernel<T, 6, 2>, dim3(grid), dim3(256), 0, stream, pdl != 0, 1, a, RG, tl, pdl);
    else if (qc_wide <= 8)
      e = launch_k(attn_qkv_kernel<T, 8, 1>, dim3(grid), dim3(256), 0, stream, pdl != 0, 1, a, RG, tl, pdl);
    else
      e = launch_k(attn_qkv_kernel<T, 10, 1>, dim3(grid), dim3(256), 0, stream, pdl != 0, 1, a, RG, tl, pdl);
  } else if (three) {
    const size_t smem = qkv_stage_bytes(3);
    static PerDevice attr3;  // function attributes are per device
    const cudaError_t ea = (cudaError_t)attr3.get(current_device(), [smem] {
      return (int)cudaFuncSetAttribute(attn_qkv_kernel<T, 3, kQR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
    });
    if (ea != cudaSuccess) return ea;
    e = launch_k(attn_qkv_kernel<T, 3, kQR>, dim3(grid), dim3(256), smem, stream, pdl != 0, 1, a, RG, tl, pdl);
  } else {
    e = launch_k(attn_qkv_kernel<T, 4, 2>, dim3(grid), dim3(256), 0, stream, pdl != 0, 1, a, RG, tl, pdl);
  }
  if (e != cudaSuccess) return e;
  if (tc) {  // the current tokens' q and K/V (the Wqkv row list comes from the union kernel)
    const int per = 3 * a.d_h;
    TcQkvLaunch q{};
    q.y = L.y; q.B = a.B; q.d = a.d; q.h = a.h; q.d_h = a.d_h; q.n_max = a.n_max; q.capQ = a.capU;
    q.Wqkv = L.Wqkv; q.rows = L.rows; q.rows_count = L.rows_count;
    q.max_rows = min(a.h, a.B * a.cap) * per;
    q.member = a.member; q.words = a.hwords; q.slot_of = a.slot_of; q.pos = a.pos;
    q.q = a.q; q.K = a.K; q.V = a.V;
    q.part = L.tc_part; q.sem = L.tc_sem;
    e = launch_qkv_tc(q, dtype_of<T>(), hdr, stream);
    if (e != cudaSuccess) return e;
  }
  // 2. split-KV softmax, one cluster per (row, head), cache bookkeeping
  e = launch_decode<T>(a, stream);
  if (e != cudaSuccess) return e;
  if (tc) {  // 3. output projection on the tensor cores (the W^O row list comes from the union kernel)
    const int Upad = tc_act_cols(a.h * a.d_h);
    const int BP = a.B <= 16 ? 16 : 32;
    coef_split_kernel<T><<<dim3((Upad + 255) / 256, BP), 256, 0, stream>>>(
        a.H, a.B, a.capU, a.d_h, a.U, a.U_count, a.h, a.member, a.hwords, static_cast<T*>(L.act_hi),
        static_cast<T*>(L.act_lo), Upad);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(2);
    if (!L.accumulate) {  // the tensor-core combine adds into out
      e = cudaMemsetAsync(L.out, 0, (size_t)a.B * a.d * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
    TcRowsLaunch r{};
    r.W = L.Wo; r.n_rows = a.h * a.d_h; r.d = a.d; r.B = a.B; r.rows_per_unit = a.d_h;
    r.rows = L.rows_o; r.rows_count = L.rows_o_count; r.max_rows = min(a.h, a.B * a.cap) * a.d_h;
    r.act_hi = L.act_hi; r.act_lo = L.act_lo; r.Upad = Upad; r.out = L.out;
    return launch_rows_tc(r, dtype_of<T>(), hdr, stream);
  }
  // 3. output projection: out (+)= sum_u sum_t H[b][u][t] Wo[U[u]][t][:]
  CombineLaunch c{};
  c.W = L.Wo; c.d = a.d;
  c.units = a.U; c.n_units = a.U_count; c.cap_units = a.capU; c.rpu = a.d_h; c.n_rows_units = a.h;
  c.coef = a.H; c.coef_stride = (size_t)a.capU * a.d_h;
  c.member = a.member; c.words = a.hwords;
  c.B = a.B; c.out = L.out; c.accumulate = L.accumulate; c.hdr = hdr;
  if (a.B == 1 && use_rows_stream((size_t)a.cap * a.d_h * a.d * sizeof(T))) {
    // long selections of long rows: stream the W^O rows (see k_stream.cu)
    if (!L.accumulate) {
      e = cudaMemsetAsync(L.out, 0, (size_t)a.d * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
    return launch_rows_stream(L.Wo, a.U, a.U_count, a.capU, a.h, a.d_h, a.d, a.H, dtype_of<T>(), L.out, hdr,
                              num_sms, stream);
  }
  return launch_rows_combine(c, dtype_of<T>(), stream);
}

template <typename T>
cudaError_t repair_t(const AttnLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  AttnArgs a = make_args(L, hdr);
  const int n_ct = 2 * a.d_h / 64;
  dim3 g((a.n_max + 63) / 64, a.cap, a.B * n_ct);
  kv_repair_gemm_kernel<T><<<g, 256, 0, stream>>>(a, n_ct);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark_valid_kernel<<<dim3(a.cap, a.B), 256, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(2);
  return e;
}

}  // namespace

cudaError_t launch_sparse_attn(const AttnLaunch& L, dv_dtype dt, WsHeader* hdr, int num_sms,
                               cudaStream_t stream) {
  if (L.B > 1) {
    RowsExpand ex{};
    if (L.rows && L.rows_o) {  // row lists of the tensor-core projections
      ex.rows[0] = L.rows; ex.count[0] = L.rows_count; ex.per[0] = 3 * L.d_h;
      ex.rows[1] = L.rows_o; ex.count[1] = L.rows_o_count; ex.per[1] = L.d_h;
    }
    cudaError_t e = launch_union(L.head_idx, L.cap, L.head_count, L.B, L.h, L.U, L.U_count,
                                 L.member, L.slot_of, hdr, stream, L.need_bits, &ex);
    if (e != cudaSuccess) return e;
  }
  switch (dt) {
    case DV_F32: return attn_t<float>(L, hdr, num_sms, stream);
    case DV_F16: return attn_t<__half>(L, hdr, num_sms, stream);
    case DV_BF16: return attn_t<__nv_bfloat16>(L, hdr, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_repair(const AttnLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (kv_tc_supported(L.d, L.d_h, dt)) return launch_kv_repair_tc(L, dt, hdr, stream);
  switch (dt) {
    case DV_F32: return repair_t<float>(L, hdr, stream);
    case DV_F16: return repair_t<__half>(L, hdr, stream);
    case DV_BF16: return repair_t<__nv_bfloat16>(L, hdr, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

// Batched sparsified MLP on the tcgen05 tensor cores.
//
// For a batch of B rows the union U of the rows' neuron sets is read once,
// which turns the gathered weight rows into a real dense contraction
// (Deja Vu reading notes, "Sparsified MLP", applied to every row with the
// row's own set as a mask):
//   up    a[u][b] = ReLU(W^1[:, U[u]] . y_b) * [U[u] in S_b]
//         M = 128 union neurons per tile, N = B padded to 16/32, K = d,
//         split over up to 8 CTAs per tile.  When the largest possible
//         union has few tiles the host sizes the split: a cluster of S CTAs
//         per tile, partials summed through distributed shared memory before
//         ReLU.  Otherwise the split is chosen on the device from the
//         union's actual size so that the grid (two CTAs per SM) fills the
//         GPU; those partial tiles are summed with fp32 atomics in L2 and the
//         tile's last CTA to finish applies the epilogue.
//         A = gathered rows of W1n (TMA gather4, 128-byte swizzle, K-major),
//         B = y (TMA tile, K-major).  Accumulator in TMEM; the epilogue writes
//         a split into two storage-type halves hi + lo (a = hi + lo to ~2^-17
//         relative), so the second product keeps fp32-level accuracy.
//   down  out[b][c] += sum_u W^2[c, U[u]] a[u][b]
//         M = 128 output columns per CTA, N = B padded, K = a chunk of U
//         (256..1024 entries, sized to fill the GPU).
//         A = gathered rows of W2n read as an MN-major operand (a neuron row
//         is 64 contiguous columns per 128-byte swizzle row), B = a_hi and
//         a_lo (two MMAs per K step).  Split-K over U with fp32 atomics.
// Weight rows that are gathered (neurons) are copied by the CTA's four
// epilogue warps with cp.async into the swizzled stage; rows that form a
// tile (an attention head's block) and the small operands come by TMA from
// one elected thread; one elected thread issues the MMAs; every wait is bounded and reports
// DV_ERR_TIMEOUT instead of hanging.  The pipeline waits use the caller's
// limit (dv_set_wait_limit_ns); the waits that unwind a CTA -- for the MMAs
// it issued and for the TMA copies still landing in its shared memory --
// take at least kUnwindNs, so no CTA frees its tensor memory or exits with
// tensor-core or copy work of its own still in flight.

#include <cuda.h>

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kTM = 128;                 // tile rows (M)
constexpr int kKB = 64;                  // K elements per stage (one 128-byte row)
// Ring depths: about 100 KB of stages per CTA, so that two CTAs share an SM
// (measured on GB300: rings of 200 KB, one CTA per SM, were 1.3-1.5x slower).
constexpr int kSU = 5;
constexpr int kSD = 4;
constexpr int kKChunk = 1024;            // union neurons per down-projection CTA, at most
constexpr long long kUnwindNs = 2000000000LL;  // two seconds
constexpr uint32_t kTmemCols = 32;
constexpr int kMaxSplit = 8;             // K splits per up-projection tile, at most
constexpr int kMinSplitKB = 24;          // K blocks per split, at least

struct UpArgs {
  const int32_t* U;
  const int32_t* U_count;
  int capU;
  const uint32_t* member;
  int words, B, d, N, Upad;
  void* act_hi;
  void* act_lo;
  WsHeader* hdr;
  long long wait_ns;
  // 1: every 128-row tile of the row list is contiguous in the weight matrix
  // (the attention's head blocks): one TMA tile load instead of 32 gathers
  int tile_rows;
  // kEpiQkv: row r of Wqkv [h * 3 * d_h][d] is (head r / (3 d_h), matrix, element)
  int h, d_h, n_max, capQ;
  const int32_t* slot_of;   // head -> slot in the batch union (q rows)
  const int32_t* pos;       // [B]
  float* q;                 // [B][capQ][d_h]
  void* K;
  void* V;
  int S;                    // > 1: CTAs (one cluster) per tile, splitting K; 1: split on the device
  float* part;              // S == 1: [tiles][BP][kTM] fp32 partial tiles, zero between calls
  int* sem;                 // S == 1: [tiles] arrival counts, zero between calls
};

// Epilogues of the up kernel: the MLP's masked ReLU split into two storage
// halves, or the attention projections (q in fp32; K/V of the current token
// rounded into the cache) of the rows that selected each head.
enum TcEpi { kEpiMlp = 0, kEpiQkv = 1 };

struct DownArgs {
  const int32_t* U;
  const int32_t* U_count;
  int capU, B, d, N;
  float* out;
  WsHeader* hdr;
  long long wait_ns;
  int tile_rows;  // 1: every 64-row chunk of the row list is contiguous (two tile loads a stage)
  int kchunk;     // union entries per CTA (grid y), a multiple of 64, <= kKChunk
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// A operand rows gathered by the four epilogue warps with cp.async: each
// thread copies eight 16-byte chunks of the stage into the 128-byte-swizzled
// K-major layout (16-byte chunk c of row r at chunk c ^ (r % 8) of the row's
// 128 bytes, rows grouped by 8 in 1024-byte atoms), waits for its copies
// S - 2 stages later, makes them visible to the async proxy and arrives on
// the stage's barrier (count 128).  Signalling S - 2 rather than S - 1
// stages back leaves the MMA of the oldest stage a stage period before its
// slot is refilled (measured on GB300: batch-32 OPT-30B-shaped MLP call 154
// -> 135 us).  TMA gather4 moves 512 bytes an instruction, which capped a
// CTA at ~13 GB/s on GB300.
// warps 0-3: loaders + epilogue; warp 4: TMA producer; warp 5: MMA issuer (the
// two single-thread roles in one warp serialised their waits: 90 against 57 us)
constexpr int kTcThreads = 192;

template <int S>
__device__ __forceinline__ bool gather_rows_pipeline(uint8_t* sA, uint32_t stage_bytes, const uint8_t* const* src,
                                                     const uint32_t* dst_off, int nk, uint32_t src_step,
                                                     uint64_t* fullA, uint64_t* empty, long long wait_ns) {
  int kb = 0, sig = 0;
  bool ok = true;
  for (; kb < nk; ++kb) {
    const int st = kb % S;
    if (kb >= S && !tc::mbar_wait(&empty[st], ((kb / S) - 1) & 1, wait_ns)) {
      ok = false;
      break;
    }
    uint8_t* base = sA + (size_t)st * stage_bytes;
#pragma unroll
    for (int q = 0; q < 8; ++q) cp_async16(base + dst_off[q], src[q] + (size_t)kb * src_step);
    cp_async_commit();
    if (kb >= S - 2) {
      cp_async_wait<S - 2>();
      tc::fence_proxy_async();
      tc::mbar_arrive(&fullA[sig % S]);
      ++sig;
    }
  }
  cp_async_wait<0>();
  tc::fence_proxy_async();
  for (; sig < kb; ++sig) tc::mbar_arrive(&fullA[sig % S]);
  return ok;
}

template <typename T, int BP, int EPI = kEpiMlp>
__global__ void __launch_bounds__(kTcThreads, 1)
    mlp_tc_up_kernel(const __grid_constant__ CUtensorMap mapY, const __grid_constant__ CUtensorMap mapT,
                     const void* W, UpArgs a) {
  constexpr uint32_t kABytes = kTM * 128, kBBytes = BP * 128;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t fullA[kSU], fullB[kSU], empty[kSU], done;
  __shared__ uint32_t tmem_base;
  __shared__ int rows[kTM];
  __shared__ int issued, consumed, flag_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int cnt = max(0, min(*a.U_count, a.capU));
  const int nk_all = a.d / kKB;
  // K splits per tile from the union's actual size (known only here): as
  // many as the grid holds, at most kMaxSplit, at least kMinSplitKB K blocks
  // each (shorter slices spend more on the pipeline's fill and the epilogue
  // than the extra CTAs gain)
  const int S = a.S;
  const int tiles = (cnt + kTM - 1) / kTM;
  const int ks = S > 1 ? S
                       : max(1, min(tiles > 0 ? (int)gridDim.x / tiles : 1, min(kMaxSplit, nk_all / kMinSplitKB)));
  const int tile = (int)blockIdx.x / ks, split = (int)blockIdx.x % ks;
  // before any barrier or TMEM use (with S > 1 the whole cluster shares the tile)
  if (tile >= tiles) return;
  const int u0 = tile * kTM;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSU * kABytes;

  if (tid < kTM) {
    int r = a.U[min(u0 + tid, cnt - 1)];
    if (r < 0 || r >= a.N) {
      set_error(a.hdr, DV_ERR_INDEX_RANGE, r);
      r = 0;
    }
    rows[tid] = r;
  }
  if (tid == 0) {
    for (int s = 0; s < kSU; ++s) {
      tc::mbar_init(&fullA[s], a.tile_rows ? 1 : kTM);
      tc::mbar_init(&fullB[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&done, 1);
    tc::fence_mbar_init();
    issued = consumed = flag_err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int kb0 = split * nk_all / ks;  // this CTA's K blocks [kb0, kb0 + nk)
  const int nk = (split + 1) * nk_all / ks - kb0;

  if (warp >= 4) {
    if (warp == 4 && lane == 0) {  // TMA producer: y (and the weight rows when they form one tile)
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kSU, it = kb / kSU;
        if (kb >= kSU && !tc::mbar_wait(&empty[s], (it - 1) & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 1);
          flag_err = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&fullB[s], kBBytes);
        tc::tma_load_2d(sB + s * kBBytes, &mapY, (kb0 + kb) * kKB, 0, &fullB[s]);
        if (a.tile_rows) {
          tc::mbar_arrive_expect_tx(&fullA[s], kABytes);
          tc::tma_load_2d(sA + s * kABytes, &mapT, (kb0 + kb) * kKB, rows[0], &fullA[s]);
        }
        issued = kb + 1;
      }
    } else if (warp == 5 && lane == 0) {  // MMA issuer
      constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
      const uint32_t idesc = tc::idesc_f16(kTM, BP, kBf16, false, false);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kSU, it = kb / kSU;
        if (!tc::mbar_wait(&fullA[s], it & 1, a.wait_ns) || !tc::mbar_wait(&fullB[s], it & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 2);
          flag_err = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t aBase = tc::saddr(sA + s * kABytes), bBase = tc::saddr(sB + s * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kKB / 16; ++kk) {
          const uint64_t ad = tc::smem_desc(aBase + kk * 32, 16, 1024, 2);
          const uint64_t bd = tc::smem_desc(bBase + kk * 32, 16, 1024, 2);
          tc::mma_f16(tmem, ad, bd, idesc, (kb | kk) != 0);
        }
        tc::mma_commit(&empty[s]);
        consumed = kb + 1;
      }
      tc::mma_commit(&done);  // arrives once every issued MMA has completed
    }
    __syncwarp();
  } else if (!a.tile_rows) {  // warps 0-3 gather the weight rows
    // thread t copies 16-byte chunk t % 8 of rows t / 8 + 16 q (q < 8): eight
    // lanes cover one row's 128 bytes, so a warp instruction reads four whole
    // 128-byte lines (a row per lane touched 32 lines: ~2.1 TB/s)
    const uint8_t* src[8];
    uint32_t off[8];
    const int ch = tid & 7;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = (tid >> 3) + 16 * q;
      src[q] = reinterpret_cast<const uint8_t*>(static_cast<const T*>(W) + (size_t)rows[r] * a.d +
                                                (size_t)kb0 * kKB + ch * 8);
      off[q] = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4));
    }
    if (!gather_rows_pipeline<kSU>(sA, kABytes, src, off, nk, kKB * sizeof(T), fullA, empty, a.wait_ns)) {
      set_error(a.hdr, DV_ERR_TIMEOUT, 7);
      flag_err = 1;
    }
  }

  // epilogue: accumulator row = tile row (union entry u0 + row)
  float v[BP];
  if (tid < kTM) {
    const bool ok = tc::mbar_wait(&done, 0, unwind_ns);
    if (!ok && lane == 0) {
      set_error(a.hdr, DV_ERR_TIMEOUT, 3);
      flag_err = 1;
    }
    __syncwarp();
    tc::fence_after_sync();
#pragma unroll
    for (int c = 0; c < BP; c += 8) tc::tmem_ld8(tmem + ((uint32_t)(warp * 32) << 16) + c, v + c);
    tc::tmem_ld_wait();
  }
  tc::fence_before_sync();
  __syncthreads();  // flag_err is final
  // no TMA write into this CTA's shared memory may still be in flight (the
  // loaders waited for their own copies); after this the ring is free
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb) {
      if (!tc::mbar_wait(&fullB[kb % kSU], (kb / kSU) & 1, unwind_ns)) break;
      if (a.tile_rows && !tc::mbar_wait(&fullA[kb % kSU], (kb / kSU) & 1, unwind_ns)) break;
    }
  }
  __syncthreads();
  const bool good = !flag_err;
  // element (tile row tr, batch row b) of the finished accumulator
  auto emit = [&](int tr, int b, float z) {
    const int u = u0 + tr;
    const bool live = good && u < cnt;
    const int row = rows[tr];
    if (EPI == kEpiMlp) {
      float x = fmaxf(z, 0.f);
      if (!live || b >= a.B || !bit_test(a.member + (size_t)b * a.words, row)) x = 0.f;
      const T h = Elem<T>::from_f(x);
      static_cast<T*>(a.act_hi)[(size_t)b * a.Upad + u] = h;
      static_cast<T*>(a.act_lo)[(size_t)b * a.Upad + u] = Elem<T>::from_f(x - Elem<T>::to_f(h));
    } else {
      if (!live || b >= a.B) return;
      const int dh3 = 3 * a.d_h;
      const int i = row / dh3, rem = row - i * dh3, m = rem / a.d_h, t = rem - m * a.d_h;
      if (!bit_test(a.member + (size_t)b * a.words, i)) return;
      if (m == 0) {
        a.q[((size_t)b * a.capQ + a.slot_of[i]) * a.d_h + t] = z;
      } else {
        const int p = a.pos[b];
        T* dst = static_cast<T*>(m == 1 ? a.K : a.V);
        if (p >= 0 && p < a.n_max) dst[(((size_t)b * a.h + i) * a.n_max + p) * a.d_h + t] = Elem<T>::from_f(z);
      }
    }
  };
  if (ks == 1) {
    if (tid < kTM) {
#pragma unroll
      for (int b = 0; b < BP; ++b) emit(tid, b, v[b]);
    }
  } else if (S > 1) {
    // park the partial tile in the (now idle) ring, then sum rows
    // [split * span, +span) over the cluster's partials
    float* red = reinterpret_cast<float*>(sA);  // [128][BP + 1]
    if (tid < kTM) {
#pragma unroll
      for (int b = 0; b < BP; ++b) red[tid * (BP + 1) + b] = good ? v[b] : 0.f;
    }
    cluster_arrive();
    cluster_wait();
    const int span = (kTM + S - 1) / S, r0 = split * span, nr = max(0, min(kTM - r0, span));
    for (int e = tid; e < nr * BP; e += kTcThreads) {
      const int b = e / nr, tr = r0 + (e - b * nr);
      float z = 0.f;
      for (int q = 0; q < S; ++q) z += ld_dsmem_f32(red + tr * (BP + 1) + b, (uint32_t)q);
      emit(tr, b, z);
    }
    cluster_arrive();  // no CTA leaves while another reads its partials
    cluster_wait();
  } else {
    // add the partial tile into part[tile] (fp32 atomics, performed in L2);
    // the last of the tile's ks CTAs to arrive applies the epilogue to the
    // sum and clears part[tile] and the count for the next call
    __shared__ int last_s;
    float* pt = a.part + (size_t)tile * BP * kTM;
    if (tid < kTM && good) {
#pragma unroll
      for (int b = 0; b < BP; ++b) atomicAdd(pt + b * kTM + tid, v[b]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) last_s = atomicAdd(a.sem + tile, 1) == ks - 1;
    __syncthreads();
    if (last_s) {
      __threadfence();
      if (tid < kTM) {
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          const float z = __ldcg(pt + b * kTM + tid);
          pt[b * kTM + tid] = 0.f;
          emit(tid, b, z);
        }
      }
      if (tid == 0) a.sem[tile] = 0;
    }
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int BP>
__global__ void __launch_bounds__(kTcThreads, 1)
    mlp_tc_down_kernel(const __grid_constant__ CUtensorMap mapHi, const __grid_constant__ CUtensorMap mapLo,
                       const __grid_constant__ CUtensorMap mapT, const void* W, DownArgs a) {
  constexpr uint32_t kABytes = kKB * 256, kBBytes = BP * 128;  // A: 64 neurons x 128 columns
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t fullA[kSD], fullB[kSD], empty[kSD], done;
  __shared__ uint32_t tmem_base;
  __shared__ int rows[kKChunk];
  __shared__ int issued, consumed, flag_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int cnt = max(0, min(*a.U_count, a.capU));
  const int c0 = blockIdx.x * kTM;
  const int k0 = blockIdx.y * a.kchunk;
  if (k0 >= cnt) return;
  const int k1 = min(cnt, k0 + a.kchunk);
  const int nk = (k1 - k0 + kKB - 1) / kKB;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sH = smem + kSD * kABytes;
  uint8_t* sL = sH + kSD * kBBytes;

  for (int i = tid; i < nk * kKB; i += blockDim.x) {
    int r = a.U[min(k0 + i, cnt - 1)];
    if (r < 0 || r >= a.N) {
      set_error(a.hdr, DV_ERR_INDEX_RANGE, r);
      r = 0;
    }
    rows[i] = r;
  }
  if (tid == 0) {
    for (int s = 0; s < kSD; ++s) {
      tc::mbar_init(&fullA[s], a.tile_rows ? 1 : kTM);
      tc::mbar_init(&fullB[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&done, 1);
    tc::fence_mbar_init();
    issued = consumed = flag_err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp >= 4) {
    if (warp == 4 && lane == 0) {  // TMA producer: the coefficient halves (and the rows when they form tiles)
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kSD, it = kb / kSD;
        if (kb >= kSD && !tc::mbar_wait(&empty[s], (it - 1) & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 4);
          flag_err = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&fullB[s], 2 * kBBytes);
        tc::tma_load_2d(sH + s * kBBytes, &mapHi, k0 + kb * kKB, 0, &fullB[s]);
        tc::tma_load_2d(sL + s * kBBytes, &mapLo, k0 + kb * kKB, 0, &fullB[s]);
        if (a.tile_rows) {
          const int r0 = rows[kb * kKB];
          tc::mbar_arrive_expect_tx(&fullA[s], kABytes);
          tc::tma_load_2d(sA + s * kABytes, &mapT, c0, r0, &fullA[s]);
          tc::tma_load_2d(sA + s * kABytes + kKB * 128, &mapT, c0 + 64, r0, &fullA[s]);
        }
        issued = kb + 1;
      }
    } else if (warp == 5 && lane == 0) {  // MMA issuer
      constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
      const uint32_t idesc = tc::idesc_f16(kTM, BP, kBf16, /*A MN-major*/ true, false);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kSD, it = kb / kSD;
        if (!tc::mbar_wait(&fullA[s], it & 1, a.wait_ns) || !tc::mbar_wait(&fullB[s], it & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 5);
          flag_err = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t aBase = tc::saddr(sA + s * kABytes);
        const uint32_t hBase = tc::saddr(sH + s * kBBytes), lBase = tc::saddr(sL + s * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kKB / 16; ++kk) {
          // A (MN-major): 16 neuron rows = two 8-row groups (1024 B apart);
          // the two 64-column halves of the tile are kKB*128 bytes apart
          const uint64_t ad = tc::smem_desc(aBase + kk * 2048, kKB * 128, 1024, 2);
          const uint64_t hd = tc::smem_desc(hBase + kk * 32, 16, 1024, 2);
          const uint64_t ld = tc::smem_desc(lBase + kk * 32, 16, 1024, 2);
          tc::mma_f16(tmem, ad, hd, idesc, (kb | kk) != 0);
          tc::mma_f16(tmem, ad, ld, idesc, 1);
        }
        tc::mma_commit(&empty[s]);
        consumed = kb + 1;
      }
      tc::mma_commit(&done);
    }
    __syncwarp();
  } else if (!a.tile_rows) {  // warps 0-3 gather the weight rows: thread = (row r, column half)
    // thread t copies 16-byte chunk t % 8 of the 128-byte segments
    // g = t / 8 + 16 q (q < 8) of the stage: segment g is column half g / 64
    // of neuron row g % 64 (eight lanes per segment: whole lines per warp
    // instruction); the rows change every stage
    const int ch = tid & 7;
    int kb = 0, sig = 0;
    bool okl = true;
    for (; kb < nk; ++kb) {
      const int st = kb % kSD;
      if (kb >= kSD && !tc::mbar_wait(&empty[st], ((kb / kSD) - 1) & 1, a.wait_ns)) {
        okl = false;
        break;
      }
      uint8_t* base = sA + (size_t)st * kABytes;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int g = (tid >> 3) + 16 * q, r = g & (kKB - 1), half = g >> 6;
        const T* src = static_cast<const T*>(W) + (size_t)rows[kb * kKB + r] * a.d + c0 + half * 64 + ch * 8;
        cp_async16(base + half * (kKB * 128) + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4), src);
      }
      cp_async_commit();
      if (kb >= kSD - 2) {
        cp_async_wait<kSD - 2>();
        tc::fence_proxy_async();
        tc::mbar_arrive(&fullA[sig % kSD]);
        ++sig;
      }
    }
    cp_async_wait<0>();
    tc::fence_proxy_async();
    for (; sig < kb; ++sig) tc::mbar_arrive(&fullA[sig % kSD]);
    if (!okl) {
      set_error(a.hdr, DV_ERR_TIMEOUT, 8);
      flag_err = 1;
    }
  }

  bool ok = true;
  float v[BP];
  if (tid < kTM) {
    ok = tc::mbar_wait(&done, 0, unwind_ns);
    if (!ok && lane == 0) set_error(a.hdr, DV_ERR_TIMEOUT, 6);
    __syncwarp();
    tc::fence_after_sync();
#pragma unroll
    for (int c = 0; c < BP; c += 8) tc::tmem_ld8(tmem + ((uint32_t)(warp * 32) << 16) + c, v + c);
    tc::tmem_ld_wait();
  }
  __syncthreads();  // flag_err is final
  if (tid < kTM && ok && !flag_err) {
    const int col = c0 + tid;
#pragma unroll
    for (int b = 0; b < BP; ++b)
      if (b < a.B) atomicAdd(a.out + (size_t)b * a.d + col, v[b]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb) {
      if (!tc::mbar_wait(&fullB[kb % kSD], (kb / kSD) & 1, unwind_ns)) break;
      if (a.tile_rows && !tc::mbar_wait(&fullA[kb % kSD], (kb / kSD) & 1, unwind_ns)) break;
    }
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---- host ------------------------------------------------------------------------

// K split of the up-projection (a small union otherwise leaves most SMs
// idle: 23 tiles of 128 rows streamed 1.8 MB each).  When even the largest
// possible union has at most half as many tiles as SMs, the host fixes the
// split: clusters of S CTAs per tile, S doubling while every CTA keeps an SM
// to itself and a slice of d has 8+ stages.  Otherwise (S = 1) the grid is
// two CTAs per SM, or one per tile of the largest union when that is more,
// and each CTA finds its tile and split from the union's actual size on the
// device (measured on GB300, OPT-30B-shaped batch 32 at 5 %: q/K/V and MLP
// calls 145 -> 137 and 135 -> 126 us; for batch 4 the host-sized clusters
// stayed faster, 63 + 53 against 71 + 59 us).
int up_splits(int tiles, int nk_all) {
  int S = 1;
  while (S < 8 && tiles * S * 2 <= 2 * num_sms_current() && nk_all >= 8 * S) S *= 2;
  return S;
}
int up_grid(int max_tiles, int S) { return S > 1 ? max_tiles * S : max(max_tiles, 2 * num_sms_current()); }

// Union entries per down-projection CTA: about two CTAs per SM over the
// column tiles, 256..1024 entries.
int down_chunk(int col_tiles, int max_rows) {
  const int want = max(1, 2 * num_sms_current() / max(1, col_tiles));
  int ch = (max_rows + want - 1) / want;
  ch = (ch + kKB - 1) / kKB * kKB;
  return max(4 * kKB, min(kKChunk, ch));
}

template <typename T, int BP>
cudaError_t run_tc(const MlpLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = !std::is_same<T, __half>::value;
  const int Upad = tc_act_cols(L.N);
  CUtensorMap mY, mHi, mLo;
  if (!make_map(&mY, L.y, L.d, L.B, BP, bf16) || !make_map(&mHi, L.act_hi, Upad, BP, BP, bf16) ||
      !make_map(&mLo, L.act_lo, Upad, BP, BP, bf16))
    return cudaErrorInvalidValue;
  const size_t smem_up = 1024 + kSU * (kTM * 128 + BP * 128);
  const size_t smem_dn = 1024 + kSD * (kKB * 256 + 2 * BP * 128);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [&] {
    cudaError_t e = cudaFuncSetAttribute(mlp_tc_up_kernel<T, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_up);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mlp_tc_down_kernel<T, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_dn);
    return (int)e;
  });
  if (ea != cudaSuccess) return ea;
  const int maxU = L.N < L.B * L.cap ? L.N : L.B * L.cap;
  UpArgs ua{L.U, L.U_count, L.N, L.member, (L.N + 31) / 32, L.B, L.d, L.N, Upad, L.act_hi, L.act_lo, hdr,
            wait_limit_ns()};
  ua.part = L.tc_part;
  ua.sem = L.tc_sem;
  const int tiles = (maxU + kTM - 1) / kTM;
  ua.S = up_splits(tiles, L.d / kKB);
  if (ua.S == 1 && (!ua.part || !ua.sem)) return cudaErrorInvalidValue;  // the device split needs them
  // neuron rows are gathered by the CTAs' own threads (mapT is not used)
  cudaError_t e = launch_k(mlp_tc_up_kernel<T, BP, kEpiMlp>, dim3(up_grid(tiles, ua.S)), dim3(kTcThreads),
                           smem_up, stream, false, ua.S, mY, mY, L.W1n, ua);
  if (e != cudaSuccess) return e;
  DownArgs da{L.U, L.U_count, L.N, L.B, L.d, L.N, L.out, hdr, wait_limit_ns()};
  da.kchunk = down_chunk(L.d / kTM, maxU);
  dim3 g(L.d / kTM, (maxU + da.kchunk - 1) / da.kchunk);
  mlp_tc_down_kernel<T, BP><<<g, kTcThreads, smem_dn, stream>>>(mHi, mLo, mHi, L.W2n, da);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

template <typename T, int BP>
cudaError_t run_qkv_tc(const TcQkvLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = !std::is_same<T, __half>::value;
  const int nrows = L.h * 3 * L.d_h;
  CUtensorMap mY, mT;
  if (!make_map(&mY, L.y, L.d, L.B, BP, bf16) || !make_map(&mT, L.Wqkv, L.d, nrows, kTM, bf16))
    return cudaErrorInvalidValue;
  const size_t smem_up = 1024 + kSU * (kTM * 128 + BP * 128);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [&] {
    return (int)cudaFuncSetAttribute(mlp_tc_up_kernel<T, BP, kEpiQkv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_up);
  });
  if (ea != cudaSuccess) return ea;
  UpArgs ua{};
  ua.U = L.rows; ua.U_count = L.rows_count; ua.capU = nrows; ua.member = L.member; ua.words = L.words;
  ua.B = L.B; ua.d = L.d; ua.N = nrows; ua.hdr = hdr; ua.wait_ns = wait_limit_ns();
  ua.h = L.h; ua.d_h = L.d_h; ua.n_max = L.n_max; ua.capQ = L.capQ; ua.slot_of = L.slot_of; ua.pos = L.pos;
  ua.q = L.q; ua.K = L.K; ua.V = L.V;
  // a head's 3 d_h rows are contiguous: with d_h = 128 every 128-row tile is
  // one head's Q, K or V block
  ua.tile_rows = (3 * L.d_h) % kTM == 0 ? 1 : 0;
  ua.part = L.part;
  ua.sem = L.sem;
  const int tiles = (L.max_rows + kTM - 1) / kTM;
  ua.S = up_splits(tiles, L.d / kKB);
  if (ua.S == 1 && (!ua.part || !ua.sem)) return cudaErrorInvalidValue;  // the device split needs them
  return launch_k(mlp_tc_up_kernel<T, BP, kEpiQkv>, dim3(up_grid(tiles, ua.S)), dim3(kTcThreads), smem_up,
                  stream, false, ua.S, mY, mT, L.Wqkv, ua);
}

template <typename T, int BP>
cudaError_t run_rows_tc(const TcRowsLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = !std::is_same<T, __half>::value;
  CUtensorMap mHi, mLo, mT;
  if (!make_map(&mHi, L.act_hi, L.Upad, BP, BP, bf16) || !make_map(&mLo, L.act_lo, L.Upad, BP, BP, bf16) ||
      !make_map(&mT, L.W, L.d, L.n_rows, kKB, bf16))
    return cudaErrorInvalidValue;
  const size_t smem_dn = 1024 + kSD * (kKB * 256 + 2 * BP * 128);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [&] {
    return (int)cudaFuncSetAttribute(mlp_tc_down_kernel<T, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_dn);
  });
  if (ea != cudaSuccess) return ea;
  DownArgs da{L.rows, L.rows_count, L.n_rows, L.B, L.d, L.n_rows, L.out, hdr, wait_limit_ns(),
              L.rows_per_unit % kKB == 0 ? 1 : 0};
  da.kchunk = down_chunk(L.d / kTM, L.max_rows);
  dim3 g(L.d / kTM, (L.max_rows + da.kchunk - 1) / da.kchunk);
  mlp_tc_down_kernel<T, BP><<<g, kTcThreads, smem_dn, stream>>>(mHi, mLo, mT, L.W, da);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace

cudaError_t launch_qkv_tc(const TcQkvLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return L.B <= 16 ? run_qkv_tc<__half, 16>(L, hdr, stream) : run_qkv_tc<__half, 32>(L, hdr, stream);
  if (dt == DV_BF16)
    return L.B <= 16 ? run_qkv_tc<__nv_bfloat16, 16>(L, hdr, stream) : run_qkv_tc<__nv_bfloat16, 32>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rows_tc(const TcRowsLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return L.B <= 16 ? run_rows_tc<__half, 16>(L, hdr, stream) : run_rows_tc<__half, 32>(L, hdr, stream);
  if (dt == DV_BF16)
    return L.B <= 16 ? run_rows_tc<__nv_bfloat16, 16>(L, hdr, stream) : run_rows_tc<__nv_bfloat16, 32>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

bool tc_mlp_supported(int B, int d, dv_dtype dt) {
  return dt != DV_F32 && B >= kTcMinBatch && B <= 32 && d % kTM == 0;
}

int tc_act_cols(int N) { return (N + kTM - 1) / kTM * kTM; }

size_t tc_part_floats(int max_rows) { return (size_t)((max_rows + kTM - 1) / kTM) * 32 * kTM; }

cudaError_t launch_sparse_mlp_tc(const MlpLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return L.B <= 16 ? run_tc<__half, 16>(L, hdr, stream) : run_tc<__half, 32>(L, hdr, stream);
  if (dt == DV_BF16)
    return L.B <= 16 ? run_tc<__nv_bfloat16, 16>(L, hdr, stream) : run_tc<__nv_bfloat16, 32>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dv

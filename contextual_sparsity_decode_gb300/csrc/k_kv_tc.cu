// KV cache fill on the tcgen05 tensor cores: the dense prompt (prefill) and
// any bulk repair of skipped heads.
//
// Deja Vu reading notes, "Typical LLM procedure": the prompt phase builds
// every layer's KV cache; "Sparsity operator for Attention": a head skipped
// at earlier steps has its K/V recomputed from the stored token embeddings
// X when it is selected.  Both are the same product over the positions
// whose K/V are missing,
//     [K_i[j] ; V_i[j]] = X[j] [W_i^K ; W_i^V]^T      for every missing j,
// which for a prompt of n positions is a dense (n x d) . (d x 2 d_h) GEMM
// per head: a real contraction, so it runs on the tensor cores.
//
// One CTA per (row b, selected head i, tile of 128 missing positions):
//   A = the 128 positions' rows of X, gathered by TMA (tile::gather4, 128-byte
//       swizzle, K-major), 64 elements of d per stage;
//   B = head i's W^K and W^V rows, adjacent in Wqkv ([i][K][..] then
//       [i][V][..]), one 2 d_h-row TMA tile per stage;
//   D = 128 x 2 d_h fp32 accumulators in tensor memory.
// The epilogue reads a position's row of D (one thread per position), rounds
// it to the storage type and writes K[b][i][j] and V[b][i][j] (2 d_h
// contiguous elements each).  A separate small kernel then marks the
// selected heads' positions valid (marking inside this kernel would race
// with sibling CTAs still ranking the missing positions).
//
// One elected thread issues the TMA loads into a 4-stage ring, one issues
// the MMAs; every wait is bounded (dv_set_wait_limit_ns) and reports
// DV_ERR_TIMEOUT; the waits that unwind a CTA take at least two seconds, so
// no CTA frees its tensor memory or exits with its own copies or MMAs still
// in flight.

#include <cuda.h>

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kTP = 128;                  // positions per CTA (MMA M)
constexpr int kKB = 64;                   // d elements per stage (one 128-byte row)
constexpr int kStages = 4;
constexpr int kThreads = 128;
constexpr long long kUnwindNs = 2000000000LL;

struct KvTcArgs {
  const int32_t* pos;
  const int32_t* head_idx;
  const int32_t* head_count;
  int cap, B, d, h, d_h, n_max;
  const uint8_t* valid;
  void* K;
  void* V;
  WsHeader* hdr;
  long long wait_ns;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 8 floats -> one 16-byte vector of the storage type.
template <typename T>
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const T lo = Elem<T>::from_f(f[2 * q]), hi = Elem<T>::from_f(f[2 * q + 1]);
    w[q] = (uint32_t)(*reinterpret_cast<const uint16_t*>(&lo)) |
           ((uint32_t)(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T, int DH>
__global__ void __launch_bounds__(kThreads, 1)
    kv_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW, KvTcArgs a) {
  constexpr int NB = 2 * DH;                          // MMA N: K and V rows of the head
  constexpr uint32_t kABytes = kTP * 128, kBBytes = NB * 128;
  constexpr uint32_t kTmemCols = NB;                  // 128 or 256 fp32 columns
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int pos_s[kTP];
  __shared__ int tmp[32];
  __shared__ int issued, consumed, flag_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pt = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int cnt = max(0, min(a.head_count[b], a.cap));
  if (s >= cnt) return;
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int p0 = a.pos[b];
  const int p = (p0 >= 0 && p0 < a.n_max) ? p0 : -1;
  if (i < 0 || i >= a.h || p < 0) {
    if (tid == 0 && pt == 0) set_error(a.hdr, p < 0 ? DV_ERR_POSITION : DV_ERR_INDEX_RANGE, p < 0 ? p0 : i);
    return;
  }

  // ranks [pt*128, pt*128 + 128) of the ascending list of positions j < p
  // whose K/V are missing (valid == 0); each thread scans 16 flags a round
  const uint8_t* vr = a.valid + ((size_t)b * a.h + i) * a.n_max;
  int seen = 0;
  for (int base = 0; base < p; base += kThreads * 16) {
    const int j0 = base + tid * 16;
    uint32_t w4[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    if (j0 < p) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(vr + j0);
      w4[0] = v4.x; w4[1] = v4.y; w4[2] = v4.z; w4[3] = v4.w;
    }
    int mine = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) mine += (j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
    int total;
    const int incl = block_inclusive_scan<kThreads>(mine, tmp, &total);
    int rank = seen + incl - mine;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if ((j0 + k < p) && (((w4[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0)) {
        const int slot = rank - pt * kTP;
        if (slot >= 0 && slot < kTP) pos_s[slot] = j0 + k;
        ++rank;
      }
    }
    seen += total;
  }
  const int np = min(kTP, seen - pt * kTP);
  __syncthreads();
  if (np <= 0) return;  // whole CTA, before any barrier init or tensor memory

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  if (tid == 0) {
    for (int q = 0; q < kStages; ++q) {
      tc::mbar_init(&full[q], 1);
      tc::mbar_init(&empty[q], 1);
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
  const int nk = (a.d + kKB - 1) / kKB;
  const int xrow0 = b * a.n_max;                 // X viewed as [B * n_max][d]
  const int wrow = (i * 3 + 1) * DH;             // first W^K row of head i in [h * 3 * d_h][d]

  if (warp == 0 && lane == 0) {  // TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kStages, it = kb / kStages;
      if (kb >= kStages && !tc::mbar_wait(&empty[st], (it - 1) & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 11);
        flag_err = 1;
        break;
      }
      tc::mbar_arrive_expect_tx(&full[st], kABytes + kBBytes);
      uint8_t* dA = sA + st * kABytes;
#pragma unroll 4
      for (int g = 0; g < kTP / 4; ++g) {
        int r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = xrow0 + pos_s[min(4 * g + q, np - 1)];
        tc::tma_gather4(dA + g * 512, &mapX, kb * kKB, r[0], r[1], r[2], r[3], &full[st]);
      }
      tc::tma_load_2d(sB + st * kBBytes, &mapW, kb * kKB, wrow, &full[st]);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc = tc::idesc_f16(kTP, NB, kBf16, false, false);
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kStages, it = kb / kStages;
      if (!tc::mbar_wait(&full[st], it & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 12);
        flag_err = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t aBase = tc::saddr(sA + st * kABytes), bBase = tc::saddr(sB + st * kBBytes);
#pragma unroll
      for (int kk = 0; kk < kKB / 16; ++kk) {
        const uint64_t ad = tc::smem_desc(aBase + kk * 32, 16, 1024, 2);
        const uint64_t bd = tc::smem_desc(bBase + kk * 32, 16, 1024, 2);
        tc::mma_f16(tmem, ad, bd, idesc, (kb | kk) != 0);
      }
      tc::mma_commit(&empty[st]);
      consumed = kb + 1;
    }
    tc::mma_commit(&done);  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // epilogue: thread = accumulator row = the tid-th missing position
  const bool ok = tc::mbar_wait(&done, 0, unwind_ns);
  if (!ok && lane == 0) set_error(a.hdr, DV_ERR_TIMEOUT, 13);
  __syncwarp();
  tc::fence_after_sync();
  __syncthreads();  // flag_err is final: both issuers are past their loops
  const bool live = ok && !flag_err && tid < np;
  const size_t row_off = (((size_t)b * a.h + i) * a.n_max + (live ? pos_s[tid] : 0)) * DH;
  T* Kd = static_cast<T*>(a.K) + row_off;
  T* Vd = static_cast<T*>(a.V) + row_off;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
  for (int c0 = 0; c0 < NB; c0 += 32) {
    float v[32];
#pragma unroll
    for (int c = 0; c < 32; c += 8) tc::tmem_ld8(lane_base + c0 + c, v + c);
    tc::tmem_ld_wait();
    if (live) {
      T* dst = c0 < DH ? Kd + c0 : Vd + (c0 - DH);
#pragma unroll
      for (int c = 0; c < 32; c += 8) *reinterpret_cast<uint4*>(dst + c) = pack8<T>(v + c);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // no TMA write into this CTA's shared memory may still be in flight
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb)
      if (!tc::mbar_wait(&full[kb % kStages], (kb / kStages) & 1, unwind_ns)) break;
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

__global__ void kv_mark_valid_kernel(KvTcArgs a) {
  const int s = blockIdx.x, b = blockIdx.y;
  const int cnt = max(0, min(a.head_count[b], a.cap));
  if (s >= cnt) return;
  const int i = a.head_idx[(size_t)b * a.cap + s];
  const int p = a.pos[b];
  if (i < 0 || i >= a.h || p < 0 || p >= a.n_max) return;
  uint8_t* vr = const_cast<uint8_t*>(a.valid) + ((size_t)b * a.h + i) * a.n_max;
  for (int j = threadIdx.x; j < p; j += blockDim.x) vr[j] = 1;
}

// ---- host ------------------------------------------------------------------------

template <typename T, int DH>
cudaError_t run_kv_tc(const AttnLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap mX, mW;
  if (!make_map(&mX, L.X, L.d, (uint64_t)L.B * L.n_max, 1, bf16) ||
      !make_map(&mW, L.Wqkv, L.d, (uint64_t)L.h * 3 * DH, 2 * DH, bf16))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kStages * (kTP * 128 + 2 * DH * 128);
  static PerDevice attr;  // function attributes are per device
  const cudaError_t ea = (cudaError_t)attr.get(current_device(), [smem] {
    return (int)cudaFuncSetAttribute(kv_tc_kernel<T, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (ea != cudaSuccess) return ea;
  KvTcArgs a{L.pos, L.head_idx, L.head_count, L.cap, L.B, L.d, L.h, L.d_h, L.n_max, L.valid, L.K, L.V, hdr,
             wait_limit_ns()};
  dim3 g((L.n_max + kTP - 1) / kTP, L.cap, L.B);
  kv_tc_kernel<T, DH><<<g, kThreads, smem, stream>>>(mX, mW, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_mark_valid_kernel<<<dim3(L.cap, L.B), 256, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(2);
  return e;
}

}  // namespace

bool kv_tc_supported(int d, int d_h, dv_dtype dt) {
  // 16-bit storage; a row of X and of Wqkv is a whole number of 16-byte
  // chunks (TMA strides); the missing positions are ranked 2048 at a time
  return (dt == DV_F16 || dt == DV_BF16) && (d_h == 64 || d_h == 128) && d % 8 == 0;
}

cudaError_t launch_kv_repair_tc(const AttnLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return L.d_h == 128 ? run_kv_tc<__half, 128>(L, hdr, stream) : run_kv_tc<__half, 64>(L, hdr, stream);
  if (dt == DV_BF16)
    return L.d_h == 128 ? run_kv_tc<__nv_bfloat16, 128>(L, hdr, stream)
                        : run_kv_tc<__nv_bfloat16, 64>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dv

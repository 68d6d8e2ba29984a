// The sparsity predictor for batches of 2..32 rows on the tcgen05 tensor cores
// ("用Deja Vu来提高 LLM 的推理速度" §2: a two-layer MLP with a sigmoid per head /
// neuron).  With B rows both products are dense contractions over the
// predictor's weights, whose rows are contiguous:
//   first   h[b][j] = ReLU(y_b . P1t[j]),   M = 128 rows of P1t, N = B padded
//           to 16 / 32, K = d; the epilogue writes h split into two
//           storage-type halves hi + lo (h = hi + lo to ~2^-16 relative);
//   second  s[b][u] = sigmoid(h_b . P2t[u]), M = 128 rows of P2t, K = r,
//           two MMAs per step (hi and lo), fp32 scores [B][N] for the
//           selection kernel.
// Both predictors run in one launch per product (their CTAs side by side).
// The first product has only r / 128 tiles per predictor (8 for r = 1024), so
// each tile is split along d over a cluster of S <= 8 CTAs: every CTA
// accumulates its slice of d in TMEM and pushes each partial row into the
// shared memory of the CTA that owns the row (128 / S rows each, distributed
// shared memory); after one cluster barrier every CTA sums its own rows over
// the S partials before ReLU and the split.
// On CUDA cores a batch of 32 read each predictor's weights once per 8-row
// tile (4x) and was bound by fp32 FMA throughput.
//
// One thread issues TMA tile loads (both operands) into a 4-stage ring, one
// issues the MMAs; the waits are bounded (dv_set_wait_limit_ns) and report
// DV_ERR_TIMEOUT; a CTA waits (at least two seconds) for its own copies and
// MMAs before it frees its tensor memory.

#include <cuda.h>

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kPM = 128;   // MMA M: weight rows per CTA
constexpr int kPKB = 64;   // K elements per stage
constexpr int kPSt = 4;
constexpr long long kUnwindNs = 2000000000LL;

struct PredTcArgs {
  int rows[2];       // r (first product) or N (second), per predictor
  int tiles0;        // row tiles of predictor 0
  int S;             // CTAs (a cluster) per tile, splitting K; 1 for the second product
  int K[2];          // d (first) or r (second)
  int B;
  // first product: h halves [BP][ld] of each predictor
  void* hi[2];
  void* lo[2];
  int ld[2];
  // second product: scores [B][N]
  float* s[2];
  WsHeader* hdr;
  long long wait_ns;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <typename T, int BP, bool kSecond>
__global__ void __launch_bounds__(128, 1)
    pred_tc_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
                   const __grid_constant__ CUtensorMap mapB0, const __grid_constant__ CUtensorMap mapB1,
                   const __grid_constant__ CUtensorMap mapL0, const __grid_constant__ CUtensorMap mapL1,
                   PredTcArgs a) {
  constexpr int kNB = kSecond ? 2 : 1;  // B operands per stage (hi, lo)
  constexpr uint32_t kABytes = kPM * 128, kBBytes = BP * 128;
  constexpr uint32_t kTmemCols = 32;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kPSt], empty[kPSt], done;
  __shared__ uint32_t tmem_base;
  __shared__ int issued, consumed, flag_err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int tile = (int)blockIdx.x / a.S, split = (int)blockIdx.x % a.S;
  const int p = tile >= a.tiles0 ? 1 : 0;
  const int m0 = (tile - (p ? a.tiles0 : 0)) * kPM;
  const int rows = p ? a.rows[1] : a.rows[0];
  const int K = p ? a.K[1] : a.K[0];
  const CUtensorMap* mA = p ? &mapA1 : &mapA0;
  const CUtensorMap* mB = p ? &mapB1 : &mapB0;
  const CUtensorMap* mL = p ? &mapL1 : &mapL0;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPSt * kABytes;  // [stage][kNB] tiles of BP rows
  float* red = reinterpret_cast<float*>(sB + kPSt * kNB * kBBytes);  // [S][128 / S][BP + 1] pushed partials (S > 1)
  if (tid == 0) {
    for (int q = 0; q < kPSt; ++q) {
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
  const int nk_all = (K + kPKB - 1) / kPKB;
  const int kb0 = split * nk_all / a.S;  // this CTA's K blocks [kb0, kb0 + nk)
  const int nk = (split + 1) * nk_all / a.S - kb0;

  if (warp == 0 && lane == 0) {  // TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kPSt, it = kb / kPSt, kx = (kb0 + kb) * kPKB;
      if (kb >= kPSt && !tc::mbar_wait(&empty[st], (it - 1) & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 31);
        flag_err = 1;
        break;
      }
      tc::mbar_arrive_expect_tx(&full[st], kABytes + kNB * kBBytes);
      tc::tma_load_2d(sA + st * kABytes, mA, kx, m0, &full[st]);
      tc::tma_load_2d(sB + (st * kNB) * kBBytes, mB, kx, 0, &full[st]);
      if (kSecond) tc::tma_load_2d(sB + (st * kNB + 1) * kBBytes, mL, kx, 0, &full[st]);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc = tc::idesc_f16(kPM, BP, kBf16, false, false);
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kPSt, it = kb / kPSt;
      if (!tc::mbar_wait(&full[st], it & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 32);
        flag_err = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t aBase = tc::saddr(sA + st * kABytes);
#pragma unroll
      for (int kk = 0; kk < kPKB / 16; ++kk) {
        const uint64_t ad = tc::smem_desc(aBase + kk * 32, 16, 1024, 2);
#pragma unroll
        for (int nb = 0; nb < kNB; ++nb) {
          const uint64_t bd = tc::smem_desc(tc::saddr(sB + (st * kNB + nb) * kBBytes) + kk * 32, 16, 1024, 2);
          tc::mma_f16(tmem, ad, bd, idesc, (kb | kk | nb) != 0);
        }
      }
      tc::mma_commit(&empty[st]);
      consumed = kb + 1;
    }
    tc::mma_commit(&done);
  }
  __syncwarp();

  const bool ok = tc::mbar_wait(&done, 0, unwind_ns);
  if (!ok && lane == 0) set_error(a.hdr, DV_ERR_TIMEOUT, 33);
  __syncwarp();
  tc::fence_after_sync();
  float v[BP];
#pragma unroll
  for (int c = 0; c < BP; c += 8) tc::tmem_ld8(tmem + ((uint32_t)(warp * 32) << 16) + c, v + c);
  tc::tmem_ld_wait();
  __syncthreads();  // flag_err is final
  const bool good = ok && !flag_err;
  if (!kSecond) {
    T* hi = static_cast<T*>(p ? a.hi[1] : a.hi[0]);
    T* lo = static_cast<T*>(p ? a.lo[1] : a.lo[0]);
    const int ld = p ? a.ld[1] : a.ld[0];
    if (a.S == 1) {
      if (good && m0 + tid < rows) {
#pragma unroll
        for (int b = 0; b < BP; ++b) {  // padding rows of y read zeros: h = 0 there
          const float x = fmaxf(v[b], 0.f);
          const T h = Elem<T>::from_f(x);
          hi[(size_t)b * ld + m0 + tid] = h;
          lo[(size_t)b * ld + m0 + tid] = Elem<T>::from_f(x - Elem<T>::to_f(h));
        }
      }
    } else {
      // push the partial rows (zeros from a CTA without K blocks) into the
      // CTA that owns them (slot `split` of its [S][span] rows), one cluster
      // barrier, then sum the owned rows from local shared memory
      const int span = kPM / a.S;
      {
        const int owner = tid / span, lr = tid - owner * span;
        float* dst = red + ((size_t)split * span + lr) * (BP + 1);
#pragma unroll
        for (int b = 0; b < BP; ++b) st_dsmem_f32(dst + b, (uint32_t)owner, (good && nk > 0) ? v[b] : 0.f);
      }
      cluster_arrive();
      cluster_wait();
      const int r0 = split * span;
      for (int e = tid; e < span * BP; e += 128) {
        const int b = e / span, lr = e - b * span, rr = r0 + lr;  // consecutive threads: consecutive rows
        float x = 0.f;
        for (int q = 0; q < a.S; ++q) x += red[((size_t)q * span + lr) * (BP + 1) + b];
        if (good && m0 + rr < rows) {
          x = fmaxf(x, 0.f);
          const T h = Elem<T>::from_f(x);
          hi[(size_t)b * ld + m0 + rr] = h;
          lo[(size_t)b * ld + m0 + rr] = Elem<T>::from_f(x - Elem<T>::to_f(h));
        }
      }
    }
  } else if (good && m0 + tid < rows) {
    float* s = p ? a.s[1] : a.s[0];
#pragma unroll
    for (int b = 0; b < BP; ++b)
      if (b < a.B) s[(size_t)b * rows + m0 + tid] = 1.f / (1.f + expf(-v[b]));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb)
      if (!tc::mbar_wait(&full[kb % kPSt], (kb / kPSt) & 1, unwind_ns)) break;
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---- host ------------------------------------------------------------------------

template <typename T, int BP, bool kSecond>
cudaError_t pred_attr(size_t smem) {
  static PerDevice attr;  // function attributes are per device
  return (cudaError_t)attr.get(current_device(), [smem] {
    return (int)cudaFuncSetAttribute(pred_tc_kernel<T, BP, kSecond>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
  });
}

template <typename T, int BP>
cudaError_t pred_tc_t(const void* y, int B, int d, const PredLaunch& P, int n_preds, WsHeader* hdr,
                      cudaStream_t stream) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap mA[2], mB[2], mL[2];
  PredTcArgs a{};
  a.B = B; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  // first product: A = P1t [r][d], B = y [B][d] (rows beyond B read zeros)
  for (int i = 0; i < 2; ++i) {
    const int q = i < n_preds ? i : 0;
    if (!make_map(&mA[i], P.P1t[q], d, P.r[q], kPM, bf16) || !make_map(&mB[i], y, d, B, BP, bf16))
      return cudaErrorInvalidValue;
    mL[i] = mB[i];
    a.rows[i] = P.r[q]; a.K[i] = d; a.hi[i] = P.h_hi[q]; a.lo[i] = P.h_lo[q]; a.ld[i] = P.r[q];
  }
  a.tiles0 = (P.r[0] + kPM - 1) / kPM;
  const int tiles = a.tiles0 + (n_preds > 1 ? (P.r[1] + kPM - 1) / kPM : 0);
  const int nk = (d + kPKB - 1) / kPKB;
  a.S = 1;  // split d while the grid is below the SM count and each split keeps 2+ K blocks
  while (a.S < 8 && tiles * a.S < num_sms_current() && nk >= 4 * a.S) a.S *= 2;
  const size_t smem1 = 1024 + kPSt * (kPM * 128 + BP * 128) + (size_t)kPM * (BP + 1) * 4;
  cudaError_t e = pred_attr<T, BP, false>(smem1);
  if (e != cudaSuccess) return e;
  e = launch_k(pred_tc_kernel<T, BP, false>, dim3(tiles * a.S), dim3(128), smem1, stream, false, a.S, mA[0],
               mA[1], mB[0], mB[1], mL[0], mL[1], a);
  if (e != cudaSuccess) return e;
  // second product: A = P2t [N][r], B = h halves [BP][r]
  for (int i = 0; i < 2; ++i) {
    const int q = i < n_preds ? i : 0;
    if (!make_map(&mA[i], P.P2t[q], P.r[q], P.N[q], kPM, bf16) ||
        !make_map(&mB[i], P.h_hi[q], P.r[q], BP, BP, bf16) || !make_map(&mL[i], P.h_lo[q], P.r[q], BP, BP, bf16))
      return cudaErrorInvalidValue;
    a.rows[i] = P.N[q]; a.K[i] = P.r[q]; a.s[i] = P.s[q];
  }
  a.tiles0 = (P.N[0] + kPM - 1) / kPM;
  a.S = 1;
  const int grid = a.tiles0 + (n_preds > 1 ? (P.N[1] + kPM - 1) / kPM : 0);
  const size_t smem2 = 1024 + kPSt * (kPM * 128 + 2 * BP * 128);
  e = pred_attr<T, BP, true>(smem2);
  if (e != cudaSuccess) return e;
  return launch_k(pred_tc_kernel<T, BP, true>, dim3(grid), dim3(128), smem2, stream, false, 1, mA[0], mA[1],
                  mB[0], mB[1], mL[0], mL[1], a);
}

}  // namespace

bool predict_tc_supported(int B, int d, dv_dtype dt, const PredLaunch& P, int n_preds) {
  if (dt == DV_F32 || B < kTcMinBatch || B > 32 || d % 8) return false;
  for (int i = 0; i < n_preds; ++i)
    if (P.r[i] % 8 || !P.h_hi[i] || !P.h_lo[i]) return false;
  return true;
}

cudaError_t launch_predict_tc(const void* y, int B, int d, dv_dtype dt, const PredLaunch& P, int n_preds,
                              WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return B <= 16 ? pred_tc_t<__half, 16>(y, B, d, P, n_preds, hdr, stream)
                                   : pred_tc_t<__half, 32>(y, B, d, P, n_preds, hdr, stream);
  if (dt == DV_BF16) return B <= 16 ? pred_tc_t<__nv_bfloat16, 16>(y, B, d, P, n_preds, hdr, stream)
                                    : pred_tc_t<__nv_bfloat16, 32>(y, B, d, P, n_preds, hdr, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dv

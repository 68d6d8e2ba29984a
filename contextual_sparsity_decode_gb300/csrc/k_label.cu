// True-sparsity labels of one layer over a sequence X [T][d] ("用Deja Vu来提高
// LLM 的推理速度" §1 Contextual Sparsity: run the sequence through the layer and
// keep the attention heads and MLP neurons whose outputs have the largest L2
// norm; §2: a threshold on that norm labels the units for the predictor).
//
//   neurons  n_j = || ReLU(X W^1[:, j]) ||_2 over the T tokens.  A dense
//            (N x d) . (d x T) product on the tcgen05 tensor cores: a CTA
//            takes 128 neurons (A = W1n rows, TMA tile) and 256 tokens
//            (B = X rows, TMA tile); each thread owns one neuron's TMEM lane
//            and sums ReLU(v)^2 over its 256 token columns, so no value
//            crosses threads; per-tile sums are added in tile order.
//   heads    m_i = || H_i ||_F with H_i [T][d_h] the head's causal attention
//            output before W_i^O.  First Q, K, V of every head for every
//            token (a second tcgen05 product: A = X rows, B = 256 rows of
//            Wqkv, K/V rounded to the storage type as a KV cache holds them,
//            Q kept in fp32), then one warp per four queries runs the
//            online softmax over keys 0..t staged through shared memory and
//            adds ||h_t||^2; per-block sums are added in block order.
// Selection (top-k or threshold on the norms) is dv_select.
//
// The tensor-core kernel follows the other tcgen05 kernels here: one thread
// issues TMA loads into a 4-stage ring, one issues the MMAs, the waits are
// bounded (dv_set_wait_limit_ns) and report DV_ERR_TIMEOUT, and a CTA waits
// (at least two seconds) for its own copies and MMAs before it frees its
// tensor memory.

#include <cuda.h>

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kLM = 128;     // MMA M
constexpr int kLN = 256;     // MMA N
constexpr int kLKB = 64;     // K elements per stage
constexpr int kLSt = 4;
constexpr long long kUnwindNs = 2000000000LL;

enum LabelMode { kNeuron = 0, kQkv = 1 };

struct LabelArgs {
  int rowsA, rowsB, d;       // rows of the A and B operands, K extent
  // kNeuron: partial[blockIdx.y][neuron]
  float* partial;
  int N;
  // kQkv: Q [h][T][d_h] fp32, K / V [h][T][d_h] storage type
  float* Q;
  void* K;
  void* V;
  int T, h, d_h;
  WsHeader* hdr;
  long long wait_ns;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

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

// D[128 x 256] = A[m0 : m0+128][:] . B[n0 : n0+256][:]^T, both K-major.
template <typename T, int MODE>
__global__ void __launch_bounds__(128, 1)
    label_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                      LabelArgs a) {
  constexpr uint32_t kABytes = kLM * 128, kBBytes = kLN * 128;
  constexpr uint32_t kTmemCols = kLN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kLSt], empty[kLSt], done;
  __shared__ uint32_t tmem_base;
  __shared__ int issued, consumed, flag_err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * kLM, n0 = blockIdx.y * kLN;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kLSt * kABytes;
  if (tid == 0) {
    for (int q = 0; q < kLSt; ++q) {
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
  const int nk = (a.d + kLKB - 1) / kLKB;

  if (warp == 0 && lane == 0) {  // TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kLSt, it = kb / kLSt;
      if (kb >= kLSt && !tc::mbar_wait(&empty[st], (it - 1) & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 21);
        flag_err = 1;
        break;
      }
      tc::mbar_arrive_expect_tx(&full[st], kABytes + kBBytes);
      tc::tma_load_2d(sA + st * kABytes, &mapA, kb * kLKB, m0, &full[st]);
      tc::tma_load_2d(sB + st * kBBytes, &mapB, kb * kLKB, n0, &full[st]);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc = tc::idesc_f16(kLM, kLN, kBf16, false, false);
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kLSt, it = kb / kLSt;
      if (!tc::mbar_wait(&full[st], it & 1, a.wait_ns)) {
        set_error(a.hdr, DV_ERR_TIMEOUT, 22);
        flag_err = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t aBase = tc::saddr(sA + st * kABytes), bBase = tc::saddr(sB + st * kBBytes);
#pragma unroll
      for (int kk = 0; kk < kLKB / 16; ++kk) {
        const uint64_t ad = tc::smem_desc(aBase + kk * 32, 16, 1024, 2);
        const uint64_t bd = tc::smem_desc(bBase + kk * 32, 16, 1024, 2);
        tc::mma_f16(tmem, ad, bd, idesc, (kb | kk) != 0);
      }
      tc::mma_commit(&empty[st]);
      consumed = kb + 1;
    }
    tc::mma_commit(&done);
  }
  __syncwarp();

  const bool ok = tc::mbar_wait(&done, 0, unwind_ns);
  if (!ok && lane == 0) set_error(a.hdr, DV_ERR_TIMEOUT, 23);
  __syncwarp();
  tc::fence_after_sync();
  __syncthreads();  // flag_err is final
  const bool good = ok && !flag_err;
  const int row = m0 + tid;  // this thread's accumulator row (TMEM lane)
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  float sq = 0.f;
  // kQkv: token `row`; column n0 + c of Wqkv's row space is (head, Q/K/V, element)
  const int dh3 = 3 * a.d_h;
#pragma unroll 1
  for (int c0 = 0; c0 < kLN; c0 += 32) {
    float v[32];
#pragma unroll
    for (int c = 0; c < 32; c += 8) tc::tmem_ld8(lane_base + c0 + c, v + c);
    tc::tmem_ld_wait();
    if (MODE == kNeuron) {
      // columns past the last token read zero rows (ReLU(0) = 0)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float r = fmaxf(v[c], 0.f);
        sq = fmaf(r, r, sq);
      }
    } else if (good && row < a.T) {
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        const int R = n0 + c0 + c;  // 8 columns in one (head, matrix) block: d_h % 8 == 0
        if (R >= a.h * dh3) break;
        const int i = R / dh3, rem = R - i * dh3, m = rem / a.d_h, e = rem - m * a.d_h;
        const size_t off = ((size_t)i * a.T + row) * a.d_h + e;
        if (m == 0) {
          float4* q = reinterpret_cast<float4*>(a.Q + off);
          q[0] = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
          q[1] = make_float4(v[c + 4], v[c + 5], v[c + 6], v[c + 7]);
        } else {
          T* dst = static_cast<T*>(m == 1 ? a.K : a.V) + off;
          *reinterpret_cast<uint4*>(dst) = pack8<T>(v + c);
        }
      }
    }
  }
  if (MODE == kNeuron && good && row < a.N) a.partial[(size_t)blockIdx.y * a.N + row] = sq;
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    for (int kb = consumed; kb < issued; ++kb)
      if (!tc::mbar_wait(&full[kb % kLSt], (kb / kLSt) & 1, unwind_ns)) break;
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// causal attention of every head over the sequence, summing ||h_t||^2

constexpr int kHQ = 32;      // queries per CTA (8 warps x 4)
constexpr int kHKT = 64;     // keys per shared-memory tile

template <typename T, int DH>
__global__ void __launch_bounds__(256) head_norm_kernel(const float* Q, const T* K, const T* V, int T_len,
                                                        float scale, float* partial) {
  constexpr int E = DH / 32;  // elements per lane
  __shared__ __align__(16) T Ks[kHKT][DH];
  __shared__ __align__(16) T Vs[kHKT][DH];
  __shared__ float red[8];
  const int i = blockIdx.x, blk = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tq0 = blk * kHQ + wid * 4;  // this warp's first query
  const size_t hoff = (size_t)i * T_len * DH;
  float q[4][E], acc[4][E], mx[4], l[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int t = tq0 + s;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      q[s][e] = t < T_len ? Q[hoff + (size_t)t * DH + lane * E + e] * scale : 0.f;
      acc[s][e] = 0.f;
    }
    mx[s] = -INFINITY;
    l[s] = 0.f;
  }
  const int kend = min(T_len, blk * kHQ + kHQ);  // keys needed by the CTA's last query
  for (int j0 = 0; j0 < kend; j0 += kHKT) {
    const int nj = min(kHKT, kend - j0);
    __syncthreads();  // the previous tile is no longer read
    constexpr int kChunks = DH * (int)sizeof(T) / 16;  // 16-byte chunks per row
    for (int e = tid; e < nj * kChunks; e += 256) {
      const int r = e / kChunks, c = e % kChunks;
      reinterpret_cast<uint4*>(&Ks[r][0])[c] = ld_cached(K + hoff + (size_t)(j0 + r) * DH + c * (16 / sizeof(T)));
      reinterpret_cast<uint4*>(&Vs[r][0])[c] = ld_cached(V + hoff + (size_t)(j0 + r) * DH + c * (16 / sizeof(T)));
    }
    __syncthreads();
    const int jmax = min(nj, tq0 + 4 - j0);  // keys of this tile any of the warp's queries sees
    for (int jj = 0; jj < jmax; ++jj) {
      const int j = j0 + jj;
      float kf[E], vf[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kf[e] = Elem<T>::to_f(Ks[jj][lane * E + e]);
        vf[e] = Elem<T>::to_f(Vs[jj][lane * E + e]);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(q[s][e], kf[e], dot);
        dot = warp_sum(dot);
        if (j <= tq0 + s && tq0 + s < T_len) {  // causal: query t sees keys 0..t
          const float mn = fmaxf(mx[s], dot);
          const float corr = expf(mx[s] - mn);
          const float p = expf(dot - mn);
          l[s] = l[s] * corr + p;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[s][e] = fmaf(p, vf[e], acc[s][e] * corr);
          mx[s] = mn;
        }
      }
    }
  }
  float sq = 0.f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if (tq0 + s >= T_len) continue;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float h = acc[s][e] / l[s];
      sq = fmaf(h, h, sq);
    }
  }
  sq = warp_sum(sq);
  if (lane == 0) red[wid] = sq;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    partial[(size_t)i * gridDim.y + blk] = t;
  }
}

// norms[u] = sqrt(sum_p partial[u * su + p * sp]), p in order
__global__ void label_reduce_kernel(const float* partial, int n_units, int n_parts, int su, int sp,
                                    float* norms) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n_units) return;
  float s = 0.f;
  for (int p = 0; p < n_parts; ++p) s += partial[(size_t)u * su + (size_t)p * sp];
  norms[u] = sqrtf(s);
}

// ---- host ------------------------------------------------------------------------

constexpr size_t kGemmSmem = 1024 + kLSt * (kLM * 128 + kLN * 128);

template <typename T, int MODE>
cudaError_t gemm_attr() {
  static PerDevice attr;  // function attributes are per device
  return (cudaError_t)attr.get(current_device(), [] {
    return (int)cudaFuncSetAttribute(label_gemm_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kGemmSmem);
  });
}

template <typename T>
cudaError_t neurons_t(const LabelLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap mA, mB;
  if (!make_map(&mA, L.W1n, L.d, L.N, kLM, bf16) || !make_map(&mB, L.X, L.d, L.T, kLN, bf16))
    return cudaErrorInvalidValue;
  cudaError_t e = gemm_attr<T, kNeuron>();
  if (e != cudaSuccess) return e;
  LabelArgs a{};
  a.rowsA = L.N; a.rowsB = L.T; a.d = L.d; a.partial = L.partial; a.N = L.N;
  a.T = L.T; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  const int parts = (L.T + kLN - 1) / kLN;
  label_gemm_kernel<T, kNeuron><<<dim3((L.N + kLM - 1) / kLM, parts), 128, kGemmSmem, stream>>>(mA, mB, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  label_reduce_kernel<<<(L.N + 255) / 256, 256, 0, stream>>>(L.partial, L.N, parts, 1, L.N, L.norms);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(2);
  return e;
}

template <typename T, int DH>
cudaError_t heads_t(const LabelLaunch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap mA, mB;
  const int rows = L.h * 3 * DH;
  if (!make_map(&mA, L.X, L.d, L.T, kLM, bf16) || !make_map(&mB, L.Wqkv, L.d, rows, kLN, bf16))
    return cudaErrorInvalidValue;
  cudaError_t e = gemm_attr<T, kQkv>();
  if (e != cudaSuccess) return e;
  LabelArgs a{};
  a.rowsA = L.T; a.rowsB = rows; a.d = L.d; a.Q = L.Q; a.K = L.K; a.V = L.V;
  a.T = L.T; a.h = L.h; a.d_h = DH; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  label_gemm_kernel<T, kQkv><<<dim3((L.T + kLM - 1) / kLM, (rows + kLN - 1) / kLN), 128, kGemmSmem, stream>>>(
      mA, mB, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int blocks = (L.T + kHQ - 1) / kHQ;
  head_norm_kernel<T, DH><<<dim3(L.h, blocks), 256, 0, stream>>>(
      L.Q, static_cast<const T*>(L.K), static_cast<const T*>(L.V), L.T, L.scale, L.partial);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  label_reduce_kernel<<<(L.h + 255) / 256, 256, 0, stream>>>(L.partial, L.h, blocks, blocks, 1, L.norms);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(3);
  return e;
}

}  // namespace

cudaError_t launch_label_neurons(const LabelLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return neurons_t<__half>(L, hdr, stream);
  if (dt == DV_BF16) return neurons_t<__nv_bfloat16>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_label_heads(const LabelLaunch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return L.d_h == 128 ? heads_t<__half, 128>(L, hdr, stream) : heads_t<__half, 64>(L, hdr, stream);
  if (dt == DV_BF16)
    return L.d_h == 128 ? heads_t<__nv_bfloat16, 128>(L, hdr, stream)
                        : heads_t<__nv_bfloat16, 64>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dv

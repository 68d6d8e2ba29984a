// q/K/V projections of one token (batch 1) on the tcgen05 tensor cores, with
// the KV repair of the selected heads folded into the same weight read
// (Deja Vu reading notes, "Sparsified Attention": only the selected heads'
// W^Q, W^K, W^V rows are read; the blog page §3.2: positions whose K/V were
// skipped while a head was unselected are recomputed from the stored layer
// inputs when the head is selected again).
//
// A tile is one (selected head i, m in {Q, K, V}) block of d_h = 128
// contiguous weight rows, the MMA's M.  Its N = 16 columns are the vectors
// the rows are multiplied with:
//   chunk 0:  the current token y (rows 0-3, one 4-row gather of y's only
//             row) and up to 12 skipped positions' stored inputs X[j];
//   chunk c:  16 further skipped positions (heads skipped for long).
// Q tiles have only y.  Each tile is split along d over a cluster of S <= 8
// CTAs; every CTA accumulates its slice of d in TMEM, pushes each partial
// row into the shared memory of the CTA that owns the row (128 / S rows each,
// distributed shared memory), and after one cluster barrier every CTA sums
// its own rows over the S partials and writes them:
// q in fp32, K/V rounded to the storage type at p and at the repaired
// positions.  The weight tiles are requested before the wait for the
// producer of y (launch overlap); the decode kernel marks the repaired
// positions valid, as after the CUDA-core projection kernel.
//
// The first stages' weight tiles are requested right after set-up, before
// the scan for skipped positions and before the wait for y.  The decode
// kernel is released at once, and a 4-stage ring leaves room for one of its
// CTAs beside two of these, so its K/V loads of already-valid positions run
// during the projection (OPT-13B-shaped step 41.4 -> 39.6 us per layer; with
// 5 stages the early release cost 1-3 %).  One thread issues the TMA copies,
// one issues the MMAs; every wait is bounded (dv_set_wait_limit_ns) and
// reports DV_ERR_TIMEOUT.
// Two warps of block 0 also append the token (X[p] = y, the valid column p)
// while its tiles stream.

#include <cuda.h>

#include <type_traits>

#include "dv_kernels.h"
#include "tc_common.cuh"
#include "tma_map.h"

namespace dv {
namespace {

constexpr int kQM = 128;   // rows per tile = d_h
constexpr int kQN = 16;    // MMA N: vectors per chunk
constexpr int kQKB = 64;   // d elements per stage
constexpr int kQThreads = 128;
constexpr int kQMaxPos = 4096;  // n_max bound: the skipped positions of a head fit one list
constexpr long long kUnwindNs = 2000000000LL;

struct Qkv1Args {
  const int32_t* U;        // selected heads [capU] (the row's head list)
  const int32_t* U_count;
  int capU;
  const int32_t* pos;
  int h, d, n_max;
  uint8_t* valid;          // [h][n_max]
  const void* y;           // [d]
  void* X;                 // [n_max][d]
  float* q;                // [capU][128]
  void* K;                 // [h][n_max][128]
  void* V;
  int S;
  int pdl;
  WsHeader* hdr;
  long long wait_ns;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// X[p] = y; valid[.][p] = 1 for the selected heads, 0 for the others (the
// column may hold flags of an earlier pass over the cache), by `nt` threads
// (t0 = this thread's index among them), without a block barrier.  Nothing
// in this call reads X[p] or the column p.
template <typename T>
__device__ void append_token(const Qkv1Args& a, int p, int nU, int t0, int nt) {
  grid_dep_wait();  // y comes from the kernel before this one
  const int C = a.d / 8;
  const uint4* src = static_cast<const uint4*>(a.y);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.X) + (size_t)p * a.d);
  for (int c = t0; c < C; c += nt) dst[c] = ld_cached(src + c);
  for (int i = t0; i < a.h; i += nt) {
    uint8_t sel = 0;
    for (int e = 0; e < nU; ++e) sel |= (uint8_t)(a.U[e] == i);
    a.valid[(size_t)i * a.n_max + p] = sel;
  }
}

template <typename T, int ST>
__global__ void __launch_bounds__(kQThreads, 1)
    qkv1_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapY,
                   const __grid_constant__ CUtensorMap mapX, Qkv1Args a) {
  constexpr uint32_t kABytes = kQM * 128, kBBytes = kQN * 128;
  constexpr uint32_t kTmemCols = 32;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[ST], empty[ST], done;
  __shared__ uint32_t tmem_base;
  __shared__ uint16_t miss_s[kQMaxPos];
  __shared__ int tmp[32];
  __shared__ int issued, consumed, flag_err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long unwind_ns = a.wait_ns > kUnwindNs ? a.wait_ns : kUnwindNs;
  const int S = a.S;
  const int tile = (int)blockIdx.x / S, split = (int)blockIdx.x % S;
  const int u = tile / 3, m = tile - 3 * (tile / 3);
  const int nU = max(0, min(*a.U_count, a.capU));
  const int p0 = a.pos[0];
  const int p = (p0 >= 0 && p0 < a.n_max) ? p0 : -1;
  const bool appender = blockIdx.x == 0;
  // the decode kernel may be scheduled at once (its CTAs fit beside two of
  // these): it requests the K/V of already-valid positions and waits for
  // this kernel before anything else
  grid_dep_launch();

  // every branch below is uniform in a cluster (one tile per cluster)
  if (p < 0 || u >= nU) {
    if (appender) {
      if (p < 0) {
        if (tid == 0) set_error(a.hdr, DV_ERR_POSITION, p0);
      } else {
        append_token<T>(a, p, nU, tid, kQThreads);
      }
    }
    return;
  }
  const int i = a.U[u];
  if (i < 0 || i >= a.h) {
    if (tid == 0 && split == 0 && m == 0) set_error(a.hdr, DV_ERR_INDEX_RANGE, i);
    if (appender) append_token<T>(a, p, nU, tid, kQThreads);
    return;
  }

  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + ST * kABytes;
  float* red = reinterpret_cast<float*>(sB + ST * kBBytes);  // [S][span][17] pushed partials (S > 1)
  if (tid == 0) {
    for (int q = 0; q < ST; ++q) {
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
  const int nk_all = (a.d + kQKB - 1) / kQKB;
  const int kb0 = split * nk_all / S;
  const int nk = (split + 1) * nk_all / S - kb0;  // >= 2: the host keeps nk_all >= 2 S
  const int wrow = (i * 3 + m) * kQM;
  // the first stages' weights now: nothing else is needed to request them
  const int first = min(nk, ST);
  if (tid == 0)
    for (int kb = 0; kb < first; ++kb) {
      tc::mbar_expect_tx(&full[kb], kABytes);
      tc::tma_load_2d(sA + kb * kABytes, &mapW, (kb0 + kb) * kQKB, wrow, &full[kb]);
    }

  // skipped positions j < p of head i (K and V tiles), ascending; p <= 4096,
  // each thread scans 32 flags
  int nmiss = 0;
  if (m > 0) {
    const uint8_t* vr = a.valid + (size_t)i * a.n_max;
    const int j0 = tid * 32;
    uint32_t w8[8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint4 v4 = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
      if (j0 + 16 * q < p) v4 = *reinterpret_cast<const uint4*>(vr + j0 + 16 * q);
      w8[4 * q] = v4.x; w8[4 * q + 1] = v4.y; w8[4 * q + 2] = v4.z; w8[4 * q + 3] = v4.w;
    }
    int mine = 0;
#pragma unroll
    for (int k = 0; k < 32; ++k) mine += (j0 + k < p) && (((w8[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0);
    int total;
    const int incl = block_inclusive_scan<kQThreads>(mine, tmp, &total);
    int r = incl - mine;
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if ((j0 + k < p) && (((w8[k >> 2] >> (8 * (k & 3))) & 0xffu) == 0)) miss_s[r++] = (uint16_t)(j0 + k);
    nmiss = total;
  }
  __syncthreads();  // miss_s is complete
  // chunk 0 takes 12 skipped positions beside y, later chunks 16
  const int nch = 1 + (nmiss > 12 ? (nmiss - 12 + kQN - 1) / kQN : 0);

  bool waited = false;

  for (int ch = 0; ch < nch; ++ch) {
    const int e0 = ch == 0 ? 0 : 12 + kQN * (ch - 1);
    const int ne = max(0, min(nmiss - e0, ch == 0 ? 12 : kQN));  // skipped positions in this chunk
    const int ng = (ne + 3) / 4;                                 // 4-row gathers of X
    const uint32_t offX = ch == 0 ? 512u : 0u;                   // chunk 0: y in rows 0-3
    const uint32_t bytes = kABytes + (uint32_t)(ng + (ch == 0 ? 1 : 0)) * 512u;
    if (warp == 0 && lane == 0 && !flag_err) {  // TMA producer
      auto issue_x = [&](int st, int x) {
        for (int g = 0; g < ng; ++g) {
          int r[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) r[q] = miss_s[e0 + min(4 * g + q, ne - 1)];
          tc::tma_gather4(sB + st * kBBytes + offX + g * 512, &mapX, x, r[0], r[1], r[2], r[3], &full[st]);
        }
      };
      int kb = 0;
      if (!waited) {
        // chunk 0: the first stages' weights are in flight; their stored
        // inputs now, y after the wait
        for (; kb < first; ++kb) {
          tc::mbar_arrive_expect_tx(&full[kb], bytes - kABytes);
          issue_x(kb, (kb0 + kb) * kQKB);
        }
        if (a.pdl) grid_dep_wait();
        waited = true;
        for (int k2 = 0; k2 < kb; ++k2)
          tc::tma_gather4(sB + k2 * kBBytes, &mapY, (kb0 + k2) * kQKB, 0, 0, 0, 0, &full[k2]);
      }
      for (; kb < nk && !flag_err; ++kb) {
        const int g = ch * nk + kb, st = g % ST;
        if (g >= ST && !tc::mbar_wait(&empty[st], ((g / ST) - 1) & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 42);
          flag_err = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&full[st], bytes);
        tc::tma_load_2d(sA + st * kABytes, &mapW, (kb0 + kb) * kQKB, wrow, &full[st]);
        if (ch == 0) tc::tma_gather4(sB + st * kBBytes, &mapY, (kb0 + kb) * kQKB, 0, 0, 0, 0, &full[st]);
        issue_x(st, (kb0 + kb) * kQKB);
      }
      issued = ch * nk + kb;
    } else if (appender && ch == 0 && warp >= 2) {  // idle until the epilogue: append the token
      append_token<T>(a, p, nU, tid - 64, kQThreads - 64);
    } else if (warp == 1 && lane == 0) {  // MMA issuer (after an error: only the commit)
      constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
      const uint32_t idesc = tc::idesc_f16(kQM, kQN, kBf16, false, false);
      for (int kb = 0; kb < nk && !flag_err; ++kb) {
        const int g = ch * nk + kb, st = g % ST;
        if (!tc::mbar_wait(&full[st], (g / ST) & 1, a.wait_ns)) {
          set_error(a.hdr, DV_ERR_TIMEOUT, 43);
          flag_err = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t aBase = tc::saddr(sA + st * kABytes), bBase = tc::saddr(sB + st * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kQKB / 16; ++kk) {
          const uint64_t ad = tc::smem_desc(aBase + kk * 32, 16, 1024, 2);
          const uint64_t bd = tc::smem_desc(bBase + kk * 32, 16, 1024, 2);
          tc::mma_f16(tmem, ad, bd, idesc, (kb | kk) != 0);
        }
        tc::mma_commit(&empty[st]);
        consumed = g + 1;
      }
      tc::mma_commit(&done);
    }
    __syncwarp();

    const bool ok = tc::mbar_wait(&done, ch & 1, unwind_ns);
    if (!ok && lane == 0) {
      set_error(a.hdr, DV_ERR_TIMEOUT, 44);
      flag_err = 1;  // later chunks issue nothing (but keep the cluster barriers)
    }
    __syncwarp();
    tc::fence_after_sync();
    float v[kQN];
#pragma unroll
    for (int c = 0; c < kQN; c += 8) tc::tmem_ld8(tmem + ((uint32_t)(warp * 32) << 16) + c, v + c);
    tc::tmem_ld_wait();
    tc::fence_before_sync();
    __syncthreads();  // flag_err is final for this chunk; TMEM may be overwritten by the next chunk
    const bool good = ok && !flag_err;
    // column c of this chunk -> position (or -1: unused); column 0 of chunk 0 is y
    auto col_pos = [&](int c) -> int {
      if (ch == 0) {
        if (c == 0) return p;
        return (c >= 4 && c - 4 < ne) ? (int)miss_s[e0 + c - 4] : -1;
      }
      return c < ne ? (int)miss_s[e0 + c] : -1;
    };
    auto store = [&](int t, int c, float z) {
      if (m == 0) {
        if (c == 0) a.q[(size_t)u * kQM + t] = z;
        return;
      }
      const int j = col_pos(c);
      if (j < 0) return;
      T* dst = static_cast<T*>(m == 1 ? a.K : a.V);
      dst[((size_t)i * a.n_max + j) * kQM + t] = Elem<T>::from_f(z);
    };
    const int ncol = m == 0 ? 1 : (ch == 0 ? 4 + ne : ne);
    if (S == 1) {
#pragma unroll
      for (int c = 0; c < kQN; ++c)
        if (good && c < ncol) store(tid, c, v[c]);
    } else {
      // push this CTA's partial rows into the CTA that owns them (slot
      // `split` of the owner's [S][span] rows), one cluster barrier, then
      // sum the owned rows from local shared memory: no remote reads, so
      // nothing waits for a second barrier before a CTA leaves
      const int span = (kQM + S - 1) / S;
      if (ch > 0) {  // the owners have finished the previous chunk's sums
        cluster_arrive();
        cluster_wait();
      }
      {
        const int owner = tid / span, lr = tid - owner * span;
        float* dst = red + ((size_t)split * span + lr) * (kQN + 1);
#pragma unroll
        for (int c = 0; c < kQN; ++c)
          if (c < ncol) st_dsmem_f32(dst + c, (uint32_t)owner, good ? v[c] : 0.f);
      }
      cluster_arrive();
      cluster_wait();
      const int r0 = split * span, nr = max(0, min(kQM - r0, span));
      for (int e = tid; e < nr * ncol; e += kQThreads) {
        const int c = e / nr, lr = e - c * nr;
        float z = 0.f;
        for (int q = 0; q < S; ++q) z += red[((size_t)q * span + lr) * (kQN + 1) + c];
        if (good) store(r0 + lr, c, z);
      }
    }
  }

  // no TMA write into this CTA's shared memory may still be in flight
  if (tid == 0) {
    for (int g = consumed; g < issued; ++g)
      if (!tc::mbar_wait(&full[g % ST], (g / ST) & 1, unwind_ns)) break;
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int ST>
cudaError_t qkv1_attr(size_t smem) {
  static PerDevice attr;  // function attributes are per device
  return (cudaError_t)attr.get(current_device(), [smem] {
    return (int)cudaFuncSetAttribute(qkv1_tc_kernel<T, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
}

template <typename T, int ST>
cudaError_t qkv1_launch(CUtensorMap& mW, CUtensorMap& mY, CUtensorMap& mX, Qkv1Args& a, int tiles, int pdl,
                        cudaStream_t stream) {
  const size_t smem = 1024 + ST * (kQM * 128 + kQN * 128) + (size_t)(kQM + 8) * (kQN + 1) * 4;
  cudaError_t e = qkv1_attr<T, ST>(smem);
  if (e != cudaSuccess) return e;
  return launch_k(qkv1_tc_kernel<T, ST>, dim3(tiles * a.S), dim3(kQThreads), smem, stream, pdl != 0, a.S, mW, mY,
                  mX, a);
}

template <typename T>
cudaError_t qkv1_t(const Qkv1Launch& L, WsHeader* hdr, cudaStream_t stream) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap mW, mY, mX;
  if (!make_map(&mW, L.Wqkv, L.d, (uint64_t)L.h * 3 * kQM, kQM, bf16) || !make_map(&mY, L.y, L.d, 1, 1, bf16) ||
      !make_map(&mX, L.X, L.d, L.n_max, 1, bf16))
    return cudaErrorInvalidValue;
  Qkv1Args a{};
  a.U = L.U; a.U_count = L.U_count; a.capU = L.capU; a.pos = L.pos;
  a.h = L.h; a.d = L.d; a.n_max = L.n_max; a.valid = L.valid;
  a.y = L.y; a.X = L.X; a.q = L.q; a.K = L.K; a.V = L.V;
  a.pdl = L.pdl; a.hdr = hdr; a.wait_ns = wait_limit_ns();
  const int tiles = 3 * L.capU;
  const int nk = (L.d + kQKB - 1) / kQKB;
  const int sms = num_sms_current();
  // Split d into S slices (one cluster of S CTAs per tile), doubling S while
  // two CTAs per SM still hold the grid and every slice keeps 4+ stages.
  // Clusters of 5 or 6 CTAs (one wave on paper) measured slower: with the
  // previous kernel still resident under launch overlap, whole clusters wait
  // for room in a GPC, so the grid keeps slack.
  a.S = 1;
  while (a.S < 8 && tiles * a.S * 2 <= 2 * sms && nk >= 8 * a.S) a.S *= 2;
  return qkv1_launch<T, 4>(mW, mY, mX, a, tiles, L.pdl, stream);
}

}  // namespace

bool qkv1_tc_supported(int B, int d, int d_h, int n_max, dv_dtype dt) {
  return B == 1 && dt != DV_F32 && d_h == kQM && d % kQKB == 0 && n_max <= kQMaxPos;
}

cudaError_t launch_qkv1_tc(const Qkv1Launch& L, dv_dtype dt, WsHeader* hdr, cudaStream_t stream) {
  if (dt == DV_F16) return qkv1_t<__half>(L, hdr, stream);
  if (dt == DV_BF16) return qkv1_t<__nv_bfloat16>(L, hdr, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dv

// Decoder-step helpers: the pre-LayerNorm of each sparse block and the
// position counter of a decode loop.

#include <atomic>

#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kLnThreads = 512;
constexpr int kLnVec = 8;  // float4 per thread: d <= 512 * 4 * 8 = 16384

__device__ __forceinline__ float block_sum_ln(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];  // same order in every thread
  __syncthreads();
  return t;
}

template <typename T> struct Store4;
template <> struct Store4<float> {
  static __device__ __forceinline__ void put(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};
template <> struct Store4<__half> {
  static __device__ __forceinline__ void put(__half* p, float4 v) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};
template <> struct Store4<__nv_bfloat16> {
  static __device__ __forceinline__ void put(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// y = (x - mean) / sqrt(var + eps) per row, rounded to the storage type.  The
// row is read once into registers (one round trip); mean and variance are
// two block reductions over the registers.
template <typename T>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(const float* x, int d, float eps, T* y) {
  __shared__ float red[kLnThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  // Launched programmatically: the input is read only after the previous
  // kernel has completed, so this is safe after any kernel.  A consumer
  // launched with overlap may start at once and request its weights while
  // the kernel before this one still runs (dv_set_launch_overlap).
  grid_dep_launch();
  grid_dep_wait();
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)b * d);
  const int n4 = d / 4;
  float4 v[kLnVec];
#pragma unroll
  for (int k = 0; k < kLnVec; ++k) {
    const int c = tid + k * kLnThreads;
    v[k] = c < n4 ? __ldcg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kLnVec; ++k) s += (v[k].x + v[k].y) + (v[k].z + v[k].w);
  const float mean = block_sum_ln(s, red) / (float)d;
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < kLnVec; ++k) {
    if (tid + k * kLnThreads < n4) {
      const float a0 = v[k].x - mean, a1 = v[k].y - mean, a2 = v[k].z - mean, a3 = v[k].w - mean;
      q = fmaf(a0, a0, q); q = fmaf(a1, a1, q); q = fmaf(a2, a2, q); q = fmaf(a3, a3, q);
    }
  }
  const float inv = 1.f / sqrtf(block_sum_ln(q, red) / (float)d + eps);
  T* yr = y + (size_t)b * d;
#pragma unroll
  for (int k = 0; k < kLnVec; ++k) {
    const int c = tid + k * kLnThreads;
    if (c < n4)
      Store4<T>::put(yr + 4 * c, make_float4((v[k].x - mean) * inv, (v[k].y - mean) * inv,
                                             (v[k].z - mean) * inv, (v[k].w - mean) * inv));
  }
}

__global__ void positions_kernel(int32_t* pos, int B, int lo, int hi) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int n = pos[b] + 1;
    pos[b] = n >= hi ? lo : n;
  }
}

}  // namespace

namespace {
std::atomic<int> g_launch_overlap{0};
constexpr long long kDefaultWaitNs = 1000000000LL;  // one second
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<long long> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launches_total() { return g_launches.load(std::memory_order_relaxed); }

int launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed); }
int set_launch_overlap(int level) { return g_launch_overlap.exchange(level > 0 ? 1 : 0); }

long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
long long set_wait_limit_ns(long long ns) {
  return g_wait_ns.exchange(ns > 0 ? ns : kDefaultWaitNs);
}

cudaError_t launch_layernorm(const float* x, int B, int d, float eps, void* y, dv_dtype dt,
                             cudaStream_t stream) {
  switch (dt) {
    case DV_F32:
      return launch_k(layernorm_kernel<float>, dim3(B), dim3(kLnThreads), 0, stream, true, 1, x, d, eps,
                      static_cast<float*>(y));
    case DV_F16:
      return launch_k(layernorm_kernel<__half>, dim3(B), dim3(kLnThreads), 0, stream, true, 1, x, d, eps,
                      static_cast<__half*>(y));
    case DV_BF16:
      return launch_k(layernorm_kernel<__nv_bfloat16>, dim3(B), dim3(kLnThreads), 0, stream, true, 1, x, d,
                      eps, static_cast<__nv_bfloat16*>(y));
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_positions_advance(int32_t* pos, int B, int lo, int hi, cudaStream_t stream) {
  positions_kernel<<<(B + 127) / 128, 128, 0, stream>>>(pos, B, lo, hi);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

int num_sms_current() {
  static PerDevice cache;  // SM counts are per device
  const int dev = current_device();
  return cache.get(dev, [dev] {
    int n = 0;
    if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    return n;
  });
}

}  // namespace dv

// Decoder-step helpers: the pre-LayerNorm of each sparse block and the
// position counter of a decode loop.

#include "dv_kernels.h"

namespace dv {
namespace {

constexpr int kLnThreads = 512;

// y = (x - mean) / sqrt(var + eps) per row, rounded to the storage type.
template <typename T>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(const float* x, int d, float eps, T* y) {
  __shared__ float red[kLnThreads / 32];
  __shared__ float stat;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float* xr = x + (size_t)b * d;
  float s = 0.f;
  for (int c = tid; c < d; c += kLnThreads) s += xr[c];
  s = warp_sum(s);
  if (lane == 0) red[wid] = s;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];
    stat = t / (float)d;
  }
  __syncthreads();
  const float mean = stat;
  float q = 0.f;
  for (int c = tid; c < d; c += kLnThreads) {
    const float v = xr[c] - mean;
    q = fmaf(v, v, q);
  }
  q = warp_sum(q);
  __syncthreads();
  if (lane == 0) red[wid] = q;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];
    stat = 1.f / sqrtf(t / (float)d + eps);
  }
  __syncthreads();
  const float inv = stat;
  T* yr = y + (size_t)b * d;
  for (int c = tid; c < d; c += kLnThreads) yr[c] = Elem<T>::from_f((xr[c] - mean) * inv);
}

__global__ void positions_kernel(int32_t* pos, int B, int lo, int hi) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int n = pos[b] + 1;
    pos[b] = n >= hi ? lo : n;
  }
}

}  // namespace

cudaError_t launch_layernorm(const float* x, int B, int d, float eps, void* y, dv_dtype dt,
                             cudaStream_t stream) {
  switch (dt) {
    case DV_F32: layernorm_kernel<float><<<B, kLnThreads, 0, stream>>>(x, d, eps, static_cast<float*>(y)); break;
    case DV_F16: layernorm_kernel<__half><<<B, kLnThreads, 0, stream>>>(x, d, eps, static_cast<__half*>(y)); break;
    case DV_BF16:
      layernorm_kernel<__nv_bfloat16><<<B, kLnThreads, 0, stream>>>(x, d, eps, static_cast<__nv_bfloat16*>(y));
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_positions_advance(int32_t* pos, int B, int lo, int hi, cudaStream_t stream) {
  positions_kernel<<<(B + 127) / 128, 128, 0, stream>>>(pos, B, lo, hi);
  return cudaGetLastError();
}

}  // namespace dv

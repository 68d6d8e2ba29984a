// Column-sliced weighted row sum as its own kernel (rows_combine.cuh): the
// attention output projection and, when the MLP is not fused, its second
// product.

#include "rows_combine.cuh"

namespace dv {
namespace {

template <typename T, int BT>
__global__ void __launch_bounds__(kRcThreads) rows_combine_kernel(CombineLaunch a, int b0) {
  rows_combine_block<T, BT>(a, b0, (int)blockIdx.x, [] {
    grid_dep_wait();
    grid_dep_launch();  // a following layernorm may be scheduled; it waits for this kernel
  });
}

template <typename T>
cudaError_t combine_t(const CombineLaunch& a, cudaStream_t stream) {
  const int grid = (a.d / Elem<T>::kVec + kRcCW - 1) / kRcCW;
  for (int b0 = 0; b0 < a.B;) {
    const int nb = a.B - b0;
    const int bt = nb >= 4 ? 4 : (nb >= 2 ? 2 : 1);
    cudaError_t e;
    switch (bt) {
      case 4: e = launch_k(rows_combine_kernel<T, 4>, dim3(grid), dim3(kRcThreads), 0, stream, true, 1, a, b0); break;
      case 2: e = launch_k(rows_combine_kernel<T, 2>, dim3(grid), dim3(kRcThreads), 0, stream, true, 1, a, b0); break;
      default: e = launch_k(rows_combine_kernel<T, 1>, dim3(grid), dim3(kRcThreads), 0, stream, true, 1, a, b0); break;
    }
    if (e != cudaSuccess) return e;
    b0 += bt;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_rows_combine(const CombineLaunch& a, dv_dtype dt, cudaStream_t stream) {
  switch (dt) {
    case DV_F32: return combine_t<float>(a, stream);
    case DV_F16: return combine_t<__half>(a, stream);
    case DV_BF16: return combine_t<__nv_bfloat16>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dv

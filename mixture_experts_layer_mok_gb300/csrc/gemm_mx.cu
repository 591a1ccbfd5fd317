// Block-scaled (MXFP8) grouped-GEMM instantiations for the MXFP8 forward:
// gate/up + SwiGLU + h requantisation, down + router scale + scatter, dense
// store (shared expert).
#include "gemm_launch.cuh"
#include "gemm_mx.cuh"
#include "internal.h"

namespace mok {

template <int BN, int EPI>
cudaError_t launch_gemm_mx(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t st) {
  using C = MxCfg<BN, EPI>;
  if (grid <= 0) return cudaSuccess;
  auto kern = gemm_mx_kernel<BN, EPI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  set_dependent_launch(&attr[0]);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, maps, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template cudaError_t launch_gemm_mx<256, EPI_SWIGLU_MX>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<256, EPI_SCALE_SCATTER>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<128, EPI_SCALE_SCATTER>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<256, EPI_STORE_ROWS>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<128, EPI_STORE_ROWS>(const GemmMaps&, const GemmParams&, int, cudaStream_t);

}  // namespace mok

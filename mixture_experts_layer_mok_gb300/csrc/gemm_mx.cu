// Block-scaled (MXFP8) grouped-GEMM instantiations for the MXFP8 forward:
// gate/up + SwiGLU + h requantisation, down + router scale + scatter, dense
// store (shared expert).
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
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(maps, p);
  return cudaGetLastError();
}

template cudaError_t launch_gemm_mx<256, EPI_SWIGLU_MX>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<256, EPI_SCALE_SCATTER>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<128, EPI_SCALE_SCATTER>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<256, EPI_STORE_ROWS>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm_mx<128, EPI_STORE_ROWS>(const GemmMaps&, const GemmParams&, int, cudaStream_t);

}  // namespace mok

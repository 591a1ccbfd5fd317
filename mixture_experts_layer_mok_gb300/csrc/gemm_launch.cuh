// Definition of launch_gemm; included only by the files that instantiate it.
#pragma once

#include "gemm.cuh"
#include "internal.h"

namespace mok {

template <int A_SRC, int B_SRC, int BN, int EPI>
cudaError_t launch_gemm(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t st) {
  using C = GemmCfg<A_SRC, B_SRC, BN, EPI>;
  if (grid <= 0) return cudaSuccess;
  auto kern = gemm_kernel<A_SRC, B_SRC, BN, EPI>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(maps, p);
  return cudaGetLastError();
}

#define MOK_INSTANTIATE_GEMM(A, B, BN, EPI) \
  template cudaError_t launch_gemm<A, B, BN, EPI>(const GemmMaps&, const GemmParams&, int, cudaStream_t);

}  // namespace mok

// Definitions of launch_gemm / launch_gemm_pair; included only by the files
// that instantiate them.
#pragma once

#include "gemm.cuh"
#include "internal.h"

namespace mok {

// Every GEMM launch allows programmatic stream serialization: its CTAs may
// start while the previous kernel on the stream finishes, and wait for it in
// griddep_wait() before reading any global memory.
inline void set_dependent_launch(cudaLaunchAttribute* a) {
  a->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a->val.programmaticStreamSerializationAllowed = 1;
}

template <int A_SRC, int B_SRC, int BN, int EPI>
cudaError_t launch_gemm(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t st) {
  using C = GemmCfg<A_SRC, B_SRC, BN, EPI>;
  if (grid <= 0) return cudaSuccess;
  auto kern = gemm_kernel<A_SRC, B_SRC, BN, EPI>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
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
  GemmParams q = p;
  resolve_item_order(q, false);
  if (!C::kDyn) q.ticket = nullptr;
  err = cudaLaunchKernelEx(&cfg, kern, maps, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// CTA-pair launch: clusters of two CTAs, as many as can be resident at once
// (at most `max_items`, the bound on pair work items), each looping over
// items.
template <int A_SRC, int B_SRC, int BN, int EPI>
cudaError_t launch_gemm_pair(const GemmMaps& maps, const GemmParams& p, long long max_items, cudaStream_t st) {
  using C = GemmCfg<A_SRC, B_SRC, BN, EPI, true>;
  if (max_items <= 0) return cudaSuccess;
  auto kern = gemm_kernel<A_SRC, B_SRC, BN, EPI, true>;
  static int resident[64] = {};   // resident clusters per device, looked up once
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_dependent_launch(&attr[1]);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
  if (resident[dev] == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    cfg.gridDim = dim3(2 * (sms / 2));
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (err != cudaSuccess) return err;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    resident[dev] = n;
  }
  const long long clusters = max_items < resident[dev] ? max_items : resident[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cfg.numAttrs = 2;
  GemmParams q = p;
  resolve_item_order(q, true);
  if (!C::kDyn) q.ticket = nullptr;
  err = cudaLaunchKernelEx(&cfg, kern, maps, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

#define MOK_INSTANTIATE_GEMM(A, B, BN, EPI) \
  template cudaError_t launch_gemm<A, B, BN, EPI>(const GemmMaps&, const GemmParams&, int, cudaStream_t);
#define MOK_INSTANTIATE_GEMM_PAIR(A, B, BN, EPI)                                                        \
  template cudaError_t launch_gemm_pair<A, B, BN, EPI>(const GemmMaps&, const GemmParams&, long long, \
                                                       cudaStream_t);

}  // namespace mok

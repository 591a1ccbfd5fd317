// Block-scaled (MXFP8) grouped-GEMM instantiations.  Forward: gate/up + SwiGLU
// + h requantisation, down + router scale (rows in schedule order), dense store
// (shared expert); single CTAs and CTA pairs.  Backward (MXFP8 mode): SwiGLU
// backward, weight gradients and the dgrad rows; single CTAs.
#include "gemm_launch.cuh"
#include "gemm_mx.cuh"
#include "internal.h"

namespace mok {

template <int BN, int EPI>
cudaError_t launch_gemm_mx(const MxMaps& maps, const GemmParams& p, int grid, cudaStream_t st) {
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
  GemmParams q = p;
  resolve_item_order(q, false);
  err = cudaLaunchKernelEx(&cfg, kern, maps, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// CTA-pair launch: as many two-CTA clusters as can be resident (at most
// max_items), each looping over pair items.
template <int BN, int EPI>
cudaError_t launch_gemm_mx_pair(const MxMaps& maps, const GemmParams& p, long long max_items, cudaStream_t st) {
  using C = MxCfg<BN, EPI, true>;
  if (max_items <= 0) return cudaSuccess;
  auto kern = gemm_mx_kernel<BN, EPI, true>;
  static int resident[64] = {};
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
  err = cudaLaunchKernelEx(&cfg, kern, maps, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

#define MOK_INSTANTIATE_MX(BN, EPI) \
  template cudaError_t launch_gemm_mx<BN, EPI>(const MxMaps&, const GemmParams&, int, cudaStream_t);
#define MOK_INSTANTIATE_MX_PAIR(BN, EPI) \
  template cudaError_t launch_gemm_mx_pair<BN, EPI>(const MxMaps&, const GemmParams&, long long, cudaStream_t);

MOK_INSTANTIATE_MX(256, EPI_SWIGLU_MX)
MOK_INSTANTIATE_MX(256, EPI_SCALE_ROWS)
MOK_INSTANTIATE_MX(128, EPI_SCALE_ROWS)
MOK_INSTANTIATE_MX(256, EPI_STORE_ROWS)
MOK_INSTANTIATE_MX(128, EPI_STORE_ROWS)
// MXFP8 backward: SwiGLU backward through down (128-wide tiles keep its
// per-thread accumulator share in registers), weight gradients, dgrad rows
MOK_INSTANTIATE_MX(128, EPI_DOWN_BWD_MX)
MOK_INSTANTIATE_MX(256, EPI_WGRAD)
MOK_INSTANTIATE_MX(128, EPI_WGRAD)
MOK_INSTANTIATE_MX_PAIR(256, EPI_SWIGLU_MX)
MOK_INSTANTIATE_MX_PAIR(256, EPI_SCALE_ROWS)
MOK_INSTANTIATE_MX_PAIR(256, EPI_STORE_ROWS)
// CTA pairs with 128-wide tiles: M = 256 over the pair, a double-buffered
// 128-column accumulator beside an 8-stage scale ring in each CTA's TMEM
MOK_INSTANTIATE_MX_PAIR(128, EPI_SWIGLU_MX)
MOK_INSTANTIATE_MX_PAIR(128, EPI_SCALE_ROWS)
MOK_INSTANTIATE_MX_PAIR(128, EPI_STORE_ROWS)

}  // namespace mok

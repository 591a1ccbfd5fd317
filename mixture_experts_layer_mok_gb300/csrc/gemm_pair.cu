// CTA-pair instantiations of the grouped GEMM engine: every TMA-fed GEMM of
// the layer with 256-wide tiles (forward gate/up, down; backward down dgrad,
// both weight gradients, gate/up dgrad; routed and shared).
#include "gemm_launch.cuh"

namespace mok {
MOK_INSTANTIATE_GEMM_PAIR(SRC_K_TILE, SRC_K_TILE, 256, EPI_SWIGLU)
MOK_INSTANTIATE_GEMM_PAIR(SRC_K_TILE, SRC_K_TILE, 256, EPI_SCALE_ROWS)
MOK_INSTANTIATE_GEMM_PAIR(SRC_K_TILE, SRC_K_TILE, 256, EPI_STORE_ROWS)
MOK_INSTANTIATE_GEMM_PAIR(SRC_K_TILE, SRC_MN_TILE, 256, EPI_DOWN_BWD)
MOK_INSTANTIATE_GEMM_PAIR(SRC_K_TILE, SRC_MN_TILE, 256, EPI_STORE_ROWS)
MOK_INSTANTIATE_GEMM_PAIR(SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD)
}  // namespace mok

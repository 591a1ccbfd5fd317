// Backward grouped-GEMM instantiations, part 2: per-expert weight gradients
// (contraction over each expert's schedule rows; token rows gathered by TMA).
#include "gemm_launch.cuh"

namespace mok {
MOK_INSTANTIATE_GEMM(SRC_MN_GATHER, SRC_MN_TILE, 256, EPI_WGRAD)
MOK_INSTANTIATE_GEMM(SRC_MN_GATHER, SRC_MN_TILE, 128, EPI_WGRAD)
MOK_INSTANTIATE_GEMM(SRC_MN_TILE, SRC_MN_GATHER, 256, EPI_WGRAD)
MOK_INSTANTIATE_GEMM(SRC_MN_TILE, SRC_MN_GATHER, 128, EPI_WGRAD)
MOK_INSTANTIATE_GEMM(SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD)
MOK_INSTANTIATE_GEMM(SRC_MN_TILE, SRC_MN_TILE, 128, EPI_WGRAD)
}  // namespace mok

// Internal launch interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mok {

constexpr int kTileRows = 128;     // rows per expert tile
constexpr int kGroupTiles = 32;    // work group of the grouped GEMMs: at most this many tiles
constexpr int kGroupPairs = 16;    // ... or tile pairs, of one expert
constexpr int kSchedChunk = 1024;  // routed rows per schedule block

struct GemmMaps;
struct GemmParams;

// Launches `kern` allowing programmatic stream serialization: it may start
// while the previous kernel on the stream finishes, so it must call
// griddep_wait() before touching global memory.
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_schedule(const int64_t* te, int T, int k, int E, int cap_tiles, int max_tiles,
                            int* hist, int* cnt, int* row0, int* row_src, int* slot_row,
                            int* tile_expert, int* tile_row0, int* tile_rows, int* pair_tile, int* unit_group,
                            int* header, cudaStream_t st);
cudaError_t launch_mx_quantize(const uint16_t* x, long long nblocks, uint8_t* codes, uint8_t* scales,
                               int num_sms, cudaStream_t st);
// Schedule rows [w0, w0 + wrows) go to rows from 0 of xp (and xb); xq (may be
// NULL): the token-order copy, with the scales row-major in xs ([T][H/32]);
// xb (may be NULL): also x's bf16 rows in schedule order (padding rows zero).
cudaError_t launch_mx_dispatch(const uint16_t* x, int T, int H, int topk, const int* slot_row, const int* row_src,
                               const int* header, long long w0, long long wrows, uint8_t* xq, uint8_t* xs,
                               uint8_t* xp, uint16_t* xb, int num_sms, cudaStream_t st);
// The dispatch's scales xs into the tensor-core scale layout: the window's
// schedule rows into xp_sc, and token order into xq_sc (may be NULL).
cudaError_t launch_mx_scale_gather(const uint8_t* xs, int T, int H, int topk, const int* row_src, const int* header,
                                   long long w0, long long wrows, uint8_t* xp_sc, uint8_t* xq_sc, cudaStream_t st);
cudaError_t launch_mx_quantize_t(const uint16_t* src, long long ld, int batch, int R, int C, int valid_rows,
                                 const int* row_src, int topk, const int* header, uint8_t* codes, uint8_t* scales,
                                 int tiled, int num_sms, cudaStream_t st, uint8_t* rcodes = nullptr,
                                 uint8_t* rscales = nullptr, int rtiled = 0);
// One matrix of row-major E8M0 scales [rows][K/32] to rearrange into the
// tensor-core scale layout at dst (rows and K multiples of 128; rows 0 = skip).
// gate_up = 1 or 2 writes the gate (1) or up (2) rows of a SwiGLU weight into
// the interleaved gate|up layout the CTA-pair SwiGLU GEMM with 128-wide tiles
// reads: with `group` rows per expert, row n of expert e lands on combined row
// e*2*group + (n/64)*128 + (gate_up == 2 ? 64 : 0) + n%64, so one 512-byte
// atom holds the scales of 64 gate rows and the 64 up rows of the same columns.
struct MxTileScaleJob {
  const uint8_t* src;
  long long rows;
  int K;
  uint8_t* dst;
  int gate_up = 0;
  int group = 0;
};
constexpr int kMaxScaleJobs = 6;
// All jobs (at most kMaxScaleJobs that are not skipped) in one launch.
cudaError_t launch_mx_tile_scales(const MxTileScaleJob* jobs, int n, cudaStream_t st);
cudaError_t launch_combine(const uint16_t* rows, const int* slot_row, const int* header, long long max_rows,
                           const uint16_t* base, int T, int k, int H, uint16_t* out, int num_sms, cudaStream_t st);
// Token rows of src into schedule order: schedule rows [w0, w0 + wrows) go to
// rows from 0 of out.
cudaError_t launch_permute_rows(const uint16_t* src, int T, int H, int topk, const int* slot_row, const int* row_src,
                                const int* header, long long w0, long long wrows, uint16_t* out, int num_sms,
                                cudaStream_t st);
// The schedule restricted to experts [e0, e0 + ne) (a macrobatch window):
// its tile list, pairs, work groups ([2][tiles of the window]), row offsets
// (ne + 1) and header, rows counted from row0[e0].
cudaError_t launch_window_view(const int* cnt, const int* row0, const int* header, int e0, int ne, int* tile_expert,
                               int* tile_row0, int* tile_rows, int* pair_tile, int* unit_group, int* wrow0,
                               int* wheader, cudaStream_t st);
cudaError_t launch_dw_reduce(const float* part, int nf, int ntiles, float* dw, cudaStream_t st);

// The next work-item counter (one int, zeroed) of the calling thread's current
// forward or backward call, or NULL outside one or once the call's counters
// are used up: a TMA-fed GEMM launch given one takes its work items in
// ticket order, else in the static order.
int* next_ticket();

// Grouped GEMM launch: instantiated for the operand sources / tile widths /
// epilogues the layer uses (gemm_fwd.cu, gemm_bwd.cu).
template <int A_SRC, int B_SRC, int BN, int EPI>
cudaError_t launch_gemm(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t st);

// CTA-pair launch of the same engine (M = 256 per pair, B split between the
// two CTAs); max_items bounds the pair work items (gemm_pair.cu).
template <int A_SRC, int B_SRC, int BN, int EPI>
cudaError_t launch_gemm_pair(const GemmMaps& maps, const GemmParams& p, long long max_items, cudaStream_t st);

// Block-scaled (MXFP8) grouped GEMM launches (gemm_mx.cu): single CTAs and
// CTA pairs.
struct MxMaps;
template <int BN, int EPI>
cudaError_t launch_gemm_mx(const MxMaps& maps, const GemmParams& p, int grid, cudaStream_t st);
template <int BN, int EPI>
cudaError_t launch_gemm_mx_pair(const MxMaps& maps, const GemmParams& p, long long max_items, cudaStream_t st);

}  // namespace mok

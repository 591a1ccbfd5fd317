// Persistent grouped GEMM engine on tcgen05 / TMEM / TMA for sm_103a.
//
// One CTA per SM, or one cluster of two CTAs per SM pair (CTA pairs:
// tcgen05.mma.cta_group::2, M = 256, each CTA holding half of B):
//   warp 0      TMA producer: tile loads of the operands that are not gathered
//               (and, on request, tile::gather4 loads of the gathered ones);
//   warp 1      MMA issuer (one thread; a pair's leader issues for both) and
//               TMEM owner;
//   warps 2..   epilogue (4 warps, or 8 for the SwiGLU backward and the weight
//               gradients): TMEM -> registers -> fused elementwise -> TMA
//               stores of 32x32 blocks (SwiGLU, router scaling, SwiGLU
//               backward with the router-weight grad, weight gradients);
//   last 4      gather producers (fused-dispatch variants only): 16-byte
//               cp.async copies of the token rows a schedule tile needs,
//               written straight into the 128-byte-swizzled stage layout the
//               tensor core reads (the on-chip form of MoK's dispatch exchange).
// The data-movement warps and the output warps overlap the MMA warp through a
// ring of shared-memory stages and a double-buffered TMEM accumulator: the
// single-GPU analogue of MoK's split of SMs into communication and compute
// roles ("Mixture-of-Kittens: a deterministic MoE megakernel for NVL72 racks",
// "Tuning the five hyperparameters before production": fwd/bwd_num_comm_sms).
//
// Work items are output tiles of 128 rows x BN columns (pairs: two such tiles
// sharing B); each is produced by exactly one CTA with a fixed K order, so
// results do not depend on which CTA takes which item or on the item order.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "ptx.cuh"

namespace mok {

constexpr int kBM = 128;        // rows of an output tile (TMEM lanes)
// Kernels that gather token rows use 64-element K-blocks (128-byte swizzle);
// the gather code below is written for that layout.
constexpr int kBK = 64;
constexpr int kChunkBytes = 64 * 128;  // one MN-major chunk: 64 K-rows x 64 elements

enum Src : int {
  SRC_K_TILE = 0,         // K-major rows [p0, p0+128) of a 2-D tensor (TMA box 64 x 128)
  SRC_K_GATHER = 1,       // K-major: the 128 token rows of a schedule tile (TMA gather4, box 64 x 1)
  SRC_MN_TILE = 2,        // MN-major: K-rows [k, k+64) of a 2-D tensor (TMA box 64 x 64)
  SRC_MN_GATHER = 3,      // MN-major: 64 token rows of a schedule range (TMA gather4, box 64 x 1)
  SRC_K_GATHER_LSU = 4,   // as SRC_K_GATHER, copied by the gather warps (cp.async)
  SRC_MN_GATHER_LSU = 5,  // as SRC_MN_GATHER, copied by the gather warps (cp.async)
};

enum Epi : int {
  EPI_SWIGLU = 0,        // gate|up accumulators -> G, U (bf16), h = silu(G) U (bf16)
  EPI_SWIGLU_MX = 1,     // same, h written as MXFP8 codes + E8M0 scales (gemm_mx_kernel)
  EPI_SCALE_ROWS = 2,    // out[p] = bf16(w[row_src[p]] * acc), rows in schedule order (0 for padding)
  EPI_STORE_ROWS = 3,    // out[row] = bf16(acc) for dense rows
  EPI_DOWN_BWD = 4,      // dH = w Z; SwiGLU backward; d_w partial = sum Z h; hw = w h
  EPI_WGRAD = 6,         // out[e][m][n] = bf16(acc), rows split over two tensors
  EPI_DOWN_BWD_MX = 7,   // EPI_DOWN_BWD with MXFP8 outputs (gemm_mx_kernel): dG|dU by rows,
                         // and dG|dU, w h transposed in 32-row blocks
};

struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b0;
  CUtensorMap b1;
  // outputs written by TMA stores (row-major bf16, box 32 rows x 32 columns,
  // 64-byte swizzle): SwiGLU G|U and h, SwiGLU backward dG|dU and w h, the
  // weight gradients' two tensors, dense rows
  CUtensorMap o0;
  CUtensorMap o1;
};

struct GemmParams {
  // ---- work decomposition
  int wgrad;       // 0: output rows are layer rows; 1: per-expert weight gradient
  int grouped;     // layer rows (or wgrad K-rows) come from the schedule
  int rows;        // dense: number of layer rows (T)
  int K;           // row GEMMs: contraction length (multiple of 64)
  int n_tiles;     // output column tiles
  int m_tiles;     // wgrad: output row tiles
  int E;           // wgrad: experts (1 for a dense weight)
  int topk;
  const int* header;  // schedule header: [0] num_tiles, [2] status (grouped only)
  const int* tile_expert;
  const int* tile_row0;
  const int* tile_rows;
  const int* row_src;
  const int* row0;
  const int* cnt;
  const int* pair_tile;  // CTA-pair GEMMs: [pairs][2] tile indices (second -1 = none)
  const int* tile_group; // work groups of the tiles and of the pairs (the schedule's unit_group):
  const int* pair_group; // position in the group (bits 0..7), group length (bits 8..15)
  // ---- operand coordinates
  int b_rows_per_expert;  // weight rows (K-major B) or K-rows (MN-major B) per expert
  int b_split;            // MN-major B: K index where map b1 takes over (0 = never)
  // ---- epilogue
  int N;             // logical width used by the epilogue (I for SwiGLU, ...)
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  const void* aux0;  // EPI_DOWN_BWD: saved gate|up pre-activations
  const float* rw;   // router weights [T*k] (grouped), NULL = 1
  float* dw_part;    // EPI_DOWN_BWD grouped: [T*k][n_tiles]
  long long ld;      // output row stride (elements)
  int split;         // EPI_WGRAD: first output row that goes to out1
  long long estride; // EPI_WGRAD: elements per expert in out0 / out1
  int* status;       // device status word
  int* ticket;       // TMA-fed GEMMs: this launch's work-item counter (zeroed), NULL = the static order
  int ticket_mode;   // 0: ticket order for long row GEMMs; 1: never (MOK_DEBUG_STATIC_ORDER);
                     // 2: always (MOK_DEBUG_TICKET_ORDER)
  int debug;         // MOK_DEBUG_* flags
  float swiglu_limit;  // SwiGLU epilogues: 0 = plain; L > 0 clamps gate to <= L, up to [-L, L]
  // ---- gathered operands (gather warps): token-row tensors [T][ld]
  const uint16_t* ga;
  long long ga_ld;
  const uint16_t* gb;
  long long gb_ld;
  // ---- MXFP8 operands: E8M0 scales in the tensor-core layout (mx_tiled_scale_offset)
  const uint8_t* sfa;
  const uint8_t* sfb0;
  const uint8_t* sfb1;
  uint8_t* sf_out;   // EPI_SWIGLU_MX: scales of h, same layout; EPI_DOWN_BWD_MX: of dG|dU rows
  uint8_t* sf_out2;  // EPI_DOWN_BWD_MX: scales of the transposed w h
  int sf_kga;        // 128-column groups of A's / B's scale layout (0 = K / 128); a weight
  int sf_kgb;        // gradient's operands span the whole row range, not one item's K
  // ---- order of the work items (never changes a result: each output tile has
  // one owner and a fixed K order)
  int group;         // row GEMMs: 0 = column tiles inside each row unit (tile or pair);
                     // g > 0 = row units in groups, the group's units inside each
                     // column tile (B's columns stream once per group while the
                     // group's A rows stay in L2): a grouped GEMM takes the
                     // schedule's groups (one expert each), a dense one groups of g
  int wg_col_outer;  // weight gradients: 1 = an expert's row units inside each
                     // column tile (B streams once, A stays in L2), 0 = the reverse
};

// Default work-item order, chosen at launch where p.group / p.wg_col_outer
// are -1 (-2: the plain order).  Row GEMMs take their row units (tiles, or
// pairs of tiles) in groups inside each column tile: while the group's A rows
// stay in L2, each B column slice (an expert's weights, a few MB) is read once
// for the whole group instead of once per row unit.  Grouped GEMMs take the
// schedule's groups, at most 32 tiles (16 pairs) of one expert, so that no
// group holds two experts' weights; dense ones group 16 row tiles.  Weight
// gradients walk an expert's row units inside each column tile when A (M rows
// per expert) is the smaller operand, so that B streams through once.
inline void resolve_item_order(GemmParams& p, bool pair) {
  if (p.group < 0) p.group = (p.group == -2) ? 0 : (pair ? 8 : 16);
  if (p.wg_col_outer < 0)
    p.wg_col_outer = (p.wg_col_outer == -2) ? 0 : (p.wgrad && static_cast<long long>(p.m_tiles) * kBM < p.ld ? 1 : 0);
}

// Work item idx of a grid of `units` row units x n_tiles column tiles -> (row
// unit u, column tile nt), in the order GemmParams::group describes.
__device__ __forceinline__ void unit_and_col(int idx, int units, int n_tiles, int group, int& u, int& nt) {
  if (group <= 0) {
    u = idx / n_tiles;
    nt = idx - u * n_tiles;
    return;
  }
  const int span = group * n_tiles;
  const int g = idx / span;
  const int r = idx - g * span;
  const int gs = min(group, units - g * group);   // the last group may be short
  nt = r / gs;
  u = g * group + (r - nt * gs);
}

// The same for a grouped GEMM, whose groups the schedule lists (each group a
// run of consecutive units of one expert): the items of a group of units [s,
// s + L) are [s n, (s + L) n), so the unit idx / n lies in idx's group, and its
// entry gives s and L.
__device__ __forceinline__ void listed_unit_and_col(const int* groups, int idx, int n, int& u, int& nt) {
  const int u0 = idx / n;
  const int g = __ldg(groups + u0);
  const int s = u0 - (g & 0xFF), len = g >> 8;
  const int r = idx - s * n;
  nt = r / len;
  u = s + (r - nt * len);
}

struct Item {
  int e, p0, rows, m0, nt, kbeg, nk;
  bool empty;  // CTA-pair GEMMs: this CTA's half of the pair has no tile
};

__device__ __forceinline__ int num_items(const GemmParams& p) {
  if (p.grouped && p.header[2] != 0) return 0;
  if (!p.wgrad) {
    const int mt = p.grouped ? p.header[0] : (p.rows + kBM - 1) / kBM;
    return mt * p.n_tiles;
  }
  return p.E * p.m_tiles * p.n_tiles;
}

__device__ __forceinline__ Item get_item(const GemmParams& p, int idx, int bk) {
  Item it;
  it.empty = false;
  if (!p.wgrad) {
    int mt;
    if (p.grouped && p.group > 0)
      listed_unit_and_col(p.tile_group, idx, p.n_tiles, mt, it.nt);
    else
      unit_and_col(idx, p.grouped ? p.header[0] : (p.rows + kBM - 1) / kBM, p.n_tiles, p.group, mt, it.nt);
    if (p.grouped) {
      it.e = __ldg(p.tile_expert + mt);
      it.p0 = __ldg(p.tile_row0 + mt);
      it.rows = __ldg(p.tile_rows + mt);
    } else {
      it.e = 0;
      it.p0 = mt * kBM;
      it.rows = min(kBM, p.rows - it.p0);
    }
    it.m0 = it.p0;
    it.kbeg = 0;
    it.nk = p.K / bk;
  } else {
    const int per_e = p.m_tiles * p.n_tiles;
    it.e = idx / per_e;
    const int r = idx - it.e * per_e;
    int mt;
    unit_and_col(r, p.m_tiles, p.n_tiles, p.wg_col_outer ? p.m_tiles : 0, mt, it.nt);
    it.m0 = mt * kBM;
    it.p0 = 0;
    it.rows = 0;
    if (p.grouped) {
      it.kbeg = __ldg(p.row0 + it.e);
      const int c = __ldg(p.cnt + it.e);
      it.nk = (c + kBM - 1) / kBM * (kBM / bk);
    } else {
      it.kbeg = 0;
      it.nk = (p.rows + bk - 1) / bk;
    }
  }
  return it;
}

// CTA-pair GEMMs: work items are pairs of 128-row tiles (rank 0 takes the
// first, rank 1 the second) sharing one B tile; weight gradients pair
// adjacent output row tiles of one expert.
__device__ __forceinline__ int num_items_pair(const GemmParams& p) {
  if (p.grouped && p.header[2] != 0) return 0;
  if (!p.wgrad) {
    const int pairs = p.grouped ? p.header[4] : ((p.rows + kBM - 1) / kBM + 1) / 2;
    return pairs * p.n_tiles;
  }
  return p.E * ((p.m_tiles + 1) / 2) * p.n_tiles;
}

__device__ __forceinline__ Item get_item_pair(const GemmParams& p, int idx, int bk, int rank) {
  Item it;
  it.empty = false;
  if (!p.wgrad) {
    int pr;
    if (p.grouped && p.group > 0)
      listed_unit_and_col(p.pair_group, idx, p.n_tiles, pr, it.nt);
    else
      unit_and_col(idx, p.grouped ? p.header[4] : ((p.rows + kBM - 1) / kBM + 1) / 2, p.n_tiles, p.group, pr, it.nt);
    if (p.grouped) {
      const int t0 = __ldg(p.pair_tile + 2 * pr);
      const int t1 = __ldg(p.pair_tile + 2 * pr + 1);
      const int t = (rank && t1 >= 0) ? t1 : t0;   // an empty half loads its partner's rows
      it.e = __ldg(p.tile_expert + t);
      it.p0 = __ldg(p.tile_row0 + t);
      it.rows = __ldg(p.tile_rows + t);
      it.empty = rank && t1 < 0;
    } else {
      it.e = 0;
      it.p0 = (2 * pr + rank) * kBM;               // past the last row: loads read zeros
      it.rows = min(kBM, p.rows - it.p0);
      it.empty = it.rows <= 0;
    }
    it.m0 = it.p0;
    it.kbeg = 0;
    it.nk = p.K / bk;
  } else {
    const int mp_n = (p.m_tiles + 1) / 2;
    const int per_e = mp_n * p.n_tiles;
    it.e = idx / per_e;
    const int r = idx - it.e * per_e;
    int mp;
    unit_and_col(r, mp_n, p.n_tiles, p.wg_col_outer ? mp_n : 0, mp, it.nt);
    const int mt = 2 * mp + rank;
    it.empty = mt >= p.m_tiles;
    it.m0 = (it.empty ? 2 * mp : mt) * kBM;
    it.p0 = 0;
    it.rows = 0;
    if (p.grouped) {
      it.kbeg = __ldg(p.row0 + it.e);
      const int c = __ldg(p.cnt + it.e);
      it.nk = (c + kBM - 1) / kBM * (kBM / bk);
    } else {
      it.kbeg = 0;
      it.nk = (p.rows + bk - 1) / bk;
    }
  }
  return it;
}

// The K-block count of work item idx, which is all the MMA issuer needs:
// constant for row GEMMs, an expert's row count for weight gradients (the same
// value get_item / get_item_pair give, without their row-unit lookups).
__device__ __forceinline__ int item_nk(const GemmParams& p, int idx, int bk, bool pair) {
  if (!p.wgrad) return p.K / bk;
  if (!p.grouped) return (p.rows + bk - 1) / bk;
  const int per_e = (pair ? (p.m_tiles + 1) / 2 : p.m_tiles) * p.n_tiles;
  const int c = __ldg(p.cnt + idx / per_e);
  return (c + kBM - 1) / kBM * (kBM / bk);
}

// Token row of schedule row q (padding rows read token 0; their partner
// operand row is zero, or the epilogue drops them).
__device__ __forceinline__ int token_of(const GemmParams& p, int q) {
  const int f = __ldg(p.row_src + q);
  return f >= 0 ? f / p.topk : 0;
}

// Token row of schedule row q, or -1 for a padding row (copied as zeros).
__device__ __forceinline__ int token_or_pad(const GemmParams& p, int q) {
  const int f = __ldg(p.row_src + q);
  return f >= 0 ? f / p.topk : -1;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void pack_bf16x32(const float* v, uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
}

// Warp-cooperative row store: each lane hands in 32 bf16 values (16 packed
// words) of its own row and the address they go to (NULL = store nothing).
// The warp stages its 32 row segments in 2 KB of shared memory (XOR-swizzled,
// conflict-free) and writes them back as 64-byte row segments, 8 rows per
// instruction, so every global store covers whole 32-byte sectors instead of
// 32 scattered 16-byte pieces.
__device__ __forceinline__ void warp_store_row64(const uint32_t* w, void* dst, uint8_t* stage, int lane) {
  uint4* s = reinterpret_cast<uint4*>(stage);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    s[lane * 4 + (j ^ sw)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  __syncwarp();
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int row = q * 8 + (lane >> 2), piece = lane & 3;
    const unsigned long long d = __shfl_sync(0xffffffffu, mine, row);
    const uint4 v = s[row * 4 + (piece ^ ((row >> 1) & 3))];
    if (d) reinterpret_cast<uint4*>(d)[piece] = v;
  }
  __syncwarp();
}

// Warp-cooperative TMA store of a 32-row x 32-column bf16 block at {col, row}
// of the output tensor: each lane hands in 16 packed words of its row; the
// warp stages them in the 64-byte-swizzled layout of the output's tensor map
// (the layout warp_store_row64 uses) and lane 0 stores the block with one
// bulk tensor copy.  Two 2 KB halves alternate, so staging the next block
// overlaps the copy of this one; `slot` tracks the half in use.
__device__ __forceinline__ void warp_store_tma(const uint32_t* w, const CUtensorMap* map, int col, int row,
                                               uint8_t* stage2, int& slot, int lane) {
  uint8_t* stage = stage2 + slot * 2048;
  if (lane == 0) bulk_wait_read<1>();   // the copy that last read this half is done reading
  __syncwarp();
  uint4* s = reinterpret_cast<uint4*>(stage);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    s[lane * 4 + (j ^ sw)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();             // generic-proxy writes, then the async-proxy read
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, col, row);
    bulk_commit();
  }
  slot ^= 1;
}

// Element i of 32 bf16 values held as 4 raw 16-byte words.
__device__ __forceinline__ float bf16_at(const uint4* raw, int i) {
  const uint32_t w = reinterpret_cast<const uint32_t*>(raw)[i >> 1];
  return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

__device__ __forceinline__ void load_raw64(const uint16_t* src, uint4* raw) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) raw[q] = __ldg(s + q);
}

__device__ __forceinline__ void load_bf16x32(const void* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = __ldg(s + q);
    uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i + 0] = __uint_as_float(ws[i] << 16);
      v[8 * q + 2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
    }
  }
}

// E8M0 exponent of a block: smallest s with amax <= 448 * 2^s, clamped to
// [-127, 127], 0 for amax == 0; decided from the fp32 exponent and mantissa.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xFF);
  if (b == 0) return 0;
  if (ef == 0) return -127;  // fp32 subnormal: far below 448 * 2^-127
  const int e = ef - 127;
  int s = e - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);  // mantissa above 1.75
  return max(-127, min(127, s));
}

// 32 values -> 32 E4M3 codes (RNE, satfinite) scaled by 2^-s; returns s + 127.
__device__ __forceinline__ uint32_t mx_quantize32(const float* v, uint8_t* codes_out) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_scale_exponent(amax);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);  // 2^-s, s <= 126
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * q + 0] * inv, v[4 * q + 1] * inv),
                                 __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * q + 2] * inv, v[4 * q + 3] * inv),
                                 __NV_SATFINITE, __NV_E4M3);
    w[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  uint4* d = reinterpret_cast<uint4*>(codes_out);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return static_cast<uint32_t>(s + 127);
}

// Byte offset of the E8M0 scale of element block (row, cblk) (cblk = column /
// 32) in the tensor-core scale layout of a tensor with `cgroups` = K/128
// column groups: one 512-byte atom per (128-row block, 128-column group),
// holding row r's four block scales of the group as one 32-bit word at byte
// (r % 32) * 16 + (r / 32) * 4 - the form a 32x128b.warpx4 copy puts into
// four TMEM columns, where the block-scaled MMA reads row r's scale at column
// r / 32, byte cblk % 4.
__host__ __device__ __forceinline__ long long mx_tiled_scale_offset(long long row, int cblk, int cgroups) {
  const long long atom = (row >> 7) * cgroups + (cblk >> 2);
  const int r = static_cast<int>(row & 127);
  return atom * 512 + (r & 31) * 16 + (r >> 5) * 4 + (cblk & 3);
}

template <int A_SRC, int B_SRC, int BN, int EPI, bool PAIR = false>
struct GemmCfg {
  static constexpr bool kAMN = (A_SRC == SRC_MN_TILE || A_SRC == SRC_MN_GATHER || A_SRC == SRC_MN_GATHER_LSU);
  static constexpr bool kBMN = (B_SRC == SRC_MN_TILE || B_SRC == SRC_MN_GATHER || B_SRC == SRC_MN_GATHER_LSU);
  static constexpr bool kALsu = (A_SRC == SRC_K_GATHER_LSU || A_SRC == SRC_MN_GATHER_LSU);
  static constexpr bool kBLsu = (B_SRC == SRC_MN_GATHER_LSU);
  static constexpr bool kHasLsu = kALsu || kBLsu;
  // epilogue warps: the SwiGLU backward's epilogue is the heaviest; with no
  // gather warps it gets two warps per TMEM lane quarter (each half the columns)
  static constexpr int kEpiWarps = ((EPI == EPI_DOWN_BWD || EPI == EPI_WGRAD) && !kHasLsu) ? 8 : 4;
  static constexpr int kGatherWarp0 = 2 + kEpiWarps;
  static constexpr int kThreads = 64 + 32 * kEpiWarps + (kHasLsu ? 128 : 0);
  // K-block per stage (elements): 64 bf16 = one 128-byte swizzled row.  The
  // layout code below also supports 32 (64-byte swizzle); measured slower,
  // since it doubles the TMA instructions per FLOP.
  static constexpr int kBK = 64;
  static constexpr int kRowBytes = kBK * 2;                 // one swizzled shared-memory row
  static constexpr int kMnChunkBytes = kRowBytes * kBK;     // MN-major chunk: kBK K-rows x kBK elements
  static constexpr uint32_t kSwz = (kBK == 64) ? 2u : 4u;   // descriptor swizzle: 128-byte / 64-byte
  static constexpr int kABytes = kBM * kBK * 2;
  // CTA pair: each CTA holds half of B's BN rows (the pair's MMA reads both)
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kTmaBytes = (kALsu ? 0 : kABytes) + (kBLsu ? 0 : kBBytes);
  // stage-full arrivals: the TMA warp's expect_tx, plus one hardware arrival per
  // gather thread when its copies for the stage have landed
  static constexpr uint32_t kFullArrivals = kHasLsu ? 1 + 128 : 1;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kEpiStageBytes = 4096;  // per epilogue warp: two 32-row x 64-byte blocks
  // work items in ticket order (TMA-fed GEMMs): a ring of kQ item slots
  static constexpr bool kDyn = !kHasLsu;
  static constexpr int kQ = 8;
  static constexpr int kStagesFit = (227 * 1024 - 1024 - kBarBytes - kEpiWarps * kEpiStageBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 16 ? 16 : kStagesFit;
  static constexpr int kTmemCols = 2 * BN;  // two accumulator buffers
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kEpiWarps * kEpiStageBytes;
  static constexpr uint32_t kIdesc = idesc_bf16(PAIR ? 2 * kBM : kBM, BN, kAMN, kBMN);
  static_assert(BN == 128 || BN == 256, "tile N");
  static_assert(!PAIR || (!kHasLsu && A_SRC != SRC_K_GATHER && A_SRC != SRC_MN_GATHER && B_SRC != SRC_MN_GATHER),
                "CTA pairs take TMA tiles only");
  static_assert(!PAIR || BN == 256, "CTA pairs split a 256-wide B tile");
  static_assert(!(kALsu && kBLsu), "one gathered operand per GEMM");
  static_assert(EPI != EPI_SWIGLU_MX, "the MXFP8 SwiGLU epilogue runs in gemm_mx_kernel");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Bounded wait that ignores the abort flag (used while draining in-flight work).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// Token of the K-row that lane `lane` of gather warp `gw` fetches for the
// shuffles of an MN-major gather (rows k0 .. k0+63 of the item's K range).
template <int B_SRC, int BN>
__device__ __forceinline__ int mn_gather_token(const GemmParams& p, const Item& it, int kb, int gw, int lane) {
  if (lane >= 16) return -1;
  int r;
  if (B_SRC == SRC_MN_GATHER_LSU && BN == 256)
    r = lane * 4 + gw;                              // rows i*4 + gw, i = 0..15
  else
    r = (lane >> 1) * 8 + gw * 2 + (lane & 1);      // rows i*8 + gw*2 + h, i = 0..7, h = 0..1
  return token_or_pad(p, it.kbeg + kb * kBK + r);
}

// One MN-major gathered chunk set: 64 K-rows x (64 * nchunk) elements; each
// K-row is a contiguous run of the token's row at column col0.
template <int NCHUNK>
__device__ __forceinline__ void gather_mn(uint8_t* dst, const uint16_t* src, long long ld, int col0, int tok_reg,
                                          int gw, int lane) {
  if (NCHUNK == 4) {  // 32 pieces of 16 B per K-row: one K-row per warp per step
    const int cc = lane >> 3, q = lane & 7;
    const uint16_t* base = src + col0 + cc * 64 + q * 8;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = i * 4 + gw;
      const int tok = __shfl_sync(0xffffffffu, tok_reg, i);
      cp_async16(dst + cc * kChunkBytes + r * 128 + ((q ^ (r & 7)) << 4),
                 base + static_cast<long long>(tok < 0 ? 0 : tok) * ld, tok >= 0 ? 16u : 0u);
    }
  } else {            // 16 pieces per K-row: two K-rows per warp per step
    const int piece = lane & 15, cc = piece >> 3, q = piece & 7;
    const uint16_t* base = src + col0 + cc * 64 + q * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = i * 8 + gw * 2 + (lane >> 4);
      const int tok = __shfl_sync(0xffffffffu, tok_reg, i * 2 + (lane >> 4));
      cp_async16(dst + cc * kChunkBytes + r * 128 + ((q ^ (r & 7)) << 4),
                 base + static_cast<long long>(tok < 0 ? 0 : tok) * ld, tok >= 0 ? 16u : 0u);
    }
  }
}

template <int A_SRC, int B_SRC, int BN, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(GemmCfg<A_SRC, B_SRC, BN, EPI, PAIR>::kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using C = GemmCfg<A_SRC, B_SRC, BN, EPI, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = bars + 2 * C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* qfull = done + 2;            // item queue: one arrival, the producer's
  uint64_t* qempty = qfull + C::kQ;      // one arrival per consumer (the leader's counts both CTAs')
  int* qslot = reinterpret_cast<int*>(qempty + C::kQ);
  static_assert((2 * C::kStages + 7 + 2 * C::kQ) * 8 + 4 * C::kQ <= C::kBarBytes, "barrier region");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pair: rank in the pair, persistent loop over the pair's items
  const int rank = PAIR ? static_cast<int>(cluster_rank()) : 0;
  const int item0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int istep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto item_at = [&](int idx, int bk) { return PAIR ? get_item_pair(p, idx, bk, rank) : get_item(p, idx, bk); };
  // Work items come in a static order (item0, item0 + istep, ...), or, with a
  // ticket counter, in ticket order: the leader's producer takes the next
  // ticket as it starts an item, so that all CTAs work on neighbouring items
  // and the operands they share stay in L2 (a static order lets the CTAs
  // drift apart over a long launch).  It hands each item to the other roles
  // (and the peer CTA) through the queue; -1 ends the sequence, -2 reports an
  // aborted wait.  The debug signal drop keeps the static order.
  const bool dyn = C::kDyn && p.ticket != nullptr && !(p.debug & 1);
  auto queue_put = [&](int k, int idx) -> bool {   // the leader's producer, one lane
    const int s = k % C::kQ;
    if (!mbar_wait<PAIR>(&qempty[s], ((k / C::kQ) & 1) ^ 1, abort_flag, p.status)) return false;
    qslot[s] = idx;
    if (PAIR) st_shared_cluster(cluster_addr(&qslot[s], 1), idx);
    mbar_arrive(&qfull[s]);
    if (PAIR) mbar_arrive_cluster(cluster_addr(&qfull[s], 1));
    return true;
  };
  auto queue_take = [&](int k) -> int {   // every other role, one lane
    const int s = k % C::kQ;
    // acquire at cluster scope only where the slot was written by the other
    // CTA (the leader's own roles read what their producer wrote)
    const bool ok = (PAIR && rank != 0) ? mbar_wait<true>(&qfull[s], (k / C::kQ) & 1, abort_flag, p.status)
                                        : mbar_wait<false>(&qfull[s], (k / C::kQ) & 1, abort_flag, p.status);
    if (!ok) return -2;
    const int idx = *reinterpret_cast<volatile int*>(&qslot[s]);
    if (PAIR && rank != 0)
      mbar_arrive_cluster(cluster_addr(&qempty[s], 0));
    else
      mbar_arrive(&qempty[s]);
    return idx;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], C::kFullArrivals);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (PAIR ? 2 : 1) * C::kEpiWarps);   // the leader's counts both CTAs' warps
    }
    for (int s = 0; s < C::kQ; ++s) {
      mbar_init(&qfull[s], 1);
      // the MMA issuer and the epilogue warps; a pair's leader also counts the
      // peer's producer and epilogue warps
      mbar_init(&qempty[s], PAIR ? 2 + 2 * C::kEpiWarps : 1 + C::kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b0);
    tma_prefetch_desc(&maps.b1);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();   // both CTAs' barriers initialised before any cross-CTA signal
  else
    __syncthreads();
  tc_fence_after();
  // everything above touches only on-chip state; the inputs below may come
  // from the kernel launched just before this one
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem_base = *tmem_slot;
  const int nitems = PAIR ? num_items_pair(p) : num_items(p);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    long long fills = 0;
    bool ok = true;
    const bool lead = !PAIR || rank == 0;
    // the leader publishes items kAhead ahead of the one it loads, so that the
    // other roles (and the peer's producer) find the next item waiting; its
    // next ticket is taken as soon as one is published
    constexpr int kAhead = 2;
    static_assert(kAhead < C::kQ, "a published slot is read back before it is reused");
    int ticket = 0, pub = 0;
    bool pub_end = false;
    if (dyn && lane == 0 && lead) ticket = atomicAdd(p.ticket, 1);
    for (int k = 0, sidx = item0;; ++k, sidx += istep) {
      int idx = sidx;
      if (dyn) {
        int v = 0;
        if (lane == 0) {
          if (lead) {
            bool put = true;
            while (put && !pub_end && pub <= k + kAhead) {
              const int pv = ticket < nitems ? ticket : -1;
              put = queue_put(pub, pv);
              if (!put) break;
              if (pv >= 0)
                ticket = atomicAdd(p.ticket, 1);
              else
                pub_end = true;
              ++pub;
            }
            v = put ? *reinterpret_cast<volatile int*>(&qslot[k % C::kQ]) : -2;
          } else {
            v = queue_take(k);
          }
        }
        idx = __shfl_sync(0xffffffffu, v, 0);
        if (idx == -2) ok = false;
        if (idx < 0) break;
      } else if (idx >= nitems) {
        break;
      }
      const Item it = item_at(idx, C::kBK);
      const int bn_out = (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_MX) ? BN / 2 : BN;
      const int n0 = it.nt * bn_out;
      // token rows of a row tile (K-major gather): rows 4*lane .. 4*lane+3
      int tok[4] = {0, 0, 0, 0};
      if (A_SRC == SRC_K_GATHER) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * lane + i;
          tok[i] = (r < it.rows) ? token_of(p, it.p0 + r) : 0;
        }
      }
      // token rows of the first K-block (MN-major gather along K)
      int ktok[4] = {0, 0, 0, 0};
      const bool mn_gather = (A_SRC == SRC_MN_GATHER || B_SRC == SRC_MN_GATHER);
      if (mn_gather && it.nk > 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ktok[i] = token_of(p, it.kbeg + 4 * (lane & 15) + i);
      }
      for (int kb = 0; kb < it.nk; ++kb) {
        int cur[4] = {ktok[0], ktok[1], ktok[2], ktok[3]};
        int w = (lane == 0) ? (mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status) ? 1 : 0) : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        // CTA pair: both CTAs' loads complete on the leader's barrier
        if (lane == 0 && (!PAIR || rank == 0)) mbar_arrive_expect_tx(&full[stage], (PAIR ? 2 : 1) * C::kTmaBytes);
        __syncwarp();
        uint8_t* sA = smem + stage * C::kStageBytes;
        uint8_t* sB = sA + C::kABytes;
        const int k0 = kb * C::kBK;
        const uint32_t lead_full = PAIR ? cluster_addr(&full[stage], 0) : 0u;
        auto ld2 = [&](void* dst, const CUtensorMap* m, int c0, int c1) {
          if (PAIR)
            tma_load_2d_pair(dst, m, lead_full, c0, c1);
          else
            tma_load_2d(dst, m, &full[stage], c0, c1);
        };
        auto ld3 = [&](void* dst, const CUtensorMap* m, int c0, int c1, int c2) {
          if (PAIR)
            tma_load_3d_pair(dst, m, lead_full, c0, c1, c2);
          else
            tma_load_3d(dst, m, &full[stage], c0, c1, c2);
        };
        // ---- A operand
        if (A_SRC == SRC_K_TILE) {
          if (lane == 0) ld2(sA, &maps.a, k0, it.p0);
        } else if (A_SRC == SRC_K_GATHER) {
          tma_gather4(sA + lane * 512, &maps.a, &full[stage], k0, tok[0], tok[1], tok[2], tok[3]);
        } else if (A_SRC == SRC_MN_TILE) {
          // one 3-D box {64 elements, 64 K-rows, 2 chunks}: chunk-major in smem
          if (lane == 0) ld3(sA, &maps.a, 0, it.kbeg + k0, it.m0 / C::kBK);
        } else if (A_SRC == SRC_MN_GATHER) {
          const int c = lane >> 4, g = lane & 15;
          tma_gather4(sA + c * kChunkBytes + g * 512, &maps.a, &full[stage], it.m0 + 64 * c, cur[0],
                      cur[1], cur[2], cur[3]);
        }
        // ---- B operand
        if (B_SRC == SRC_K_TILE) {
          if (lane == 0) {
            if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_MX) {
              // gate rows then up rows; a CTA pair splits them between its CTAs
              const int r = it.e * p.b_rows_per_expert + n0;
              if (!PAIR || rank == 0) ld2(sB, &maps.b0, k0, r);
              if (!PAIR || rank == 1) ld2(PAIR ? sB : sB + (BN / 2) * C::kRowBytes, &maps.b1, k0, r);
            } else {   // BN rows (one half per CTA of a pair)
              ld2(sB, &maps.b0, k0, it.e * p.b_rows_per_expert + n0 + rank * C::kBRows);
            }
          }
        } else if (B_SRC == SRC_MN_TILE) {
          if (lane == 0) {  // one 3-D box {64 elements, 64 K-rows, kBRows/64 chunks}
            int krow = k0;
            const CUtensorMap* m = &maps.b0;
            if (p.b_split > 0 && krow >= p.b_split) {
              m = &maps.b1;
              krow -= p.b_split;
            }
            const int kr = p.wgrad ? (it.kbeg + k0) : (it.e * p.b_rows_per_expert + krow);
            ld3(sB, m, 0, kr, (n0 + rank * C::kBRows) / C::kBK);
          }
        } else if (B_SRC == SRC_MN_GATHER) {
          const int g = lane & 15;
#pragma unroll
          for (int cc = 0; cc < BN / 128; ++cc) {
            const int c = (lane >> 4) + 2 * cc;
            tma_gather4(sB + c * kChunkBytes + g * 512, &maps.b0, &full[stage], n0 + 64 * c,
                        cur[0], cur[1], cur[2], cur[3]);
          }
        }
        ++fills;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        // prefetch the next K-block's token rows (latency hidden by the next wait)
        if (mn_gather && kb + 1 < it.nk) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ktok[i] = token_of(p, it.kbeg + (kb + 1) * kBK + 4 * (lane & 15) + i);
        }
      }
      if (!ok) break;
    }
    if (!ok && lane == 0 && (!PAIR || rank == 0)) {
      // drain: wait until every load issued into a stage has landed (a CTA
      // pair's loads all complete on the leader's barriers)
      const long long n = fills < C::kStages ? fills : C::kStages;
      int s = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < n; ++i) {
        if (--s < 0) {
          s = C::kStages - 1;
          ph ^= 1;
        }
        mbar_drain(&full[s], ph);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {   // a CTA pair's leader issues for both
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool first = true;
      for (int k = 0, sidx = item0;; ++k, sidx += istep) {
        int idx = sidx;
        if (dyn) {
          idx = queue_take(k);
          if (idx < 0) break;
        } else if (idx >= nitems) {
          break;
        }
        const int nk = item_nk(p, idx, C::kBK, PAIR);
        if (nk == 0) continue;
        if (!mbar_wait(&tempty[abuf], aphase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t acc = tmem_base + static_cast<uint32_t>(abuf * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          // gathered rows were written through the generic proxy (cp.async):
          // order them before the tensor core's async-proxy reads
          if (C::kHasLsu) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t b0 = a0 + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < C::kBK / 16; ++kk) {
            // K-major: 16 elements = 32 bytes along the swizzled row; MN-major: 16
            // K-rows; SBO = 8 rows, LBO (MN-major) = one chunk of kBK elements
            const uint64_t ad = C::kAMN ? smem_desc(a0 + kk * 16 * C::kRowBytes, C::kMnChunkBytes, 8 * C::kRowBytes, C::kSwz)
                                        : smem_desc(a0 + kk * 32, 16, 8 * C::kRowBytes, C::kSwz);
            const uint64_t bd = C::kBMN ? smem_desc(b0 + kk * 16 * C::kRowBytes, C::kMnChunkBytes, 8 * C::kRowBytes, C::kSwz)
                                        : smem_desc(b0 + kk * 32, 16, 8 * C::kRowBytes, C::kSwz);
            if (PAIR)
              umma_bf16_pair(acc, ad, bd, C::kIdesc, (kb | kk) ? 1u : 0u);
            else
              umma_bf16(acc, ad, bd, C::kIdesc, (kb | kk) ? 1u : 0u);
          }
          if (PAIR)
            umma_commit_pair(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        const bool drop = (p.debug & 1) && first && blockIdx.x == 0;
        if (!drop) {
          if (PAIR)
            umma_commit_pair(&tfull[abuf], 0x3);
          else
            umma_commit(&tfull[abuf]);
        }
        first = false;
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1;
        }
      }
      // every MMA issued by this thread must finish before TMEM is released
      if (PAIR)
        umma_commit_pair(done, 0x1);
      else
        umma_commit(done);
      mbar_drain(done, 0);
    }
  } else if (warp >= C::kGatherWarp0) {
    // ------------------------------------------------------------ gather warps
    if constexpr (C::kHasLsu) {
      const int gw = warp - C::kGatherWarp0;
      constexpr bool kMN = (A_SRC == SRC_MN_GATHER_LSU || B_SRC == SRC_MN_GATHER_LSU);
      const int bn_out = (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_MX) ? BN / 2 : BN;
      // token of tile row (lane>>2)*16 + gw*4 + (lane&3) for a K-major gather
      auto row_token = [&](const Item& t) {
        const int r = (lane >> 2) * 16 + gw * 4 + (lane & 3);
        return (r < t.rows) ? token_or_pad(p, t.p0 + r) : -1;
      };
      auto k_token = [&](const Item& t, int kb) {
        return (kb < t.nk) ? mn_gather_token<B_SRC, BN>(p, t, kb, gw, lane) : -1;
      };
      int stage = 0;
      uint32_t phase = 0;
      int idx = blockIdx.x;
      Item it{};
      int rtok = -1, kt0 = -1, kt1 = -1, kt2 = -1;  // current item's tokens (K-blocks kb..kb+2)
      if (idx < nitems) {
        it = get_item(p, idx, C::kBK);
        if (A_SRC == SRC_K_GATHER_LSU) rtok = row_token(it);
        if (kMN) {
          kt0 = k_token(it, 0);
          kt1 = k_token(it, 1);
          kt2 = k_token(it, 2);
        }
      }
      bool ok = true;
      while (idx < nitems && ok) {
        // the next item's descriptor and first tokens load while this one runs
        const int nidx = idx + gridDim.x;
        const bool has_next = nidx < nitems;
        Item nit{};
        if (has_next) nit = get_item(p, nidx, C::kBK);
        int nrtok = -1, nkt0 = -1, nkt1 = -1, nkt2 = -1;
        auto fetch_next = [&]() {
          if (!has_next) return;
          if (A_SRC == SRC_K_GATHER_LSU) nrtok = row_token(nit);
          if (kMN) {
            nkt0 = k_token(nit, 0);
            nkt1 = k_token(nit, 1);
            nkt2 = k_token(nit, 2);
          }
        };
        const int n0 = it.nt * bn_out;
        for (int kb = 0; kb < it.nk; ++kb) {
          const int cur = kt0;
          kt0 = kt1;
          kt1 = kt2;
          if (kMN) kt2 = k_token(it, kb + 3);   // three K-blocks ahead
          if (kb == it.nk - 1) fetch_next();
          int w = (lane == 0) ? (mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status) ? 1 : 0) : 0;
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + C::kABytes;
          const int k0 = kb * C::kBK;
          if (A_SRC == SRC_K_GATHER_LSU) {
            const int c = lane & 7;
            const uint16_t* base = p.ga + k0 + c * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = i * 16 + gw * 4 + (lane >> 3);
              const int tok = __shfl_sync(0xffffffffu, rtok, i * 4 + (lane >> 3));
              cp_async16(sA + row * 128 + ((c ^ (row & 7)) << 4),
                         base + static_cast<long long>(tok < 0 ? 0 : tok) * p.ga_ld, tok >= 0 ? 16u : 0u);
            }
          } else if (A_SRC == SRC_MN_GATHER_LSU) {
            gather_mn<2>(sA, p.ga, p.ga_ld, it.m0, cur, gw, lane);
          }
          if (B_SRC == SRC_MN_GATHER_LSU) gather_mn<BN / 64>(sB, p.gb, p.gb_ld, n0, cur, gw, lane);
          // the stage's full barrier completes when every thread's copies have landed
          cp_async_mbar_arrive_noinc(&full[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (it.nk == 0) fetch_next();
        idx = nidx;
        it = nit;
        rtok = nrtok;
        kt0 = nkt0;
        kt1 = nkt1;
        kt2 = nkt2;
      }
      // no copy may still be in flight when the CTA exits
      cp_async_wait_all();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;    // tile row of this thread
    uint8_t* wstage = smem + C::kStages * C::kStageBytes + C::kBarBytes + (warp - 2) * C::kEpiStageBytes;
    int tslot = 0;   // half of wstage the next TMA store stages into
    int abuf = 0;
    uint32_t aphase = 0;
    // weight gradients: the tensor map and row coordinate of a 32-row block
    // (row m of expert e: rows below `split` go to out0, the rest to out1)
    auto wgrad_dst = [&](const Item& t, int mblock, const CUtensorMap*& map, int& row) {
      if (mblock < p.split) {
        map = &maps.o0;
        row = t.e * p.split + mblock;
      } else {
        map = &maps.o1;
        row = t.e * (p.m_tiles * kBM - p.split) + (mblock - p.split);
      }
    };
    for (int k = 0, sidx = item0;; ++k, sidx += istep) {
      int idx = sidx;
      if (dyn) {
        int v = 0;
        if (lane == 0) v = queue_take(k);
        idx = __shfl_sync(0xffffffffu, v, 0);
        if (idx < 0) break;
      } else if (idx >= nitems) {
        break;
      }
      const Item it = item_at(idx, C::kBK);
      const int bn_out = (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_MX) ? BN / 2 : BN;
      const int n0 = it.nt * bn_out;
      const bool live = !it.empty;   // an empty half of a CTA pair stores nothing
      // this warp's 32-column chunks: all of them, or one half when two warps
      // share a lane quarter
      constexpr int kChunks = BN / 32;
      const int epi_half = (warp - 2) >> 2;
      const int epi_c0 = (C::kEpiWarps == 8) ? epi_half * (kChunks / 2) : 0;
      const int epi_c1 = (C::kEpiWarps == 8) ? epi_c0 + kChunks / 2 : kChunks;
      if (it.nk == 0) {
        // weight gradient of an expert with no rows: zeros
        if (EPI == EPI_WGRAD && live) {
          const CUtensorMap* omap;
          int orow;
          wgrad_dst(it, it.m0 + q * 32, omap, orow);
          uint32_t zw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) zw[i] = 0u;
          for (int c = epi_c0; c < epi_c1; ++c) warp_store_tma(zw, omap, n0 + c * 32, orow, wstage, tslot, lane);
        }
        continue;
      }
      // SwiGLU backward: row state and the first chunk of the saved gate|up,
      // fetched before the accumulator is ready
      int f_bwd = -1;
      bool v_bwd = false;
      float wt_bwd = 1.f;
      uint4 ng[4], nu[4];
      if constexpr (EPI == EPI_DOWN_BWD) {
        const int prow = it.p0 + r;
        if (p.grouped) {
          f_bwd = (live && r < it.rows) ? __ldg(p.row_src + prow) : -1;
          v_bwd = f_bwd >= 0;
          if (v_bwd) wt_bwd = __ldg(p.rw + f_bwd);
        } else {
          v_bwd = live && r < it.rows;
        }
        if (v_bwd) {
          const uint16_t* gu = static_cast<const uint16_t*>(p.aux0) + static_cast<long long>(prow) * 2 * p.N + n0 +
                               epi_c0 * 32;
          // the rest of this row's gate|up for the tile (128-byte lines of two
          // 32-column chunks; the first line is loaded just below) into L2
          // while the accumulator fills, so that each chunk's loads hit L2
          for (int c = 2; c < epi_c1 - epi_c0; c += 2) {
            prefetch_l2(gu + c * 32);
            prefetch_l2(gu + p.N + c * 32);
          }
          load_raw64(gu, ng);
          load_raw64(gu + p.N, nu);
        }
      }
      int w = (lane == 0) ? (mbar_wait(&tfull[abuf], aphase, abort_flag, p.status) ? 1 : 0) : 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(abuf * BN) +
                          (static_cast<uint32_t>(q * 32) << 16);
      uint32_t wv[16];

      if constexpr (EPI == EPI_SWIGLU) {
        // G|U [rows][2N] and h [rows][N] (bf16), through the maps o0 and o1
        const bool valid = r < it.rows;
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          float g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + BN / 2 + c * 32, u);
          if (!valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = u[i] = 0.f;
          }
          float hv[32];
          const float lim = p.swiglu_limit;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float gc = g[i], uc = u[i];
            if (lim > 0.f) {   // clamped SwiGLU (G|U are saved unclamped for the backward)
              gc = fminf(gc, lim);
              uc = fminf(fmaxf(uc, -lim), lim);
            }
            const float sg = __fdividef(1.f, 1.f + __expf(-gc));
            hv[i] = gc * sg * uc;
          }
          // G|U and h by TMA (rows past a dense layer's end are clipped)
          const int orow = it.p0 + q * 32;
          pack_bf16x32(g, wv);
          if (live) warp_store_tma(wv, &maps.o0, n0 + c * 32, orow, wstage, tslot, lane);
          pack_bf16x32(u, wv);
          if (live) warp_store_tma(wv, &maps.o0, p.N + n0 + c * 32, orow, wstage, tslot, lane);
          pack_bf16x32(hv, wv);
          if (live) warp_store_tma(wv, &maps.o1, n0 + c * 32, orow, wstage, tslot, lane);
        }
      } else if constexpr (EPI == EPI_SCALE_ROWS) {
        // router-weighted rows in schedule order by TMA; the combine reads
        // them back per (token, k) through slot_row
        const int f = (live && r < it.rows) ? __ldg(p.row_src + it.p0 + r) : -1;
        const float wt = f >= 0 ? __ldg(p.rw + f) : 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= wt;
          pack_bf16x32(v, wv);
          if (live) warp_store_tma(wv, &maps.o0, n0 + c * 32, it.p0 + q * 32, wstage, tslot, lane);
        }
      } else if constexpr (EPI == EPI_STORE_ROWS) {
        // dense rows by TMA (rows past the layer's end are clipped)
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
          pack_bf16x32(v, wv);
          if (live) warp_store_tma(wv, &maps.o0, n0 + c * 32, it.p0 + q * 32, wstage, tslot, lane);
        }
      } else if constexpr (EPI == EPI_DOWN_BWD) {
        // out0 = dgu [rows][2N], out1 = hw [rows][N]; aux0 = gu [rows][2N]
        const int prow = it.p0 + r;
        const uint16_t* gu = static_cast<const uint16_t*>(p.aux0) + static_cast<long long>(prow) * 2 * p.N + n0;
        // router-weight partial sums, one per half of the tile's columns (the
        // same split whether one warp or two cover the row)
        float dpart = 0.f;
        const float lim = p.swiglu_limit;
        float* dwp = (p.grouped && v_bwd) ? p.dw_part + (static_cast<long long>(f_bwd) * p.n_tiles + it.nt) * 2
                                          : nullptr;
#pragma unroll 1
        for (int c = epi_c0; c < epi_c1; ++c) {
          if (C::kEpiWarps == 4 && c == kChunks / 2) {
            if (dwp) dwp[0] = dpart;
            dpart = 0.f;
          }
          uint32_t wdg[16], wdu[16], whv[16];
#pragma unroll
          for (int half = 0; half < 2; ++half) {   // 16 accumulator columns at a time
            float z[16];
            tmem_ld16(tb + c * 32 + half * 16, z);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              float a[2] = {0.f, 0.f}, b[2] = {0.f, 0.f}, hh[2] = {0.f, 0.f};
              if (v_bwd) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  const int e = half * 16 + i + t;
                  float g = bf16_at(ng, e), u = bf16_at(nu, e);
                  float mg = 1.f, mu = 1.f;   // the clamp's derivative (SwiGLU limit)
                  if (lim > 0.f) {
                    mg = (g <= lim) ? 1.f : 0.f;
                    mu = (fabsf(u) <= lim) ? 1.f : 0.f;
                    g = fminf(g, lim);
                    u = fminf(fmaxf(u, -lim), lim);
                  }
                  const float sg = __fdividef(1.f, 1.f + __expf(-g));
                  const float sl = g * sg;
                  const float h = sl * u;
                  dpart = fmaf(z[i + t], h, dpart);
                  const float dh = wt_bwd * z[i + t];
                  a[t] = dh * u * sg * (1.f + g * (1.f - sg)) * mg;
                  b[t] = dh * sl * mu;
                  hh[t] = wt_bwd * h;
                }
              }
              wdg[(half * 16 + i) >> 1] = pack_bf16(a[0], a[1]);
              wdu[(half * 16 + i) >> 1] = pack_bf16(b[0], b[1]);
              whv[(half * 16 + i) >> 1] = pack_bf16(hh[0], hh[1]);
            }
          }
          if (v_bwd && c + 1 < epi_c1) {   // next chunk's gate|up, in flight during the stores
            load_raw64(gu + (c + 1) * 32, ng);
            load_raw64(gu + p.N + (c + 1) * 32, nu);
          }
          if (live) {   // dG|dU and w h by TMA (dense rows past the end are clipped)
            const int orow = it.p0 + q * 32;
            warp_store_tma(wdg, &maps.o0, n0 + c * 32, orow, wstage, tslot, lane);
            warp_store_tma(wdu, &maps.o0, p.N + n0 + c * 32, orow, wstage, tslot, lane);
            warp_store_tma(whv, &maps.o1, n0 + c * 32, orow, wstage, tslot, lane);
          }
        }
        if (dwp) dwp[C::kEpiWarps == 8 ? epi_half : 1] = dpart;
      } else if constexpr (EPI == EPI_WGRAD) {
        const CUtensorMap* omap;
        int orow;
        wgrad_dst(it, it.m0 + q * 32, omap, orow);
#pragma unroll 1
        for (int c = epi_c0; c < epi_c1; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
          pack_bf16x32(v, wv);
          if (live) warp_store_tma(wv, omap, n0 + c * 32, orow, wstage, tslot, lane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // the accumulator buffer is free again (a pair: on the leader's barrier)
        if (PAIR && rank != 0)
          mbar_arrive_cluster(cluster_addr(&tempty[abuf], 0));
        else
          mbar_arrive(&tempty[abuf]);
      }
      if (++abuf == 2) {
        abuf = 0;
        aphase ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();   // this warp's TMA stores are complete before the CTA ends
  }

  tc_fence_before();
  if (PAIR)
    cluster_sync();   // the leader's MMAs into this CTA's TMEM are done before either frees it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace mok

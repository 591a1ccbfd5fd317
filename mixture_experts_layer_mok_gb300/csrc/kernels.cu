// Schedule builder, MXFP8 quantiser, and the fixed-order combine kernels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.cuh"
#include "internal.h"

namespace mok {

// ===========================================================================
// Schedule ("Mixture-of-Kittens: a deterministic MoE megakernel for NVL72
// racks", "The two API layers and the schedule object": routing decisions are
// materialised into a dispatch/combine plan before any compute kernel runs).
// Three launches: per-chunk histograms; one block scans them into per-expert
// counts, padded row offsets and the tile list; per-chunk stable scatter.
// Above kPrefixChunks chunks a fourth launch, one block per expert, turns the
// histograms into per-expert chunk offsets first.
// ===========================================================================

__global__ void sched_count_kernel(const int64_t* __restrict__ te, int n, int E,
                                   int* __restrict__ hist, int* __restrict__ header) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int sh_cnt[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) sh_cnt[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * kSchedChunk;
  const int end = min(n, base + kSchedChunk);
  bool bad = false;
  for (int i = base + threadIdx.x; i < end; i += blockDim.x) {
    const int64_t e = te[i];
    if (e < 0 || e >= E)
      bad = true;
    else
      atomicAdd(&sh_cnt[static_cast<int>(e)], 1);
  }
  if (bad) atomicCAS(&header[2], 0, 2 /* MOK_ERR_INDEX */);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[blockIdx.x * E + i] = sh_cnt[i];
}

// Exclusive scan over a 1024-thread block.
__device__ int block_exclusive_scan(int v, int* tmp /* >= 32 ints */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    tmp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0) ? tmp[warp - 1] : 0;
  *total = tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + x - v;
}

// Work-group entries of a run of `len` units (tiles or pairs) of one expert
// from unit `first`: groups of at most `cap` consecutive units, the run cut
// evenly; an entry packs the unit's position in its group (bits 0..7) and the
// group's length (bits 8..15).
__device__ void write_groups(int* g, int first, int len, int cap) {
  if (len <= 0) return;
  const int ng = (len + cap - 1) / cap, gsz = (len + ng - 1) / ng;
  for (int i = 0; i < len; ++i) {
    const int gj = i / gsz * gsz;
    g[first + i] = (i - gj) | (min(gsz, len - gj) << 8);
  }
}

// Large schedules: the per-expert chunk offsets, one block per expert.  Column
// e of hist [nchunks][E] becomes each chunk's exclusive offset within expert
// e, and cnt[e] its total; each thread takes a run of consecutive chunks.
__global__ void __launch_bounds__(256) sched_prefix_kernel(int E, int nchunks, int* __restrict__ hist,
                                                           int* __restrict__ cnt, const int* __restrict__ header) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int tmp[32];
  if (header[2] != 0) return;
  const int e = blockIdx.x;
  const int per = (nchunks + blockDim.x - 1) / blockDim.x;
  const int k0 = min(nchunks, static_cast<int>(threadIdx.x) * per), k1 = min(nchunks, k0 + per);
  int sum = 0;
  for (int k = k0; k < k1; ++k) sum += hist[static_cast<long long>(k) * E + e];
  int total;
  int run = block_exclusive_scan(sum, tmp, &total);
  for (int k = k0; k < k1; ++k) {
    const long long i = static_cast<long long>(k) * E + e;
    const int v = hist[i];
    hist[i] = run;
    run += v;
  }
  if (threadIdx.x == 0) cnt[e] = total;
}

// Chunk counts above which the per-expert offsets get their own launch.
constexpr int kPrefixChunks = 64;

__global__ void __launch_bounds__(1024) sched_scan_kernel(int n, int E, int nchunks, int cap_tiles,
                                                          int max_tiles, int* __restrict__ hist,
                                                          int* __restrict__ cnt, int* __restrict__ row0,
                                                          int* __restrict__ row_src,
                                                          int* __restrict__ tile_expert,
                                                          int* __restrict__ tile_row0,
                                                          int* __restrict__ tile_rows,
                                                          int* __restrict__ pair_tile,
                                                          int* __restrict__ unit_group,
                                                          int* __restrict__ header) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int tmp[32];
  const int e = threadIdx.x;  // E <= 1024: one thread per expert
  const long long max_rows = static_cast<long long>(max_tiles) * kTileRows;
  if (header[2] != 0) {
    if (threadIdx.x == 0) {
      header[0] = 0;
      header[1] = 0;
      header[3] = 0;
      header[4] = 0;
      header[5] = cap_tiles;
    }
    return;
  }
  // each chunk's count becomes its exclusive offset within its expert (done
  // already by sched_prefix_kernel for more than kPrefixChunks chunks).  The
  // chunks are split over `tpe` threads per expert (all 1024 threads when E
  // is small): each sums its run of chunks, the runs' sums are scanned in
  // shared memory, and each thread rewrites its run from its base, sixteen
  // loads in flight per round.
  const bool prefixed = nchunks > kPrefixChunks;
  __shared__ int part[1024];
  int tpe = 1;
  while (tpe * 2 * E <= 1024) tpe *= 2;
  const int ee = threadIdx.x / tpe, sub = threadIdx.x % tpe;
  const int per = (nchunks + tpe - 1) / tpe;
  const int k0 = min(nchunks, sub * per), k1 = min(nchunks, k0 + per);
  int sum = 0;
  if (ee < E && !prefixed) {
    int k = k0;
    for (; k + 16 <= k1; k += 16) {
      int v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = hist[(k + q) * E + ee];
#pragma unroll
      for (int q = 0; q < 16; ++q) sum += v[q];
    }
    for (; k < k1; ++k) sum += hist[k * E + ee];
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  if (ee < E && !prefixed) {
    int run = 0;
    for (int q = 0; q < sub; ++q) run += part[ee * tpe + q];
    int k = k0;
    for (; k + 16 <= k1; k += 16) {
      int v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = hist[(k + q) * E + ee];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        hist[(k + q) * E + ee] = run;
        run += v[q];
      }
    }
    for (; k < k1; ++k) {
      const int v = hist[k * E + ee];
      hist[k * E + ee] = run;
      run += v;
    }
  }
  __syncthreads();
  int c = 0;
  if (e < E && prefixed) {
    c = cnt[e];
  } else if (e < E) {
    for (int q = 0; q < tpe; ++q) c += part[e * tpe + q];
    cnt[e] = c;
  }
  int total_rows;
  const int padded = (c + kTileRows - 1) / kTileRows * kTileRows;
  const int r0 = block_exclusive_scan(padded, tmp, &total_rows);
  if (e < E) row0[e] = r0;
  if (e == 0) row0[E] = total_rows;
  const int ntile = (c + kTileRows - 1) / kTileRows;
  const int prim = min(ntile, cap_tiles);
  int total_prim, total_ovf;
  const int prim_off = block_exclusive_scan(prim, tmp, &total_prim);
  const int ovf_off = block_exclusive_scan(ntile - prim, tmp, &total_ovf);
  if (e < E) {
    for (int i = 0; i < ntile; ++i) {
      const int idx = (i < prim) ? prim_off + i : total_prim + ovf_off + (i - prim);
      tile_expert[idx] = e;
      tile_row0[idx] = r0 + i * kTileRows;
      tile_rows[idx] = min(kTileRows, c - i * kTileRows);
    }
    for (int q = r0 + c; q < r0 + padded; ++q) row_src[q] = -1;
  }
  const int num_tiles = total_prim + total_ovf;
  // tile pairs for CTA-pair GEMMs: consecutive tiles of one expert within the
  // primary list, then within the overflow list; an odd tile pairs with none
  const int pp = (prim + 1) / 2, po = (ntile - prim + 1) / 2;
  int total_pp, total_po;
  const int pp_off = block_exclusive_scan(pp, tmp, &total_pp);
  const int po_off = block_exclusive_scan(po, tmp, &total_po);
  if (e < E) {
    for (int j = 0; j < pp; ++j) {
      pair_tile[2 * (pp_off + j)] = prim_off + 2 * j;
      pair_tile[2 * (pp_off + j) + 1] = (2 * j + 1 < prim) ? prim_off + 2 * j + 1 : -1;
    }
    const int no = ntile - prim;
    for (int j = 0; j < po; ++j) {
      pair_tile[2 * (total_pp + po_off + j)] = total_prim + ovf_off + 2 * j;
      pair_tile[2 * (total_pp + po_off + j) + 1] = (2 * j + 1 < no) ? total_prim + ovf_off + 2 * j + 1 : -1;
    }
    write_groups(unit_group, prim_off, prim, kGroupTiles);
    write_groups(unit_group, total_prim + ovf_off, no, kGroupTiles);
    write_groups(unit_group + max_tiles, pp_off, pp, kGroupPairs);
    write_groups(unit_group + max_tiles, total_pp + po_off, po, kGroupPairs);
  }
  const int num_pairs = total_pp + total_po;
  for (int i = num_pairs + threadIdx.x; i < max_tiles; i += blockDim.x) {
    pair_tile[2 * i] = -1;
    pair_tile[2 * i + 1] = -1;
    unit_group[max_tiles + i] = -1;
  }
  for (int i = num_tiles + threadIdx.x; i < max_tiles; i += blockDim.x) {
    tile_expert[i] = -1;
    tile_row0[i] = -1;
    tile_rows[i] = -1;
    unit_group[i] = -1;
  }
  for (long long q = total_rows + threadIdx.x; q < max_rows; q += blockDim.x) row_src[q] = -1;
  if (threadIdx.x == 0) {
    header[0] = num_tiles;
    header[1] = total_rows;
    header[3] = total_prim;
    header[4] = num_pairs;
    header[5] = cap_tiles;
  }
}

// Stable scatter: within a chunk, rows are placed in ascending flat index f.
// Each round of 256 consecutive f: rank within the warp from match_any, plus
// the counts of the same expert in lower warps of the round, plus the running
// offset of the expert.
__global__ void __launch_bounds__(256) sched_scatter_kernel(const int64_t* __restrict__ te, int n, int E,
                                                            const int* __restrict__ hist,
                                                            const int* __restrict__ row0,
                                                            int* __restrict__ row_src,
                                                            int* __restrict__ slot_row,
                                                            const int* __restrict__ header) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int sh[];
  int* run = sh;               // [E]
  int* wcnt = sh + E;          // [8][E]
  if (header[2] != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = row0[i] + hist[blockIdx.x * E + i];
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * kSchedChunk;
  const int end = min(n, base + kSchedChunk);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = base; r < end; r += 256) {
    const int f = r + threadIdx.x;
    const bool valid = f < end;
    const int e = valid ? static_cast<int>(te[f]) : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(m) - 1;
    const int rank = __popc(m & lt_mask);
    if (valid && lane == leader) wcnt[warp * E + e] = __popc(m);
    __syncthreads();
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += wcnt[w * E + e];
      const int pos = run[e] + before + rank;
      row_src[pos] = f;
      slot_row[f] = pos;
    }
    __syncthreads();
    if (valid && lane == leader) {
      atomicAdd(&run[e], __popc(m));
      wcnt[warp * E + e] = 0;
    }
    __syncthreads();
  }
}

cudaError_t launch_schedule(const int64_t* te, int T, int k, int E, int cap_tiles, int max_tiles,
                            int* hist, int* cnt, int* row0, int* row_src, int* slot_row,
                            int* tile_expert, int* tile_row0, int* tile_rows, int* pair_tile, int* unit_group,
                            int* header, cudaStream_t st) {
  const int n = T * k;
  const int nchunks = (n + kSchedChunk - 1) / kSchedChunk;
  cudaError_t err = cudaMemsetAsync(header, 0, 8 * sizeof(int), st);
  if (err != cudaSuccess) return err;
  err = launch_dependent(sched_count_kernel, dim3(nchunks), dim3(256), E * sizeof(int), st, te, n, E, hist, header);
  if (err != cudaSuccess) return err;
  if (nchunks > kPrefixChunks) {
    err = launch_dependent(sched_prefix_kernel, dim3(E), dim3(256), 0, st, E, nchunks, hist, cnt,
                           static_cast<const int*>(header));
    if (err != cudaSuccess) return err;
  }
  err = launch_dependent(sched_scan_kernel, dim3(1), dim3(1024), 0, st, n, E, nchunks, cap_tiles, max_tiles, hist, cnt,
                         row0, row_src, tile_expert, tile_row0, tile_rows, pair_tile, unit_group, header);
  if (err != cudaSuccess) return err;
  const size_t smem = 9 * E * sizeof(int);
  if (smem > 48 * 1024) {
    err = cudaFuncSetAttribute(sched_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  err = launch_dependent(sched_scatter_kernel, dim3(nchunks), dim3(256), smem, st, te, n, E,
                         static_cast<const int*>(hist), static_cast<const int*>(row0), row_src, slot_row,
                         static_cast<const int*>(header));
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// Macrobatch window view ("Mixture-of-Kittens: a deterministic MoE megakernel
// for NVL72 racks", "Tuning the five hyperparameters before production":
// macrobatch_size is the size of the token ring buffer).  The schedule
// restricted to experts [e0, e0 + ne), with rows counted from the window's
// first schedule row row0[e0]: its tile list in the schedule's own order
// (primary tiles, at most cap_tiles of each expert, then the overflow list),
// tile pairs, work groups (those of the tiles, then of the pairs),
// per-expert row offsets (ne + 1 entries) and header.  Tile
// experts stay absolute (they index the weights).  One 1024-thread block, one
// thread per expert of the window.
// ===========================================================================
__global__ void __launch_bounds__(1024) window_view_kernel(const int* __restrict__ cnt, const int* __restrict__ row0,
                                                           const int* __restrict__ header, int e0, int ne,
                                                           int* __restrict__ tile_expert, int* __restrict__ tile_row0,
                                                           int* __restrict__ tile_rows, int* __restrict__ pair_tile,
                                                           int* __restrict__ unit_group, int* __restrict__ wrow0,
                                                           int* __restrict__ wheader) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int tmp[32];
  if (header[2] != 0) {   // no schedule: an empty view that carries the status
    if (threadIdx.x < 8) wheader[threadIdx.x] = threadIdx.x == 2 ? header[2] : 0;
    return;
  }
  const int i = threadIdx.x, e = e0 + i;
  const int cap = header[5];
  const int base = row0[e0];
  const int c = i < ne ? cnt[e] : 0;
  const int ntile = (c + kTileRows - 1) / kTileRows;
  const int prim = min(ntile, cap);
  int total_prim, total_ovf, total_pp, total_po;
  const int prim_off = block_exclusive_scan(prim, tmp, &total_prim);
  const int ovf_off = block_exclusive_scan(ntile - prim, tmp, &total_ovf);
  const int pp = (prim + 1) / 2, po = (ntile - prim + 1) / 2;
  const int pp_off = block_exclusive_scan(pp, tmp, &total_pp);
  const int po_off = block_exclusive_scan(po, tmp, &total_po);
  if (i < ne) {
    const int r = row0[e] - base;
    wrow0[i] = r;
    for (int t = 0; t < ntile; ++t) {
      const int idx = (t < prim) ? prim_off + t : total_prim + ovf_off + (t - prim);
      tile_expert[idx] = e;
      tile_row0[idx] = r + t * kTileRows;
      tile_rows[idx] = min(kTileRows, c - t * kTileRows);
    }
    for (int j = 0; j < pp; ++j) {
      pair_tile[2 * (pp_off + j)] = prim_off + 2 * j;
      pair_tile[2 * (pp_off + j) + 1] = (2 * j + 1 < prim) ? prim_off + 2 * j + 1 : -1;
    }
    const int no = ntile - prim;
    for (int j = 0; j < po; ++j) {
      pair_tile[2 * (total_pp + po_off + j)] = total_prim + ovf_off + 2 * j;
      pair_tile[2 * (total_pp + po_off + j) + 1] = (2 * j + 1 < no) ? total_prim + ovf_off + 2 * j + 1 : -1;
    }
    const int tiles = total_prim + total_ovf;   // the window's pair groups follow its tile groups
    write_groups(unit_group, prim_off, prim, kGroupTiles);
    write_groups(unit_group, total_prim + ovf_off, no, kGroupTiles);
    write_groups(unit_group + tiles, pp_off, pp, kGroupPairs);
    write_groups(unit_group + tiles, total_pp + po_off, po, kGroupPairs);
  }
  if (i == 0) {
    const int rows = row0[e0 + ne] - base;
    wrow0[ne] = rows;
    wheader[0] = total_prim + total_ovf;
    wheader[1] = rows;
    wheader[2] = 0;
    wheader[3] = total_prim;
    wheader[4] = total_pp + total_po;
    wheader[5] = cap;
    wheader[6] = 0;
    wheader[7] = 0;
  }
}

cudaError_t launch_window_view(const int* cnt, const int* row0, const int* header, int e0, int ne, int* tile_expert,
                               int* tile_row0, int* tile_rows, int* pair_tile, int* unit_group, int* wrow0,
                               int* wheader, cudaStream_t st) {
  cudaError_t err = launch_dependent(window_view_kernel, dim3(1), dim3(1024), 0, st, cnt, row0, header, e0, ne,
                                     tile_expert, tile_row0, tile_rows, pair_tile, unit_group, wrow0, wheader);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// MXFP8 quantiser ("Mixture-of-Kittens: a deterministic MoE megakernel for
// NVL72 racks", "Tuning the five hyperparameters before production": MXFP8
// weights are prequantised by a separate mxfp8_quantize).  One thread per
// 1x32 block: 64 bytes in, 32 code bytes and one scale byte out.
// ===========================================================================
__global__ void __launch_bounds__(256) mx_quantize_kernel(const uint16_t* __restrict__ x, long long nblocks,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nblocks;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    float v[32];
    load_bf16x32(x + b * 32, v);
    scales[b] = static_cast<uint8_t>(mx_quantize32(v, codes + b * 32));
  }
}

static int grid_for(long long work, int per_block, int num_sms) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

cudaError_t launch_mx_quantize(const uint16_t* x, long long nblocks, uint8_t* codes, uint8_t* scales,
                               int num_sms, cudaStream_t st) {
  if (nblocks == 0) return cudaSuccess;
  cudaError_t err = launch_dependent(mx_quantize_kernel, dim3(grid_for(nblocks, 256, num_sms)), dim3(256), 0, st, x,
                                     nblocks, codes, scales);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// MXFP8 dispatch: every token row of x is quantised once (E4M3 codes + E8M0
// scales, OCP MX v1.0 blocks of 32) and written to its own row of the
// token-order copy (the shared expert's operand) and to the k schedule rows
// that route it (the routed experts' operand: MoK's dispatch exchange, done on
// one GPU as a write into schedule order).  Padding rows of the schedule get
// zero codes.  Only the schedule rows of the window [w0, w0 + wrows) are
// written, at row p - w0 (the whole schedule is the window [0, max_rows); a
// macrobatch ring passes one window of experts at a time), and the
// token-order copy only when xq is not NULL.  The scales go, with the
// token-order copy, to xs: row-major [T][H/32], every store a whole 32-byte
// sector; mx_scale_gather_kernel lays them out for the GEMMs.  (Stored from
// here into the tensor-core layout, each 4-byte scale word would share its
// sector with seven rows of other tokens written at other times, and every
// partly written sector that L2 evicts costs a read-modify-write.)  One warp
// per job: tokens, then the window's schedule rows.
// ===========================================================================
__global__ void __launch_bounds__(256, 3) mx_dispatch_kernel(
    const uint16_t* __restrict__ x, int T, int H, int topk, const int* __restrict__ slot_row,
    const int* __restrict__ row_src, const int* __restrict__ header, long long w0, long long wrows,
    uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, uint8_t* __restrict__ xp, uint16_t* __restrict__ xb) {
  griddep_wait();
  griddep_launch_dependents();
  if (header[2] != 0) return;
  // per warp: the codes of one 32-block chunk of a row (1 KB) and, when the
  // bf16 rows are wanted too, its bf16 values (2 KB), so that every store
  // instruction of the copies writes 512 contiguous bytes
  __shared__ __align__(16) uint8_t stage[8][1024];
  __shared__ __align__(16) uint8_t stage_b[8][2048];
  uint8_t* wst = stage[threadIdx.x >> 5];
  uint4* wsb = reinterpret_cast<uint4*>(stage_b[threadIdx.x >> 5]);
  const long long P = header[1];
  const int lane = threadIdx.x & 31;
  const int nb = H / 32;             // blocks per row (a multiple of 4)
  const long long jobs = T + wrows;
  for (long long j = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; j < jobs;
       j += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    if (j < T) {
      const long long t = j;
      // schedule rows of this token's k copies, spread over the lanes
      const int p_lo = lane < topk ? __ldg(slot_row + t * topk + lane) : -1;
      const int p_hi = lane + 32 < topk ? __ldg(slot_row + t * topk + lane + 32) : -1;
      // without the token-order copy, a token none of whose rows falls in the
      // window is not read at all
      if (!xq && !__any_sync(0xffffffffu, (p_lo >= w0 && p_lo - w0 < wrows) || (p_hi >= w0 && p_hi - w0 < wrows)))
        continue;
      const uint16_t* xrow = x + t * H;
      // raw bf16 of this lane's block in the current chunk, the next chunk's
      // loaded while this one is quantised and stored
      uint4 raw[4];
      if (lane < nb) load_raw64(xrow + lane * 32, raw);
      for (int b0 = 0; b0 < nb; b0 += 32) {
        const int b = b0 + lane;
        const bool act = b < nb;       // whole aligned groups of 4 lanes share this
        float v[32];
        uint4 vraw[4] = {raw[0], raw[1], raw[2], raw[3]};
        if (act) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = bf16_at(vraw, i);
        }
        if (b0 + 32 + lane < nb) load_raw64(xrow + (b0 + 32 + lane) * 32, raw);
        uint8_t codes[32];
        uint32_t sc = 127;
        if (act) sc = mx_quantize32(v, codes);
        if (act) {
          uint4* sw = reinterpret_cast<uint4*>(wst + lane * 32);
          sw[0] = reinterpret_cast<const uint4*>(codes)[0];
          sw[1] = reinterpret_cast<const uint4*>(codes)[1];
          if (xb) {   // this lane's 64 bf16 bytes, pieces swizzled against bank conflicts
#pragma unroll
            for (int q = 0; q < 4; ++q) wsb[lane * 4 + (q ^ (lane & 3))] = vraw[q];
          }
        }
        __syncwarp();
        // this chunk's bytes [32 * b0, 32 * min(nb, b0 + 32)) of each copy's row:
        // lane l stores the 16-byte pieces l and l + 32
        const int bytes = 32 * (min(nb, b0 + 32) - b0);
        const uint4 q0 = 16 * lane < bytes ? reinterpret_cast<const uint4*>(wst)[lane] : make_uint4(0, 0, 0, 0);
        const uint4 q1 = 16 * (lane + 32) < bytes ? reinterpret_cast<const uint4*>(wst)[lane + 32] : q0;
        __syncwarp();
        const long long off = static_cast<long long>(b0) * 32;
        if (xq) {
          uint4* d = reinterpret_cast<uint4*>(xq + t * H + off);
          if (16 * lane < bytes) d[lane] = q0;
          if (16 * (lane + 32) < bytes) d[lane + 32] = q1;
          // the chunk's scale bytes, 4 per word from every fourth lane: one
          // store of up to 32 contiguous bytes
          const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 1);
          const uint32_t s2 = __shfl_down_sync(0xffffffffu, sc, 2);
          const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 3);
          if (act && (lane & 3) == 0)
            *reinterpret_cast<uint32_t*>(xs + t * nb + b) = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
        for (int jj = 0; jj < topk; ++jj) {   // all lanes take part in the shuffle
          const long long pr = __shfl_sync(0xffffffffu, jj < 32 ? p_lo : p_hi, jj & 31) - w0;
          if (pr < 0 || pr >= wrows) continue;   // the same for every lane
          uint4* dp = reinterpret_cast<uint4*>(xp + static_cast<long long>(pr) * H + off);
          if (16 * lane < bytes) dp[lane] = q0;
          if (16 * (lane + 32) < bytes) dp[lane + 32] = q1;
          if (xb) {   // the chunk's bf16 bytes: its piece i (16 bytes) is piece
                      // (i % 4) ^ ((i / 4) % 4) of block i / 4 in the staging layout
            uint4* db = reinterpret_cast<uint4*>(xb + static_cast<long long>(pr) * H + off);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = lane + 32 * q, blk = i >> 2;
              if (16 * i < 2 * bytes) db[i] = wsb[blk * 4 + ((i & 3) ^ (blk & 3))];
            }
          }
        }
        __syncwarp();   // the staging is read before the next chunk overwrites it
      }
    } else {
      const long long pr = j - T;
      if (w0 + pr >= P || __ldg(row_src + w0 + pr) >= 0) continue;
      uint4* d = reinterpret_cast<uint4*>(xp + pr * H);
      for (int i = lane; i < H / 16; i += 32) d[i] = make_uint4(0, 0, 0, 0);
      if (xb) {
        uint4* db = reinterpret_cast<uint4*>(xb + pr * H);
        for (int i = lane; i < H / 8; i += 32) db[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

cudaError_t launch_mx_dispatch(const uint16_t* x, int T, int H, int topk, const int* slot_row, const int* row_src,
                               const int* header, long long w0, long long wrows, uint8_t* xq, uint8_t* xs,
                               uint8_t* xp, uint16_t* xb, int num_sms, cudaStream_t st) {
  const long long jobs = T + wrows;
  cudaError_t err = launch_dependent(mx_dispatch_kernel, dim3(grid_for(jobs * 32, 256, num_sms)), dim3(256), 0, st, x,
                                     T, H, topk, slot_row, row_src, header, w0, wrows, xq, xs, xp, xb);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// The dispatch's scales, row-major by token (xs [T][H/32]), into the
// tensor-core scale layout (mx_tiled_scale_offset): for the window's schedule
// rows [w0, w0 + wrows) at rows from 0 of xp_sc (a row takes its token's
// scales; padding rows and rows from P on unit scales), and, when xq_sc is not
// NULL, for token order (rows from T on: unit scales).  One block of 128
// threads per 128-row block, 32 column groups (one 128-byte piece of each
// source row) per pass: warp w reads rows 32 w .. 32 w + 31, one whole piece
// per load, into a shared-memory tile of the pass's 512-byte atoms (stride
// 129 words: no bank conflicts), and the block then stores the atoms whole.
// ===========================================================================
__global__ void __launch_bounds__(128) mx_scale_gather_kernel(const uint8_t* __restrict__ xs, int T, int nb, int topk,
                                                              const int* __restrict__ row_src,
                                                              const int* __restrict__ header, long long w0,
                                                              long long wrows, uint8_t* __restrict__ xp_sc,
                                                              uint8_t* __restrict__ xq_sc) {
  griddep_wait();
  griddep_launch_dependents();
  if (header[2] != 0) return;
  constexpr int kChunk = 32;                    // column groups (scale words of a row) per pass
  constexpr int kStride = 129;                  // words per atom in shared memory
  __shared__ uint32_t sw[kChunk * kStride];
  const long long P = header[1];
  const int cg = nb / 4;
  const long long sgroups = wrows / 128;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long g = blockIdx.x;
  long long src = -1;                           // the token of row 32 warp + lane
  uint32_t* out;
  if (g < sgroups) {
    const long long p = w0 + 128 * g + 32 * warp + lane;
    const int rs = p < P ? __ldg(row_src + p) : -1;
    if (rs >= 0) src = rs / topk;
    out = reinterpret_cast<uint32_t*>(xp_sc);
  } else {
    g -= sgroups;
    const long long t = 128 * g + 32 * warp + lane;
    if (t < T) src = t;
    out = reinterpret_cast<uint32_t*>(xq_sc);
  }
  out += g * cg * 128;
  const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs);
  const int words = nb / 4;                     // scale words per source row
  for (int c0 = 0; c0 < cg; c0 += kChunk) {
    const int nc = min(kChunk, cg - c0);
    uint32_t v[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) {              // row 32 warp + l: lane c loads its word c0 + c
      const long long sl = __shfl_sync(0xffffffffu, src, l);
      v[l] = (sl >= 0 && lane < nc) ? __ldg(xw + sl * words + c0 + lane) : 0x7F7F7F7Fu;
    }
    // row r sits at word (r % 32) * 4 + r / 32 of its atom
#pragma unroll
    for (int l = 0; l < 32; ++l)
      if (lane < nc) sw[lane * kStride + l * 4 + warp] = v[l];
    __syncthreads();
    for (int c = 0; c < nc; ++c) out[static_cast<long long>(c0 + c) * 128 + threadIdx.x] = sw[c * kStride + threadIdx.x];
    __syncthreads();
  }
}

cudaError_t launch_mx_scale_gather(const uint8_t* xs, int T, int H, int topk, const int* row_src, const int* header,
                                   long long w0, long long wrows, uint8_t* xp_sc, uint8_t* xq_sc, cudaStream_t st) {
  const long long blocks = wrows / 128 + (xq_sc ? (static_cast<long long>(T) + 127) / 128 : 0);
  if (blocks == 0) return cudaSuccess;
  cudaError_t err = launch_dependent(mx_scale_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, st, xs,
                                     T, H / 32, topk, row_src, header, w0, wrows, xp_sc, xq_sc);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// Transposing MXFP8 quantiser: bf16 rows -> E4M3 codes of the transpose, one
// E8M0 scale per 32 consecutive input rows of each column.  This is the
// operand form of a GEMM whose contraction runs along the rows: the weight
// gradients (contraction over an expert's rows) and the dgrad GEMMs (over a
// weight's leading axis).  Input row r of batch b is src[b][r] (dense; zero
// from valid_rows on), or, with row_src, the token row of schedule row r
// (src[row_src[r] / topk]; zero for padding rows).  With a schedule header,
// rows from P on read as zero and a failed schedule skips the work.  Output
// codes [batch][C][R]; scales row-major [batch*C][R/32], or (tiled) in the
// tensor-core scale layout with rows batch*C and K = R.  One block per
// 128-row x 64-column tile: coalesced row loads into shared memory (cp.async,
// the next tile's while this one is quantised), one thread per (column,
// 32-row block) quantising into a shared-memory output tile, then whole
// 128-byte code rows and one 4-byte scale word per column out to global
// memory.  With rcodes, the same read also yields the codes
// along the rows (blocks of 32 columns, scales rscales, row-major or tiled):
// both orientations of one tensor from a single pass over it.
// ===========================================================================
__global__ void __launch_bounds__(256) mx_quantize_t_kernel(const uint16_t* __restrict__ src, long long ld, int batch,
                                                            int R, int C, int valid_rows,
                                                            const int* __restrict__ row_src, int topk,
                                                            const int* __restrict__ header,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales, int tiled,
                                                            uint8_t* __restrict__ rcodes,
                                                            uint8_t* __restrict__ rscales, int rtiled) {
  griddep_wait();
  griddep_launch_dependents();
  int vrows = valid_rows;
  if (header) {
    if (header[2] != 0) return;
    vrows = min(vrows, header[1]);
  }
  constexpr int kOutStride = 144;   // bytes per output row in shared memory (128 + 16: no bank conflicts)
  // two input tiles (the next one loads by cp.async while this one is
  // quantised); row r's 16-byte piece p sits at piece p ^ (r & 7), so that
  // both column reads (one element of 32 rows) and row reads (half a row per
  // thread) spread over the banks
  __shared__ __align__(16) uint16_t tile[2][128][64];
  __shared__ __align__(16) uint8_t out[64 * kOutStride];
  __shared__ uint32_t osc[64];
  const int rtiles = (R + 127) / 128, ctiles = C / 64;
  const int ntiles = batch * rtiles * ctiles;   // below 2^31 (the launch checks)
  const int c = threadIdx.x & 63, rb = threadIdx.x >> 6;
  // tile t -> (batch b, first row r0, first column c0), in 32-bit arithmetic
  // and once per tile (the next tile's coordinates are kept for its turn)
  struct Coord {
    int b, r0, c0;
  };
  auto coords = [&](int t) {
    const int rest = t / ctiles;
    Coord x;
    x.c0 = (t - rest * ctiles) * 64;
    x.b = rest / rtiles;
    x.r0 = (rest - x.b * rtiles) * 128;
    return x;
  };
  auto issue = [&](const Coord& tc, int buf) {   // cp.async of the tile's rows (zeros past the valid rows)
    const int b = tc.b, r0 = tc.r0, c0 = tc.c0;
    // this thread copies piece (tid & 7) of rows (tid >> 3) + 32 j, j < 4: their
    // source rows first (independent index loads), then the four copies
    const int piece = threadIdx.x & 7;
    long long srow[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + (threadIdx.x >> 3) + 32 * j;
      srow[j] = (r < R && r < vrows) ? r : -1;
      if (row_src && srow[j] >= 0) {
        const int f = __ldg(row_src + r);
        srow[j] = f >= 0 ? f / topk : -1;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = (threadIdx.x >> 3) + 32 * j;
      const uint16_t* g =
          src + (static_cast<long long>(b) * R + (srow[j] >= 0 ? srow[j] : 0)) * ld + c0 + piece * 8;
      cp_async16(&tile[buf][row][(piece ^ (row & 7)) * 8], g, srow[j] >= 0 ? 16u : 0u);
    }
  };
  int buf = 0;
  Coord cur = {0, 0, 0};
  if (static_cast<int>(blockIdx.x) < ntiles) {
    cur = coords(blockIdx.x);
    issue(cur, 0);
  }
  cp_async_commit();
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int b = cur.b, r0 = cur.r0, c0 = cur.c0;
    if (t + static_cast<int>(gridDim.x) < ntiles) {
      cur = coords(t + gridDim.x);
      issue(cur, buf ^ 1);
    }
    cp_async_commit();
    cp_async_wait<1>();   // this tile's copies have landed (the next tile's may still fly)
    __syncthreads();
    {   // column c0 + c, rows r0 + 32 rb ..: codes into the output tile
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int row = rb * 32 + i;
        v[i] = __uint_as_float(static_cast<uint32_t>(tile[buf][row][(((c >> 3) ^ (row & 7)) << 3) | (c & 7)]) << 16);
      }
      uint8_t q[32];
      const uint32_t s = mx_quantize32(v, q);
      uint4* o = reinterpret_cast<uint4*>(out + c * kOutStride + rb * 32);
      o[0] = reinterpret_cast<const uint4*>(q)[0];
      o[1] = reinterpret_cast<const uint4*>(q)[1];
      reinterpret_cast<uint8_t*>(osc)[c * 4 + rb] = static_cast<uint8_t>(s);
    }
    if (rcodes) {   // row r0 + (tid >> 1), columns c0 + 32 (tid & 1) ..: a block along the row
      const int row = threadIdx.x >> 1, hb = threadIdx.x & 1;
      const long long orr = static_cast<long long>(b) * R + r0 + row;
      if (r0 + row < R) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = reinterpret_cast<const uint4*>(&tile[buf][row][0])[(hb * 4 + j) ^ (row & 7)];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * j + 2 * k] = __uint_as_float(ws[k] << 16);
            v[8 * j + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
          }
        }
        uint8_t q[32];
        const uint32_t s = mx_quantize32(v, q);
        uint4* d = reinterpret_cast<uint4*>(rcodes + orr * C + c0 + hb * 32);
        d[0] = reinterpret_cast<const uint4*>(q)[0];
        d[1] = reinterpret_cast<const uint4*>(q)[1];
        const int cb = (c0 >> 5) + hb;
        if (rtiled)
          rscales[mx_tiled_scale_offset(orr, cb, C / 128)] = static_cast<uint8_t>(s);
        else
          rscales[orr * (C / 32) + cb] = static_cast<uint8_t>(s);
      }
    }
    __syncthreads();   // the output tile is complete; the input buffer may be refilled
    const long long orow0 = static_cast<long long>(b) * C + c0;
    for (int i = threadIdx.x; i < 64 * 8; i += 256) {   // 8 pieces of 16 code bytes per output row
      const int row = i >> 3, piece = i & 7;
      if (r0 + piece * 16 < R)
        *reinterpret_cast<uint4*>(codes + (orow0 + row) * R + r0 + piece * 16) =
            *reinterpret_cast<const uint4*>(out + row * kOutStride + piece * 16);
    }
    if (threadIdx.x < 64) {   // the column's four block scales
      const long long orow = orow0 + threadIdx.x;
      const uint32_t word = osc[threadIdx.x];
      if (tiled) {
        *reinterpret_cast<uint32_t*>(scales + mx_tiled_scale_offset(orow, r0 / 32, R / 128)) = word;
      } else if ((R / 32) % 4 == 0 && (reinterpret_cast<uintptr_t>(scales) & 3u) == 0) {
        *reinterpret_cast<uint32_t*>(scales + orow * (R / 32) + r0 / 32) = word;
      } else {
        for (int k = 0; k < 4 && r0 + 32 * k < R; ++k)
          scales[orow * (R / 32) + r0 / 32 + k] = static_cast<uint8_t>(word >> (8 * k));
      }
    }
    buf ^= 1;
  }
  cp_async_wait<0>();   // no copy is left in flight when the block exits
}

cudaError_t launch_mx_quantize_t(const uint16_t* src, long long ld, int batch, int R, int C, int valid_rows,
                                 const int* row_src, int topk, const int* header, uint8_t* codes, uint8_t* scales,
                                 int tiled, int num_sms, cudaStream_t st, uint8_t* rcodes, uint8_t* rscales,
                                 int rtiled) {
  const long long tiles = static_cast<long long>(batch) * ((R + 127) / 128) * (C / 64);
  if (tiles == 0) return cudaSuccess;
  if (tiles >= (1ll << 31)) return cudaErrorInvalidValue;   // the kernel indexes tiles in 32 bits
  // up to 32 blocks per SM, far more than are resident at once (5): blocks
  // that start as others finish keep more tiles' copies in flight than a
  // single resident wave walking its tiles does (measured on one GB300: 8, 16,
  // 32, 64 and 128 per SM; 32 was fastest)
  const long long cap = static_cast<long long>(num_sms) * 32;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  cudaError_t err = launch_dependent(mx_quantize_t_kernel, dim3(grid), dim3(256), 0, st, src, ld, batch, R, C,
                                     valid_rows, row_src, topk, header, codes, scales, tiled, rcodes, rscales, rtiled);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Row-major E8M0 scales [rows][K/32] -> the tensor-core scale layout, for up
// to kMaxScaleJobs matrices in one launch (a forward or a backward needs six;
// separate launches would each wait for the last).  One block per (128-row
// block of one job, 16 column groups): coalesced row reads into shared memory,
// coalesced atom writes out of it.  The blocks of one 128-row block are
// neighbours in the grid, so that the pieces of a row they read share its
// L2 lines while those are resident (in row-block order the lines came from
// DRAM once per block).
struct TileScaleJobs {
  const uint8_t* src[kMaxScaleJobs];
  uint8_t* dst[kMaxScaleJobs];
  int K[kMaxScaleJobs];
  int gate_up[kMaxScaleJobs];   // 0: row r -> row r; 1 / 2: gate / up rows into the interleaved layout
  int group[kMaxScaleJobs];     // rows per expert of an interleaved job
  int rb0[kMaxScaleJobs + 1];   // job j owns 128-row blocks [rb0[j], rb0[j+1])
  int n;
  int ny;                       // blocks per 128-row block (16 column groups each)
};

__global__ void __launch_bounds__(256) mx_tile_scales_kernel(const __grid_constant__ TileScaleJobs J) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ uint32_t tile[128][17];
  const int xb = static_cast<int>(blockIdx.x / J.ny);   // 128-row block over all jobs
  int j = 0;
  while (j + 1 < J.n && xb >= J.rb0[j + 1]) ++j;
  const int cg = J.K[j] / 128;
  const int g0 = static_cast<int>(blockIdx.x % J.ny) * 16;
  if (g0 >= cg) return;   // this job has fewer column groups than the widest one
  const long long rb = xb - J.rb0[j];
  const int ng = min(16, cg - g0);
  const uint32_t* s = reinterpret_cast<const uint32_t*>(J.src[j]);  // one word = one column group of a row
  uint8_t* dst = J.dst[j];
  // all eight loads of a thread in flight before any of them is stored (one
  // at a time, the block's 8 KB took several memory latencies)
  uint32_t v[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = threadIdx.x + 256 * q, row = i >> 4, g = i & 15;
    v[q] = g < ng ? __ldg(s + (rb * 128 + row) * cg + g0 + g) : 0u;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = threadIdx.x + 256 * q;
    tile[i >> 4][i & 15] = v[q];
  }
  __syncthreads();
  if (J.gate_up[j] == 0) {
    for (int i = threadIdx.x; i < 128 * 16; i += 256) {
      const int g = i >> 7, w = i & 127;       // atom g, word w = (row % 32) * 4 + row / 32
      if (g >= ng) continue;
      const int row = (w >> 2) + 32 * (w & 3);
      reinterpret_cast<uint32_t*>(dst + ((rb * cg) + g0 + g) * 512)[w] = tile[row][g];
    }
  } else {
    // interleaved gate|up rows: each 64-row half of this block goes to half of
    // a combined 128-row atom (gate rows first, up rows second)
    const long long grp = J.group[j];
    for (int i = threadIdx.x; i < 128 * 16; i += 256) {
      const int g = i >> 7, row = i & 127;
      if (g >= ng) continue;
      const long long src_row = rb * 128 + row;
      const long long e = src_row / grp, nr = src_row - e * grp;
      const long long comb = e * 2 * grp + (nr >> 6) * 128 + (J.gate_up[j] == 2 ? 64 : 0) + (nr & 63);
      const int r = static_cast<int>(comb & 127);
      reinterpret_cast<uint32_t*>(dst + (((comb >> 7) * cg) + g0 + g) * 512)[(r & 31) * 4 + (r >> 5)] = tile[row][g];
    }
  }
}

cudaError_t launch_mx_tile_scales(const MxTileScaleJob* jobs, int n, cudaStream_t st) {
  TileScaleJobs J = {};
  long long total = 0;
  int ymax = 0, m = 0;
  for (int i = 0; i < n; ++i) {
    if (jobs[i].rows <= 0) continue;
    if (m == kMaxScaleJobs || jobs[i].rows % 128 || jobs[i].K <= 0 || jobs[i].K % 128) return cudaErrorInvalidValue;
    if (jobs[i].gate_up != 0 && (jobs[i].group <= 0 || jobs[i].group % 128 || jobs[i].rows % jobs[i].group))
      return cudaErrorInvalidValue;
    J.src[m] = jobs[i].src;
    J.dst[m] = jobs[i].dst;
    J.K[m] = jobs[i].K;
    J.gate_up[m] = jobs[i].gate_up;
    J.group[m] = jobs[i].group;
    J.rb0[m] = static_cast<int>(total);
    total += jobs[i].rows / 128;
    if (total > 0x7fffffffll) return cudaErrorInvalidValue;
    ymax = max(ymax, (jobs[i].K / 128 + 15) / 16);
    ++m;
  }
  if (m == 0) return cudaSuccess;
  if (total * ymax > 0x7fffffffll) return cudaErrorInvalidValue;
  J.rb0[m] = static_cast<int>(total);
  J.n = m;
  J.ny = ymax;
  cudaError_t err = launch_dependent(mx_tile_scales_kernel, dim3(static_cast<unsigned>(total * ymax)), dim3(256), 0,
                                     st, J);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// Fixed-order combine: out[t] = bf16(base[t] + sum_{j<k} rows[slot_row[t*k + j]]),
// summed in fp32, base first, then j ascending (no floating-point atomics):
// the expert outputs sit in schedule order and are gathered back per
// (token, k) here.  One thread per 8 columns of one token.
// ===========================================================================
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const int* __restrict__ slot_row,
                                                      const int* __restrict__ header, long long max_rows,
                                                      const uint16_t* __restrict__ base, int T, int k,
                                                      int H, uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  if (header[2] != 0) return;   // no schedule (bad expert id): slot_row was never written
  const int per_row = H / 8;
  const long long total = static_cast<long long>(T) * per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / per_row;
    const int c = static_cast<int>(i - t * per_row) * 8;
    float acc[8];
    if (base) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(base + t * H + c));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __uint_as_float(ws[q] << 16);
        acc[2 * q + 1] = __uint_as_float(ws[q] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    }
    for (int j = 0; j < k; ++j) {
      long long row = __ldg(slot_row + t * k + j);
      row = row < 0 ? 0 : (row >= max_rows ? max_rows - 1 : row);   // in bounds whatever the array holds
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(rows + row * H + c));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(ws[q] << 16);
        acc[2 * q + 1] += __uint_as_float(ws[q] & 0xFFFF0000u);
      }
    }
    *reinterpret_cast<uint4*>(out + t * H + c) =
        make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                   pack_bf16(acc[6], acc[7]));
  }
}

cudaError_t launch_combine(const uint16_t* rows, const int* slot_row, const int* header, long long max_rows,
                           const uint16_t* base, int T, int k, int H, uint16_t* out, int num_sms, cudaStream_t st) {
  const long long total = static_cast<long long>(T) * (H / 8);
  cudaError_t err = launch_dependent(combine_kernel, dim3(grid_for(total, 256, num_sms)), dim3(256), 0, st, rows,
                                     slot_row, header, max_rows, base, T, k, H, out);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ===========================================================================
// Dispatch permutation: out[p - w0] = src[row_src[p] / k] for every schedule
// row p of the window [w0, w0 + wrows) below P (zeros for padding rows), so
// the routed GEMMs read their gathered operand as dense TMA tiles.  The whole
// schedule is the window [0, max_rows); a macrobatch ring passes the rows of
// one window of experts.  Token-major: one warp per token reads its row once
// and writes it to those of the token's k schedule rows (slot_row) that fall
// in the window, four 16-byte pieces per lane in flight, each store
// instruction 512 contiguous bytes; then one warp per padding row of the
// window writes zeros.  Bandwidth bound: T*H*2 bytes read, the window's rows
// *H*2 written (a row-major walk over schedule rows would read each token row
// k times).
// ===========================================================================
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint16_t* __restrict__ src, int T, int H, int topk,
                                                           const int* __restrict__ slot_row,
                                                           const int* __restrict__ row_src,
                                                           const int* __restrict__ header, long long w0,
                                                           long long wrows, uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  if (header[2] != 0) return;
  const long long P = header[1];
  const int lane = threadIdx.x & 31;
  const int per_row = H / 8;  // 16-byte pieces per row
  const long long jobs = T + wrows;
  for (long long j = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; j < jobs;
       j += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    if (j < T) {
      const int p_lo = lane < topk ? __ldg(slot_row + j * topk + lane) : -1;
      const int p_hi = lane + 32 < topk ? __ldg(slot_row + j * topk + lane + 32) : -1;
      // a token none of whose rows falls in the window is not read at all
      if (!__any_sync(0xffffffffu, (p_lo >= w0 && p_lo - w0 < wrows) || (p_hi >= w0 && p_hi - w0 < wrows))) continue;
      const uint4* s = reinterpret_cast<const uint4*>(src + j * H);
      for (int i0 = 0; i0 < per_row; i0 += 128) {
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i0 + lane + 32 * q < per_row) v[q] = __ldg(s + i0 + lane + 32 * q);
        for (int jj = 0; jj < topk; ++jj) {   // all lanes take part in the shuffle
          const long long pr = __shfl_sync(0xffffffffu, jj < 32 ? p_lo : p_hi, jj & 31) - w0;
          if (pr < 0 || pr >= wrows) continue;   // the same for every lane
          uint4* d = reinterpret_cast<uint4*>(out + pr * H);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (i0 + lane + 32 * q < per_row) d[i0 + lane + 32 * q] = v[q];
        }
      }
    } else {
      const long long pr = j - T;
      if (w0 + pr >= P || __ldg(row_src + w0 + pr) >= 0) continue;
      uint4* d = reinterpret_cast<uint4*>(out + pr * H);
      for (int i = lane; i < per_row; i += 32) d[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

cudaError_t launch_permute_rows(const uint16_t* src, int T, int H, int topk, const int* slot_row, const int* row_src,
                                const int* header, long long w0, long long wrows, uint16_t* out, int num_sms,
                                cudaStream_t st) {
  if (wrows == 0) return cudaSuccess;
  cudaError_t err = launch_dependent(permute_rows_kernel, dim3(grid_for((T + wrows) * 32, 256, num_sms)), dim3(256),
                                     0, st, src, T, H, topk, slot_row, row_src, header, w0, wrows, out);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// d_w[f] = sum over column tiles n (ascending) of part[f][n].
__global__ void dw_reduce_kernel(const float* __restrict__ part, int nf, int ntiles,
                                 float* __restrict__ dw) {
  griddep_wait();
  griddep_launch_dependents();
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= nf) return;
  float s = 0.f;
  for (int n = 0; n < ntiles; ++n) s += part[static_cast<long long>(f) * ntiles + n];
  dw[f] = s;
}

cudaError_t launch_dw_reduce(const float* part, int nf, int ntiles, float* dw, cudaStream_t st) {
  if (nf == 0) return cudaSuccess;
  cudaError_t err = launch_dependent(dw_reduce_kernel, dim3((nf + 255) / 256), dim3(256), 0, st, part, nf, ntiles, dw);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace mok

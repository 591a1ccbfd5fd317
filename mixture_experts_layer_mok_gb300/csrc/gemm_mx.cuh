// Persistent grouped GEMM on the block-scaled tensor-core path
// (tcgen05.mma kind::mxf8f6f4, E4M3 operands with E8M0 scales per 32 K-elements)
// for the MXFP8 forward and the MXFP8 backward.
//
// One CTA per SM, 320 threads:
//   warp 0      TMA producer: operand tiles (128-byte rows of E4M3 codes) and
//               the matching 512-byte scale atoms (1-D bulk copies);
//   warp 1      MMA issuer (one thread) and TMEM owner: per stage it copies the
//               scale atoms into TMEM (tcgen05.cp) and issues four K=32 MMAs;
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each half the
//               columns.
// A 256-column accumulator is single-buffered (the scale ring takes the rest
// of TMEM); a 128-column one is double-buffered.  The epilogue reads its share
// of the accumulator into registers and releases TMEM at once, so the next
// tile's MMAs overlap the epilogue's arithmetic and stores; the SwiGLU
// backward instead reads its 128-column buffer as it goes.
//
// Row GEMMs take their rows from the schedule's tile list (or dense rows);
// weight-gradient GEMMs contract over an expert's row range, with both
// operands stored transposed (the layer's rows as K).
//
// Follows "Mixture-of-Kittens: a deterministic MoE megakernel for NVL72 racks"
// (MXFP8 forward and backward; experts as fused SwiGLU grouped GEMMs) with
// MXFP8 as the OCP Microscaling v1.0 format: E4M3 elements, one E8M0
// power-of-two scale per block of 32 along K.
#pragma once

#include "gemm.cuh"

namespace mok {

// Tensor maps of a block-scaled GEMM: the E4M3 operand tiles and, for CTA
// pairs, the scale atoms viewed as rows of 128 bytes (4 rows per atom), so
// that the peer CTA's atoms also complete on the leader's barrier.
struct MxMaps {
  CUtensorMap a, b0, b1;
  CUtensorMap sfa, sfb0, sfb1;
  // EPI_DOWN_BWD_MX: its E4M3 outputs, stored by TMA in 32 x 32-byte boxes
  // (dG|dU by rows, dG|dU transposed, w h transposed)
  CUtensorMap o0, o1, o2;
};

template <int BN, int EPI, bool PAIR = false>
struct MxCfg {
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kBK = 128;                      // E4M3 elements (= bytes) per stage: one swizzled row
  static constexpr int kABytes = kBM * kBK;
  // CTA pair: each CTA holds half of B's rows, and the scales of all of them
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kBBytes = kBRows * kBK;
  static constexpr int kSfaBytes = 512;                // one scale atom: 128 rows x 4 blocks
  static constexpr int kSfbBytes = (BN / 128) * 512;
  static constexpr int kSfStride = 2048;               // per stage: A atom at 0, B atoms at 512, 1024
  static constexpr int kTmaBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarBytes = 512;
  // per epilogue warp: one 32-row staging block (2 KB); the MXFP8 SwiGLU
  // backward stages its three 32 x 32 output blocks (dG, dU, w h)
  // per epilogue warp: the staging of its TMA stores (a 32 x 32 bf16 block;
  // the SwiGLU adds a 32 x 32 block of E4M3 codes; the MXFP8 SwiGLU backward
  // stages its three 32 x 32 output blocks)
  static constexpr int kEpiStageBytes =
      EPI == EPI_DOWN_BWD_MX ? 3 * 2048 : (EPI == EPI_SWIGLU_MX ? 2048 + 1024 : 2048);
  static constexpr int kStagesFit =
      (227 * 1024 - 1024 - kBarBytes - kEpiWarps * kEpiStageBytes) / (kStageBytes + kSfStride);
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  // TMEM: accumulator columns (two buffers of BN when they fit beside the
  // scale ring, else one), then one 16-column scale slot per stage (A: 4
  // columns at +0, B: 4 columns per 128 rows at +8)
  static constexpr int kTmemCols = 512;
  static constexpr int kAccBufs = (2 * BN + 16 * kStages <= kTmemCols) ? 2 : 1;
  static constexpr int kSfCol0 = kAccBufs * BN;
  static constexpr int kSmemBytes =
      1024 + kStages * (kStageBytes + kSfStride) + kBarBytes + kEpiWarps * kEpiStageBytes;
  static_assert(BN == 128 || BN == 256, "tile N");
  // SwiGLU tiles pair 128 gate rows with 128 up rows (whole scale atoms); a
  // CTA pair's 128-wide tile pairs 64 gate with 64 up rows, whose scales sit
  // in one atom of the interleaved gate|up layout
  static_assert(EPI != EPI_SWIGLU_MX || BN == 256 || PAIR, "SwiGLU tile");
  static_assert(kSfCol0 + 16 * kStages <= kTmemCols, "TMEM scale ring");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// A 32 x 32 bf16 block staged in shared memory: 32 rows of 16 packed words,
// word w of row l at l*16 + (w ^ (l & 15)), so that both a lane reading its
// own row and a lane reading one column (across the 32 rows) spread over the
// banks.
__device__ __forceinline__ void stage_put(uint32_t* blk, int row, int w, uint32_t val) {
  blk[row * 16 + (w ^ (row & 15))] = val;
}

__device__ __forceinline__ uint32_t mx_store_codes(const float* v, uint8_t* dst) {
  uint8_t q[32];
  const uint32_t s = mx_quantize32(v, q);
  if (dst) {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = reinterpret_cast<const uint4*>(q)[0];
    d[1] = reinterpret_cast<const uint4*>(q)[1];
  }
  return s;
}

// MXFP8 block along this lane's row of a staged block: the 32 E4M3 codes go to
// dst (NULL = nowhere); returns the E8M0 scale code.
__device__ __forceinline__ uint32_t mx_row_from_stage(const uint32_t* blk, int lane, uint8_t* dst) {
  float v[32];
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    const uint32_t x = blk[lane * 16 + (w ^ (lane & 15))];
    v[2 * w] = __uint_as_float(x << 16);
    v[2 * w + 1] = __uint_as_float(x & 0xFFFF0000u);
  }
  return mx_store_codes(v, dst);
}

// MXFP8 block down column `lane` of a staged block (its 32 rows): the 32 E4M3
// codes go to dst (a row of the transposed tensor); returns the scale code.
__device__ __forceinline__ uint32_t mx_col_from_stage(const uint32_t* blk, int lane, uint8_t* dst) {
  float v[32];
  const int wc = lane >> 1;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t x = blk[i * 16 + (wc ^ (i & 15))];
    v[i] = __uint_as_float((lane & 1) ? (x & 0xFFFF0000u) : (x << 16));
  }
  return mx_store_codes(v, dst);
}

// Warp-cooperative TMA store of a 32-row x 32-column bf16 block at {col, row}
// through one 2 KB staging block (the 64-byte-swizzled layout of the output's
// tensor map): each lane hands in 16 packed words of its row.  The staging is
// reused once the previous bulk copy of lane 0 has read it.
__device__ __forceinline__ void warp_store_tma1(const uint32_t* w, const CUtensorMap* map, int col, int row,
                                                uint8_t* stage, int lane) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  uint4* s = reinterpret_cast<uint4*>(stage);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    s[lane * 4 + (j ^ sw)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();   // generic-proxy writes, then the async-proxy read
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, col, row);
    bulk_commit();
  }
}

// The same for a 32-row x 32-byte block of E4M3 codes (unswizzled 1 KB
// staging, row r at byte 32 r): each lane hands in its row's 32 codes.
__device__ __forceinline__ void warp_store_codes_tma(const uint8_t* codes, const CUtensorMap* map, int col, int row,
                                                     uint8_t* stage, int lane) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  uint4* s = reinterpret_cast<uint4*>(stage + lane * 32);
  s[0] = reinterpret_cast<const uint4*>(codes)[0];
  s[1] = reinterpret_cast<const uint4*>(codes)[1];
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, col, row);
    bulk_commit();
  }
}

// Shared-memory descriptor of a 512-byte scale atom as the tcgen05.cp source:
// 32 rows of 16 bytes, no swizzle, 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sf_atom_desc(uint32_t saddr) { return smem_desc(saddr, 128, 128, 0); }

template <int BN, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(MxCfg<BN, EPI, PAIR>::kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ MxMaps maps, const GemmParams p) {
  using C = MxCfg<BN, EPI, PAIR>;
  static_assert(EPI == EPI_SWIGLU_MX || EPI == EPI_SCALE_ROWS || EPI == EPI_STORE_ROWS || EPI == EPI_WGRAD ||
                    EPI == EPI_DOWN_BWD_MX,
                "epilogue");
  static_assert(!PAIR || (EPI != EPI_WGRAD && EPI != EPI_DOWN_BWD_MX), "backward epilogues run on single CTAs");
  static_assert(EPI != EPI_DOWN_BWD_MX || (BN == 128 && C::kAccBufs == 2),
                "MXFP8 SwiGLU backward: 64 columns per thread, double-buffered accumulator");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sf_smem = smem + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_smem + C::kStages * C::kSfStride);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = bars + 2 * C::kStages;   // per accumulator buffer
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 128-column groups of the A and B scale layouts
  const int kga = p.sf_kga > 0 ? p.sf_kga : p.K / C::kBK;
  const int kgb = p.sf_kgb > 0 ? p.sf_kgb : p.K / C::kBK;
  // CTA pair: rank in the pair, persistent loop over the pair's items
  const int rank = PAIR ? static_cast<int>(cluster_rank()) : 0;
  const int item0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int istep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto item_at = [&](int idx) { return PAIR ? get_item_pair(p, idx, C::kBK, rank) : get_item(p, idx, C::kBK); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (PAIR ? 2 : 1) * C::kEpiWarps);   // the leader's counts both CTAs' warps
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
  constexpr bool kSwiGLU = (EPI == EPI_SWIGLU_MX);
  constexpr int kBnOut = kSwiGLU ? BN / 2 : BN;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      for (int idx = item0; idx < nitems && ok; idx += istep) {
        const Item it = item_at(idx);
        const int n0 = it.nt * kBnOut;
        // row GEMMs: A rows are layer rows p0.., B rows the expert's weight
        // rows; weight gradients: A rows m0.., B rows n0.. of tensors whose
        // columns are the layer rows, the expert's K range starting at kbeg
        const bool wg = p.wgrad != 0;
        const long long arow = wg ? it.m0 : it.p0;
        const long long brow = wg ? n0 : static_cast<long long>(it.e) * p.b_rows_per_expert + n0;
        // scale atoms of the item's A rows and B rows (B: gate then up, or two
        // consecutive 128-row blocks; a pair's 128-wide SwiGLU tile: one atom of
        // the interleaved gate|up layout, 2 * b_rows_per_expert rows per expert),
        // as atom indices at K-block 0
        const long long atom_a = (arow >> 7) * static_cast<long long>(kga);
        const long long brow_sf =
            (PAIR && BN == 128 && kSwiGLU) ? 2ll * it.e * p.b_rows_per_expert + 2ll * n0 : brow;
        const long long atom_b0 = (brow_sf >> 7) * static_cast<long long>(kgb);
        const long long atom_b1 = kSwiGLU ? atom_b0 : atom_b0 + kgb;
        for (int kb = 0; kb < it.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          // CTA pair: both CTAs' loads complete on the leader's barrier
          if (!PAIR || rank == 0) mbar_arrive_expect_tx(&full[stage], (PAIR ? 2 : 1) * C::kTmaBytes);
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + C::kABytes;
          uint8_t* sS = sf_smem + stage * C::kSfStride;
          const int k0 = kb * C::kBK;
          if constexpr (PAIR) {
            const uint32_t lf = cluster_addr(&full[stage], 0);
            tma_load_2d_pair(sA, &maps.a, lf, k0, it.p0);
            if (kSwiGLU)   // the leader holds the gate rows, the peer the up rows
              tma_load_2d_pair(sB, rank == 0 ? &maps.b0 : &maps.b1, lf, k0, static_cast<int>(brow));
            else
              tma_load_2d_pair(sB, &maps.b0, lf, k0, static_cast<int>(brow) + rank * C::kBRows);
            tma_load_2d_pair(sS, &maps.sfa, lf, 0, static_cast<int>((atom_a + kb) * 4));
            tma_load_2d_pair(sS + 512, &maps.sfb0, lf, 0, static_cast<int>((atom_b0 + kb) * 4));
            if (BN == 256)
              tma_load_2d_pair(sS + 1024, kSwiGLU ? &maps.sfb1 : &maps.sfb0, lf, 0,
                               static_cast<int>((atom_b1 + kb) * 4));
          } else {
            // K coordinate of this K-block in the operand tensors, and which B
            // tensor holds it (a K range split over two weights: b_split)
            const int ka = (wg ? it.kbeg : 0) + k0;
            int kbb = ka;
            bool second = false;
            if (!wg && p.b_split > 0 && k0 >= p.b_split) {
              kbb = k0 - p.b_split;
              second = true;
            }
            const long long kba = ka / C::kBK, kbq = kbb / C::kBK;   // K-block index within each scale layout
            tma_load_2d(sA, &maps.a, &full[stage], ka, static_cast<int>(arow));
            if (kSwiGLU) {
              tma_load_2d(sB, &maps.b0, &full[stage], k0, static_cast<int>(brow));
              tma_load_2d(sB + (BN / 2) * C::kBK, &maps.b1, &full[stage], k0, static_cast<int>(brow));
            } else {
              tma_load_2d(sB, second ? &maps.b1 : &maps.b0, &full[stage], kbb, static_cast<int>(brow));
            }
            const uint8_t* sfb = (kSwiGLU || second) ? p.sfb1 : p.sfb0;
            bulk_load(sS, p.sfa + (atom_a + kba) * 512, 512, &full[stage]);
            bulk_load(sS + 512, (kSwiGLU ? p.sfb0 : sfb) + (atom_b0 + kbq) * 512, 512, &full[stage]);
            if (BN == 256) bulk_load(sS + 1024, sfb + (atom_b1 + kbq) * 512, 512, &full[stage]);
          }
          ++fills;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && (!PAIR || rank == 0)) {
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
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {   // a CTA pair's leader issues for both
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool first = true;
      for (int idx = item0; idx < nitems; idx += istep) {
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
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t b0 = a0 + C::kABytes;
          const uint32_t s0 = smem_u32(sf_smem + stage * C::kSfStride);
          const uint32_t sfa_t = tmem_base + C::kSfCol0 + stage * 16;
          const uint32_t sfb_t = sfa_t + 8;
          // scale atoms -> TMEM (executed in order with the MMAs below; a pair's
          // copy moves each CTA's atoms into its own TMEM)
          if (PAIR) {
            tmem_cp_32x128b_warpx4_pair(sfa_t, sf_atom_desc(s0));
            tmem_cp_32x128b_warpx4_pair(sfb_t, sf_atom_desc(s0 + 512));
            if (BN == 256) tmem_cp_32x128b_warpx4_pair(sfb_t + 4, sf_atom_desc(s0 + 1024));
          } else {
            tmem_cp_32x128b_warpx4(sfa_t, sf_atom_desc(s0));
            tmem_cp_32x128b_warpx4(sfb_t, sf_atom_desc(s0 + 512));
            if (BN == 256) tmem_cp_32x128b_warpx4(sfb_t + 4, sf_atom_desc(s0 + 1024));
          }
#pragma unroll
          for (int kk = 0; kk < C::kBK / 32; ++kk) {
            // K-major 128-byte swizzled rows: 32 E4M3 elements = 32 bytes per step
            const uint64_t ad = smem_desc(a0 + kk * 32, 16, 8 * C::kBK, 2);
            const uint64_t bd = smem_desc(b0 + kk * 32, 16, 8 * C::kBK, 2);
            if (PAIR)
              umma_mxf8_pair(acc, ad, bd, idesc_mxf8(2 * kBM, BN, kk, kk), sfa_t, sfb_t, (kb | kk) ? 1u : 0u);
            else
              umma_mxf8(acc, ad, bd, idesc_mxf8(kBM, BN, kk, kk), sfa_t, sfb_t, (kb | kk) ? 1u : 0u);
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
        if (++abuf == C::kAccBufs) {
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;      // which half of the columns
    const int r = q * 32 + lane;           // tile row of this thread
    uint8_t* wstage = sf_smem + C::kStages * C::kSfStride + C::kBarBytes + (warp - 2) * C::kEpiStageBytes;
    int abuf = 0;
    uint32_t aphase = 0;
    constexpr int kCols = BN / 2;          // accumulator columns per thread
    // weight gradients: destination of output row m of expert e (rows below
    // `split` go to out0, the rest to out1), at column col
    auto wgrad_row = [&](const Item& t, int m, int col) -> uint16_t* {
      const int mrows = p.m_tiles * kBM;
      if (m < p.split)
        return static_cast<uint16_t*>(p.out0) + (static_cast<long long>(t.e) * p.split + m) * p.ld + col;
      return static_cast<uint16_t*>(p.out1) +
             (static_cast<long long>(t.e) * (mrows - p.split) + (m - p.split)) * p.ld + col;
    };
    for (int idx = item0; idx < nitems; idx += istep) {
      const Item it = item_at(idx);
      if (it.nk == 0) {
        if constexpr (EPI == EPI_WGRAD) {   // an expert with no rows: zero gradient
          uint32_t zw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) zw[i] = 0u;
          uint16_t* dst = wgrad_row(it, it.m0 + r, it.nt * kBnOut + half * kCols);
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) warp_store_row64(zw, dst + c * 32, wstage, lane);
        }
        continue;
      }
      const int n0 = it.nt * kBnOut;
      const int prow = it.p0 + r;
      const bool live = !it.empty;     // an empty half of a CTA pair stores nothing
      const bool valid = live && r < it.rows;
      int f = -1;
      float wt = 1.f;
      if (EPI == EPI_SCALE_ROWS && valid) {
        f = __ldg(p.row_src + prow);
        if (f >= 0) wt = __ldg(p.rw + f);
      }
      int w = (lane == 0) ? (mbar_wait(&tfull[abuf], aphase, abort_flag, p.status) ? 1 : 0) : 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(abuf * BN) + (static_cast<uint32_t>(q * 32) << 16);
      // the accumulator buffer goes back to the MMA (a pair: on the leader's barrier)
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank != 0)
            mbar_arrive_cluster(cluster_addr(&tempty[abuf], 0));
          else
            mbar_arrive(&tempty[abuf]);
        }
        if (++abuf == C::kAccBufs) {
          abuf = 0;
          aphase ^= 1;
        }
      };
      // this thread's share of the accumulator, then TMEM goes back to the MMA
      // (the SwiGLU backward reads its chunks as it goes, from a second buffer)
      float v[EPI == EPI_DOWN_BWD_MX ? 1 : kCols];
      if constexpr (EPI != EPI_DOWN_BWD_MX) {
        // all loads in flight at once, one wait: the MMA waits for this drain
        uint32_t ta[kCols / 32];
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
          if (kSwiGLU)   // gate columns [half*BN/4, +BN/4) to v[0, kCols/2), up columns BN/2 later
            ta[c] = tb + (c < kCols / 64 ? half * (BN / 4) + c * 32 : BN / 2 + half * (BN / 4) + (c - kCols / 64) * 32);
          else
            ta[c] = tb + half * kCols + c * 32;
        }
        tmem_ld32_multi<kCols / 32>(ta, v);
        release_acc();
      }

      uint32_t wv[16];
      const int orow = it.p0 + q * 32;     // first row of this warp's 32 rows
      if constexpr (EPI == EPI_SWIGLU_MX) {
        // map o0 = G|U [rows][2N] (bf16), o1 = h codes [rows][N], sf_out = h
        // scales; both stored by TMA in 32-row blocks (rows past a dense
        // layer's end are clipped; a grouped tile's padding rows are zeros)
        constexpr int kH = kCols / 2;        // h columns of this thread
        const int col0 = n0 + half * kH;
        float* g = v;
        float* u = v + kH;
        if (!valid) {
#pragma unroll
          for (int i = 0; i < kCols; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < kH / 32; ++c) {
          pack_bf16x32(g + c * 32, wv);
          if (live) warp_store_tma1(wv, &maps.o0, col0 + c * 32, orow, wstage, lane);
          pack_bf16x32(u + c * 32, wv);
          if (live) warp_store_tma1(wv, &maps.o0, p.N + col0 + c * 32, orow, wstage, lane);
        }
        uint32_t sc = 0;
#pragma unroll
        for (int c = 0; c < kH / 32; ++c) {
          float* hv = g + c * 32;        // h overwrites the gate values (already stored)
          const float lim = p.swiglu_limit;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x = hv[i], uc = u[c * 32 + i];
            if (lim > 0.f) {   // clamped SwiGLU (G|U are saved unclamped for the backward)
              x = fminf(x, lim);
              uc = fminf(fmaxf(uc, -lim), lim);
            }
            const float sg = __fdividef(1.f, 1.f + __expf(-x));
            hv[i] = x * sg * uc;
          }
          uint8_t codes[32];
          const uint32_t s8 = mx_quantize32(hv, codes);
          sc |= s8 << (8 * c);
          if (live) warp_store_codes_tma(codes, &maps.o1, col0 + c * 32, orow, wstage + 2048, lane);
        }
        // the scales of this thread's blocks are adjacent bytes of its row's word
        // (rows past the end of a dense layer get the unit scales of zeros)
        if (live) {
          uint8_t* sdst = p.sf_out + mx_tiled_scale_offset(prow, col0 / 32, p.N / 128);
          if (kH == 64) {
            *reinterpret_cast<uint16_t*>(sdst) = static_cast<uint16_t>(sc);
          } else {
            *sdst = static_cast<uint8_t>(sc);
          }
        }
      } else if constexpr (EPI == EPI_WGRAD) {
        // out[e][m][n] = bf16(acc): every row of a weight-gradient tile is real
        uint16_t* dst = wgrad_row(it, it.m0 + r, n0 + half * kCols);
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
          pack_bf16x32(v + c * 32, wv);
          warp_store_row64(wv, dst + c * 32, wstage, lane);
        }
      } else if constexpr (EPI == EPI_DOWN_BWD_MX) {
        // dgrad through down + SwiGLU backward, with the MXFP8 operands of the
        // next GEMMs as outputs, each quantised from the bf16-rounded value and
        // stored by TMA: map o0 = dG|dU codes [rows][2N] by rows (scales sf_out,
        // tensor-core layout), o1 = dG|dU codes transposed [2N][ld] and o2 =
        // (w h) codes transposed [N][ld], both in 32-row blocks (scales in out2
        // and sf_out2); ld = rows of the transposed tensors (schedule rows, or
        // tokens padded to 128).  Padding rows and dense rows past the end count
        // as zeros (o0 clips the latter).
        int f = -1;
        bool v_ok;
        float wt = 1.f;
        if (p.grouped) {
          f = valid ? __ldg(p.row_src + prow) : -1;
          v_ok = f >= 0;
          if (v_ok) wt = __ldg(p.rw + f);
        } else {
          v_ok = valid;
        }
        const int col0 = n0 + half * kCols;
        const uint16_t* gu = static_cast<const uint16_t*>(p.aux0) + static_cast<long long>(prow) * 2 * p.N + col0;
        const long long ldt = p.ld;
        const int cgr = 2 * p.N / 128, cgt = static_cast<int>(ldt / 128);
        const int rblk = (it.p0 + q * 32) / 32;                // 32-row block of this warp's rows
        const long long tcol = it.p0 + q * 32;                 // its first row in the transposed tensors
        uint32_t* blk_g = reinterpret_cast<uint32_t*>(wstage);   // staged dG, dU, w h blocks
        uint32_t* blk_u = blk_g + 512;
        uint32_t* blk_h = blk_g + 1024;
        const float lim = p.swiglu_limit;
        float dpart = 0.f;
        uint32_t rsc_g = 0, rsc_u = 0;
        const int prow0 = it.p0 + q * 32;                      // the warp's first row
        // saved gate|up of the next 16 columns, loaded one slice ahead
        uint4 pg[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)}, pu[2] = {pg[0], pg[1]};
        auto fetch_gu = [&](int col) {
          if (v_ok) {
            const uint4* sg4 = reinterpret_cast<const uint4*>(gu + col);
            const uint4* su4 = reinterpret_cast<const uint4*>(gu + p.N + col);
            pg[0] = __ldg(sg4); pg[1] = __ldg(sg4 + 1);
            pu[0] = __ldg(su4); pu[1] = __ldg(su4 + 1);
          }
        };
        fetch_gu(0);
#pragma unroll 1
        for (int c = 0; c < kCols / 32; ++c) {
          if (lane == 0) bulk_wait_read<0>();   // the last chunk's code boxes have left the blocks
          __syncwarp();
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {   // 16 columns at a time keep the registers low
            const uint4 ng[2] = {pg[0], pg[1]}, nu[2] = {pu[0], pu[1]};
            if (c * 32 + hf * 16 + 16 < kCols) fetch_gu(c * 32 + hf * 16 + 16);
            float z[16];
            tmem_ld16(tb + half * kCols + c * 32 + hf * 16, z);
            // no branch on the row: a padding row (or a dense row past the end)
            // has zero gate|up and a zero accumulator row, so every output is 0
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              float a[2], b[2], hh[2];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                float g = bf16_at(ng, i + t), u = bf16_at(nu, i + t);
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
                const float dh = wt * z[i + t];
                a[t] = dh * u * sg * (1.f + g * (1.f - sg)) * mg;
                b[t] = dh * sl * mu;
                hh[t] = wt * h;
              }
              const int wi = hf * 8 + (i >> 1);
              stage_put(blk_g, lane, wi, pack_bf16(a[0], a[1]));
              stage_put(blk_u, lane, wi, pack_bf16(b[0], b[1]));
              stage_put(blk_h, lane, wi, pack_bf16(hh[0], hh[1]));
            }
          }
          __syncwarp();
          // each staged block -> its codes: lane j takes column j (transposed
          // output) and row j (row output); the codes then replace the block in
          // shared memory (transposed box at +0, row box at +1 KB) for the TMA stores
          const int tg0 = col0 + c * 32;
          const int tg = tg0 + lane;
          uint8_t* dguT_sc = static_cast<uint8_t*>(p.out2);
#pragma unroll 1
          for (int o = 0; o < 3; ++o) {
            uint32_t* blk = o == 0 ? blk_g : (o == 1 ? blk_u : blk_h);
            uint32_t cq[8], rq[8];
            const uint32_t cs = mx_col_from_stage(blk, lane, reinterpret_cast<uint8_t*>(cq));
            uint32_t rs = 0;
            if (o < 2) rs = mx_row_from_stage(blk, lane, reinterpret_cast<uint8_t*>(rq));
            __syncwarp();
            uint4* box = reinterpret_cast<uint4*>(blk);
            box[lane * 2] = make_uint4(cq[0], cq[1], cq[2], cq[3]);
            box[lane * 2 + 1] = make_uint4(cq[4], cq[5], cq[6], cq[7]);
            if (o < 2) {
              box[64 + lane * 2] = make_uint4(rq[0], rq[1], rq[2], rq[3]);
              box[64 + lane * 2 + 1] = make_uint4(rq[4], rq[5], rq[6], rq[7]);
            }
            if (live) {
              const int trow = (o == 1 ? p.N : 0) + tg;
              (o == 2 ? p.sf_out2 : dguT_sc)[mx_tiled_scale_offset(trow, rblk, cgt)] = static_cast<uint8_t>(cs);
            }
            if (o == 0) rsc_g |= rs << (8 * c);
            if (o == 1) rsc_u |= rs << (8 * c);
          }
          fence_proxy_async_smem();   // generic-proxy writes, then the TMA stores read them
          __syncwarp();
          if (lane == 0 && live) {
            tma_store_2d(&maps.o1, blk_g, static_cast<int>(tcol), tg0);          // dG transposed
            tma_store_2d(&maps.o1, blk_u, static_cast<int>(tcol), p.N + tg0);    // dU transposed
            tma_store_2d(&maps.o2, blk_h, static_cast<int>(tcol), tg0);          // w h transposed
            tma_store_2d(&maps.o0, blk_g + 256, tg0, prow0);                    // dG rows (clipped past the end)
            tma_store_2d(&maps.o0, blk_u + 256, p.N + tg0, prow0);              // dU rows
            bulk_commit();
          }
        }
        release_acc();
        // this thread's two row blocks of dG and of dU are adjacent bytes of
        // its row's scale word (rows past a dense layer's end: unit scales)
        if (live) {
          *reinterpret_cast<uint16_t*>(p.sf_out + mx_tiled_scale_offset(prow, col0 / 32, cgr)) =
              static_cast<uint16_t>(rsc_g);
          *reinterpret_cast<uint16_t*>(p.sf_out + mx_tiled_scale_offset(prow, (p.N + col0) / 32, cgr)) =
              static_cast<uint16_t>(rsc_u);
        }
        if (p.grouped && v_ok) p.dw_part[(static_cast<long long>(f) * p.n_tiles + it.nt) * 2 + half] = dpart;
      } else {
        // map o0 = rows in schedule order (router-weighted: the combine reads
        // them back per (token, k) through slot_row; a tile's padding rows get
        // zeros), or dense rows (clipped past the layer's end), by TMA
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
          if (EPI == EPI_SCALE_ROWS) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c * 32 + i] *= wt;
          }
          pack_bf16x32(v + c * 32, wv);
          if (live) warp_store_tma1(wv, &maps.o0, n0 + half * kCols + c * 32, orow, wstage, lane);
        }
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

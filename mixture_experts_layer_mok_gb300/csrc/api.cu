// C ABI of libmok (declared in include/mok.h): argument checks, carving of the
// caller's buffers, TMA descriptor encoding and the launch sequence of the
// forward and backward passes.  No allocation happens here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "../../include/mok.h"
#include "gemm.cuh"
#include "gemm_mx.cuh"
#include "internal.h"

using namespace mok;

namespace {

thread_local char g_err[512] = "";

mok_status_t fail(mok_status_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

#define MOK_CUDA(call)                                                                     \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return fail(MOK_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_),    \
                  __FILE__, __LINE__);                                                     \
  } while (0)

// ---------------------------------------------------------------- device info
struct DevInfo {
  int checked = 0;
  int ok = 0;
  int num_sms = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

mok_status_t device_info(int* num_sms) {
  int dev = 0;
  MOK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOK_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    MOK_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    MOK_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    MOK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    d.ok = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.checked = 1;
  }
  if (!d.ok) return fail(MOK_ERR_UNSUPPORTED, "libmok runs on sm_103 (GB300) devices only");
  *num_sms = d.num_sms;
  return MOK_OK;
}

// ---------------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [outer][inner] with a box of box_outer rows x bk elements
// (bk = the kernel's K-block: 64 -> 128-byte swizzle, 32 -> 64-byte swizzle);
// out-of-range elements read as zero.
mok_status_t make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_outer, int bk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(bk), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box %u", (int)r,
                (unsigned long long)outer, (unsigned long long)inner, box_outer);
  return MOK_OK;
}

// MN-major operand tile of `tile_width` columns as one 3-D box: dims
// {bk elements, rows, width/bk chunks}, box {bk, bk K-rows, tile_width/bk},
// landing chunk-major in shared memory (the layout the MMA descriptors expect).
mok_status_t make_map_mn(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, int tile_width,
                         int bk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(bk), rows, width / bk};
  const cuuint64_t strides[2] = {width * 2, static_cast<cuuint64_t>(bk) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(bk),
                             static_cast<cuuint32_t>(tile_width / bk)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled (MN tile) failed (%d) for [%llu x %llu], tile %d", (int)r,
                (unsigned long long)rows, (unsigned long long)width, tile_width);
  return MOK_OK;
}

// 2-D tensor of E4M3 codes [outer][inner] (bytes) with a box of box_outer rows
// x 128 bytes, 128-byte swizzle; out-of-range elements read as zero.
mok_status_t make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {128, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled (E4M3) failed (%d) for [%llu x %llu] box %u", (int)r,
                (unsigned long long)outer, (unsigned long long)inner, box_outer);
  return MOK_OK;
}

// Row-major bf16 output [rows][cols] for TMA stores: box 32 rows x 32 columns
// with 64-byte swizzle (the epilogue's staging layout); rows and columns past
// the tensor's end are not written.
mok_status_t make_map_out(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d) for [%llu x %llu]", (int)r,
                (unsigned long long)rows, (unsigned long long)cols);
  return MOK_OK;
}

// Byte tensor [outer][inner] (E4M3 codes) for TMA stores of 32 x 32-byte
// boxes, no swizzle; rows and columns past the tensor's end are not written.
mok_status_t make_map_codes_out(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled (code output) failed (%d) for [%llu x %llu]", (int)r,
                (unsigned long long)outer, (unsigned long long)inner);
  return MOK_OK;
}

// E8M0 scales in the tensor-core scale layout as rows of 128 bytes, four per
// 512-byte atom (box: one atom), for the TMA loads of CTA-pair GEMMs.
mok_status_t make_map_sf(CUtensorMap* m, const void* base, long long atoms) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(atoms) * 4};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, 4};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOK_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d), %lld atoms", (int)r, atoms);
  return MOK_OK;
}

// K-block of the GEMM kernels (elements per stage); the map builders also
// support 32 (64-byte swizzle).
constexpr int kTileBK = 64;
constexpr int kGatherBK = 64;

// ---------------------------------------------------------------- carving
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long max_tiles_of(int T, int k, int E) {
  return (static_cast<long long>(T) * k + static_cast<long long>(kTileRows - 1) * E) / kTileRows;
}

struct SchedLayout {
  int32_t *cnt, *row0, *row_src, *slot_row, *tile_expert, *tile_row0, *tile_rows, *header, *hist, *pair_tile,
      *unit_group;
};

size_t carve_schedule(void* buf, int T, int k, int E, SchedLayout* L) {
  const long long mt = max_tiles_of(T, k, E);
  const long long n = static_cast<long long>(T) * k;
  const long long nchunks = (n + kSchedChunk - 1) / kSchedChunk;
  Carver c(buf);
  L->cnt = c.take<int32_t>(E);
  L->row0 = c.take<int32_t>(E + 1);
  L->row_src = c.take<int32_t>(mt * kTileRows);
  L->slot_row = c.take<int32_t>(n);
  L->tile_expert = c.take<int32_t>(mt);
  L->tile_row0 = c.take<int32_t>(mt);
  L->tile_rows = c.take<int32_t>(mt);
  L->header = c.take<int32_t>(8);
  L->pair_tile = c.take<int32_t>(2 * mt);
  L->unit_group = c.take<int32_t>(2 * mt);
  L->hist = c.take<int32_t>(nchunks * E);
  return c.off + 256;
}

struct CtxExtra {  // forward scratch beyond the public context fields
  // MXFP8 mode: weight scales in the tensor-core scale layout
  uint8_t *wg_sc, *wu_sc, *wd_sc, *wsg_sc, *wsu_sc, *wsd_sc;
  int32_t* view;      // macrobatch ring: the windows' schedule views
  int32_t* tickets;   // work-item counters of the GEMM launches
  uint8_t* xs;        // MXFP8 modes: the dispatch's scales of x, row-major [T][H/32]
};

// Work-item counters a call needs: one per TMA-fed GEMM launch, at most two
// (forward) or four (backward) routed GEMMs per window, windows at most E,
// plus the shared expert's.
int fwd_tickets(int E) { return 8 + 2 * E; }
int bwd_tickets(int E) { return 8 + 4 * E; }

// ---------------------------------------------------------------- macrobatch ring
// Rows of the ring for a macrobatch size: 0 (no ring: every schedule-order
// buffer spans all max_rows rows) for 0 or a size that holds every row, else
// the size rounded up to whole 128-row tiles.
long long ring_rows_of(long long macrobatch, long long max_rows) {
  if (macrobatch <= 0) return 0;
  const long long r = (macrobatch + kTileRows - 1) / kTileRows * kTileRows;
  return r >= max_rows ? 0 : r;
}

// Ints of the windows' schedule views: the tiles, pairs and work groups of all
// windows (max_tiles tiles at most), ne + 1 row offsets and an 8-int header
// per window (at most E windows).
long long view_ints(long long max_tiles, int E) { return 7 * max_tiles + 10ll * E; }

// Bytes of E8M0 scales of a [rows][K] tensor in the tensor-core scale layout
// (rows padded to whole 128-row blocks).
long long tiled_scale_bytes(long long rows, long long K) { return (rows + 127) / 128 * 128 * (K / 32); }

// The context: gu (saved) and slots (read by the combine) span every schedule
// row; the rest of the schedule-order scratch spans `ring` rows (0: every row).
size_t carve_ctx(void* buf, int T, int k, int E, int H, int I, int Is, int mode, long long ring, mok_ctx_t* ctx,
                 CtxExtra* X) {
  const long long mt = max_tiles_of(T, k, E);
  const long long mr = mt * kTileRows;
  const long long rr = ring ? ring : mr;
  const bool mx = (mode == MOK_MODE_MXFP8_FWD || mode == MOK_MODE_MXFP8);
  Carver c(buf);
  memset(ctx, 0, sizeof(*ctx));
  memset(X, 0, sizeof(*X));
  ctx->T = T; ctx->k = k; ctx->E = E; ctx->H = H; ctx->I = I; ctx->I_s = Is; ctx->mode = mode;
  ctx->max_tiles = static_cast<int>(mt);
  ctx->ring_rows = ring;
  ctx->status = c.take<int32_t>(8);
  ctx->gu = c.take<uint16_t>(mr * 2 * I);
  ctx->slots = c.take<uint16_t>(mr * H);
  if (!mx) {
    ctx->x_perm = c.take<uint16_t>(rr * H);
    ctx->h = c.take<uint16_t>(rr * I);
  } else {
    // the bf16 token rows in schedule order for the bf16 backward's gate/up
    // weight gradient, written during a one-pass forward (MXFP8 forward mode
    // only; a backward after a ring forward makes its own)
    if (mode == MOK_MODE_MXFP8_FWD && !ring) ctx->x_perm = c.take<uint16_t>(mr * H);
    ctx->xq = c.take<uint8_t>(static_cast<long long>(T) * H);
    ctx->xq_sc = c.take<uint8_t>(tiled_scale_bytes(T, H));
    X->xs = c.take<uint8_t>(static_cast<long long>(T) * (H / 32));
    ctx->xq_perm = c.take<uint8_t>(rr * H);
    ctx->xq_perm_sc = c.take<uint8_t>(tiled_scale_bytes(rr, H));
    ctx->hq = c.take<uint8_t>(rr * I);
    ctx->hq_sc = c.take<uint8_t>(tiled_scale_bytes(rr, I));
    // gate and up scales back to back: the CTA-pair 128-wide SwiGLU GEMM reads
    // the same bytes as one interleaved gate|up tensor of 2 E I rows
    X->wg_sc = c.take<uint8_t>(2 * tiled_scale_bytes(static_cast<long long>(E) * I, H));
    X->wu_sc = X->wg_sc ? X->wg_sc + tiled_scale_bytes(static_cast<long long>(E) * I, H) : nullptr;
    X->wd_sc = c.take<uint8_t>(tiled_scale_bytes(static_cast<long long>(E) * H, I));
  }
  if (Is > 0) {
    ctx->gu_s = c.take<uint16_t>(static_cast<long long>(T) * 2 * Is);
    ctx->shared_out = c.take<uint16_t>(static_cast<long long>(T) * H);
    if (!mx) {
      ctx->h_s = c.take<uint16_t>(static_cast<long long>(T) * Is);
    } else {
      ctx->hq_s = c.take<uint8_t>(static_cast<long long>(T) * Is);
      ctx->hq_s_sc = c.take<uint8_t>(tiled_scale_bytes(T, Is));
      X->wsg_sc = c.take<uint8_t>(2 * tiled_scale_bytes(Is, H));
      X->wsu_sc = X->wsg_sc ? X->wsg_sc + tiled_scale_bytes(Is, H) : nullptr;
      X->wsd_sc = c.take<uint8_t>(tiled_scale_bytes(H, Is));
    }
  }
  if (ring) X->view = c.take<int32_t>(view_ints(mt, E));
  X->tickets = c.take<int32_t>(fwd_tickets(E));
  return c.off + 256;
}

struct BwdLayout {
  uint16_t *dgu, *hw, *dgu_s, *hs, *dx_s, *dy_perm, *xb_perm;
  float* dw_part;
  // MOK_MODE_MXFP8: E4M3 operands of the backward GEMMs and their E8M0 scales
  // (tensor-core scale layout).  Row-quantised: dy (schedule and token order),
  // dG|dU.  Transposed (blocks along the rows): dy, x, dG|dU, w h, and the
  // shared expert's.  Weight scales of the caller's transposed copies.
  uint8_t *dyq, *dyq_sc, *dyq_tok, *dyq_tok_sc, *dyT, *dyT_sc, *dyT_tok, *dyT_tok_sc;
  uint8_t *xT, *xT_sc, *xT_tok, *xT_tok_sc, *dguq, *dguq_sc, *dguT, *dguT_sc, *hwT, *hwT_sc;
  uint8_t *dgusq, *dgusq_sc, *dgusT, *dgusT_sc, *hsT, *hsT_sc;
  uint8_t *wtg_sc, *wtu_sc, *wtd_sc, *wtsg_sc, *wtsu_sc, *wtsd_sc;
  int32_t* view;      // macrobatch ring: the windows' schedule views
  int32_t* tickets;   // work-item counters of the GEMM launches
};

int tile_n(int N) { return (N % 256 == 0) ? 256 : 128; }

// CTA pairs (M = 256 over two SMs sharing each B tile) for the 256-wide
// TMA-fed GEMMs, unless the caller turns them off.
bool pair_on(const mok_config_t* cfg, int bn) { return bn == 256 && !(cfg->debug_flags & MOK_DEBUG_NO_CTA_PAIR); }

// Work items per SM from which a row GEMM takes its items in ticket order.
// Over a long launch the CTAs of the static order drift apart and the
// operands they share fall out of L2 (at T=65536 the dgrad through gate/up
// read 58 GB per launch that way, 19.5 GB in ticket order, and ran 3%
// faster); on a short launch the hand-over of each item through the queue
// costs more than that (T=4096: 5-10% slower).  The weight gradients keep
// the static order at every size (in ticket order they read less but did
// not run faster).
constexpr long long kTicketItemsPerSm = 200;

// One TMA-fed GEMM as CTA pairs or as single CTAs; items / pair_items bound
// the work items of each form.
template <int A, int B, int BN, int EPI>
cudaError_t launch_tiles(const GemmMaps& m, const GemmParams& p, long long items, long long pair_items, bool pair,
                         int sms, cudaStream_t st) {
  GemmParams q = p;
  if (q.ticket_mode == 2 || (q.ticket_mode == 0 && !q.wgrad && items >= kTicketItemsPerSm * sms))
    q.ticket = next_ticket();
  if constexpr (BN == 256) {
    if (pair) return launch_gemm_pair<A, B, BN, EPI>(m, q, pair_items, st);
  }
  return launch_gemm<A, B, BN, EPI>(m, q, items < sms ? static_cast<int>(items) : sms, st);
}

// Pair work items: row tiles taken two at a time.
long long row_pairs(long long rows) { return ((rows + 127) / 128 + 1) / 2; }

// The backward workspace: dw_part (read by the fixed-order reduction) spans
// every routed row; the schedule-order scratch spans `ring` rows (0: every
// row).  The dx rows in schedule order go to the context's slots, the
// forward's scratch, which its combine has consumed.
size_t carve_bwd(void* buf, int T, int k, int E, int H, int I, int Is, int mode, long long ring, BwdLayout* L) {
  const long long mt = max_tiles_of(T, k, E);
  const long long mr = mt * kTileRows;
  const long long rr = ring ? ring : mr;
  const long long n = static_cast<long long>(T) * k;
  const long long Tl = T, Tp = (Tl + 127) / 128 * 128;
  const bool mx = (mode == MOK_MODE_MXFP8);
  Carver c(buf);
  memset(L, 0, sizeof(*L));
  if (!mx) {   // the MXFP8 backward keeps these only as E4M3 codes
    L->dgu = c.take<uint16_t>(rr * 2 * I);
    L->hw = c.take<uint16_t>(rr * I);
  }
  // two column halves per N tile (128-wide tiles in the MXFP8 backward)
  L->dw_part = c.take<float>(n * 2 * (I / (mx ? 128 : tile_n(I))));
  if (!mx) {
    L->dy_perm = c.take<uint16_t>(rr * H);
    // x's rows in schedule order: a one-pass MXFP8 forward leaves them in the
    // context; with a ring they are made window by window
    if (mode == MOK_MODE_BF16 || ring) L->xb_perm = c.take<uint16_t>(rr * H);
  }
  if (Is > 0) {
    if (!mx) {
      L->dgu_s = c.take<uint16_t>(Tl * 2 * Is);
      L->hs = c.take<uint16_t>(Tl * Is);
    }
    L->dx_s = c.take<uint16_t>(Tl * H);
  }
  if (mx) {
    L->dyq = c.take<uint8_t>(rr * H);
    L->dyq_sc = c.take<uint8_t>(tiled_scale_bytes(rr, H));
    L->dyq_tok = c.take<uint8_t>(Tp * H);   // rows up to the 128-row boundary (zeros past T)
    L->dyq_tok_sc = c.take<uint8_t>(tiled_scale_bytes(Tl, H));
    L->dyT = c.take<uint8_t>(rr * H);
    L->dyT_sc = c.take<uint8_t>(tiled_scale_bytes(H, rr));
    L->xT = c.take<uint8_t>(rr * H);
    L->xT_sc = c.take<uint8_t>(tiled_scale_bytes(H, rr));
    L->dguq = c.take<uint8_t>(rr * 2 * I);
    L->dguq_sc = c.take<uint8_t>(tiled_scale_bytes(rr, 2 * I));
    L->dguT = c.take<uint8_t>(rr * 2 * I);
    L->dguT_sc = c.take<uint8_t>(tiled_scale_bytes(2 * I, rr));
    L->hwT = c.take<uint8_t>(rr * I);
    L->hwT_sc = c.take<uint8_t>(tiled_scale_bytes(I, rr));
    L->wtg_sc = c.take<uint8_t>(tiled_scale_bytes(static_cast<long long>(E) * H, I));
    L->wtu_sc = c.take<uint8_t>(tiled_scale_bytes(static_cast<long long>(E) * H, I));
    L->wtd_sc = c.take<uint8_t>(tiled_scale_bytes(static_cast<long long>(E) * I, H));
    if (Is > 0) {
      L->dyT_tok = c.take<uint8_t>(Tp * H);
      L->dyT_tok_sc = c.take<uint8_t>(tiled_scale_bytes(H, Tp));
      L->xT_tok = c.take<uint8_t>(Tp * H);
      L->xT_tok_sc = c.take<uint8_t>(tiled_scale_bytes(H, Tp));
      L->dgusq = c.take<uint8_t>(Tl * 2 * Is);
      L->dgusq_sc = c.take<uint8_t>(tiled_scale_bytes(Tl, 2 * Is));
      L->dgusT = c.take<uint8_t>(Tp * 2 * Is);
      L->dgusT_sc = c.take<uint8_t>(tiled_scale_bytes(2 * Is, Tp));
      L->hsT = c.take<uint8_t>(Tp * Is);
      L->hsT_sc = c.take<uint8_t>(tiled_scale_bytes(Is, Tp));
      L->wtsg_sc = c.take<uint8_t>(tiled_scale_bytes(H, Is));
      L->wtsu_sc = c.take<uint8_t>(tiled_scale_bytes(H, Is));
      L->wtsd_sc = c.take<uint8_t>(tiled_scale_bytes(Is, H));
    }
  }
  if (ring) L->view = c.take<int32_t>(view_ints(mt, E));
  L->tickets = c.take<int32_t>(bwd_tickets(E));
  return c.off + 256;
}

mok_status_t check_shapes(int T, int k, int E, int H, int I, int Is) {
  if (T < 1 || k < 1 || k > 64 || E < 1 || E > 1024)
    return fail(MOK_ERR_INVALID_ARG, "need T >= 1, 1 <= k <= 64, 1 <= E <= 1024 (T=%d k=%d E=%d)", T, k, E);
  if (static_cast<long long>(T) * k >= (1ll << 31) - 128ll * E)
    return fail(MOK_ERR_INVALID_ARG, "T*k too large");
  if (H < 128 || H % 128 || I < 128 || I % 128 || Is < 0 || Is % 128)
    return fail(MOK_ERR_UNSUPPORTED, "need H, I (and I_s) multiples of 128 (H=%d I=%d I_s=%d)", H, I, Is);
  return MOK_OK;
}

// Work-item order: -1 lets the launch pick the L2-friendly order (see
// resolve_item_order), -2 keeps the plain order (MOK_DEBUG_PLAIN_ORDER);
// MOK_DEBUG_STATIC_ORDER / MOK_DEBUG_TICKET_ORDER keep every launch off the
// ticket counters / put every one on them.
GemmParams base_params(const mok_config_t* cfg, const mok_schedule_t* s, int* status, int debug) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  const int order = (cfg && (cfg->debug_flags & MOK_DEBUG_PLAIN_ORDER)) ? -2 : -1;
  p.group = order;
  p.wg_col_outer = order;
  p.ticket_mode = !cfg ? 0
                  : (cfg->debug_flags & MOK_DEBUG_STATIC_ORDER) ? 1
                  : (cfg->debug_flags & MOK_DEBUG_TICKET_ORDER) ? 2
                                                                 : 0;
  p.topk = s ? s->k : 1;
  if (s) {
    p.header = s->header;
    p.tile_expert = s->tile_expert;
    p.tile_row0 = s->tile_row0;
    p.tile_rows = s->tile_rows;
    p.row_src = s->row_src;
    p.row0 = s->row0;
    p.cnt = s->cnt;
    p.pair_tile = s->pair_tile;
    p.tile_group = s->unit_group;
    p.pair_group = s->unit_group ? s->unit_group + s->max_tiles : nullptr;
  }
  p.status = status;
  p.debug = debug;
  p.E = 1;
  return p;
}

// Windows of whole experts for a ring of `ring` rows ("Mixture-of-Kittens: a
// deterministic MoE megakernel for NVL72 racks", "Tuning the five
// hyperparameters before production": macrobatch_size): in expert order, each
// expert padded to whole 128-row tiles, a window takes the next expert while
// its rows fit the ring.  first[w] = window w's first expert, first.back() =
// E; ring 0: one window.  An expert larger than the ring: MOK_ERR_CAPACITY.
mok_status_t plan_windows(const int32_t* cnt, int E, long long ring, std::vector<int>* first) {
  first->assign(1, 0);
  long long used = 0;
  for (int e = 0; e < E; ++e) {
    if (cnt[e] < 0) return fail(MOK_ERR_INVALID_ARG, "expert %d has a negative row count", e);
    const long long padded = (static_cast<long long>(cnt[e]) + kTileRows - 1) / kTileRows * kTileRows;
    if (ring > 0 && padded > ring)
      return fail(MOK_ERR_CAPACITY, "expert %d has %lld padded rows; the macrobatch ring holds %lld", e, padded,
                  ring);
    if (ring > 0 && used + padded > ring) {
      first->push_back(e);
      used = 0;
    }
    used += padded;
  }
  first->push_back(E);
  return MOK_OK;
}

// One window of the routed experts: experts [e0, e0 + ne) and their schedule
// rows [r0, r0 + rows).  `s` is the schedule itself when one window covers it,
// else the window's view (launch_window_view): its own tile list, pairs, work
// groups and header, tile rows and row0 counted from r0, cnt and row_src
// offset to the window; s.max_tiles is then the window's tile count.  Tile
// experts stay absolute.
struct Win {
  mok_schedule_t s;
  int e0, ne;
  long long r0, rows;
};

// The windows of a call.  Without a ring: one window over the whole schedule
// (nothing is read back).  With one: the expert counts and the header are
// read back (synchronising cs), the windows planned, and each window's view
// built on cs into `view`.  A failed schedule gives no window: the routed
// kernels would do nothing, and the status travels on in the header.
mok_status_t make_windows(const mok_schedule_t* s, long long ring, int32_t* view, cudaStream_t cs,
                          std::vector<Win>* out) {
  out->clear();
  const long long mt = s->max_tiles;
  if (ring == 0) {
    out->push_back(Win{*s, 0, s->E, 0, mt * kTileRows});
    return MOK_OK;
  }
  const int E = s->E;
  std::vector<int32_t> cnt(E), hdr(8);
  MOK_CUDA(cudaMemcpyAsync(hdr.data(), s->header, 8 * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
  MOK_CUDA(cudaMemcpyAsync(cnt.data(), s->cnt, E * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
  MOK_CUDA(cudaStreamSynchronize(cs));
  if (hdr[2] != 0) return MOK_OK;
  std::vector<int> first;
  mok_status_t st = plan_windows(cnt.data(), E, ring, &first);
  if (st) return st;
  const int nw = static_cast<int>(first.size()) - 1;
  const int cap = hdr[5];
  long long r0 = 0, tile_off = 0, pair_off = 0;
  for (int w = 0; w < nw; ++w) {
    Win v;
    v.s = *s;
    v.e0 = first[w];
    v.ne = first[w + 1] - first[w];
    v.r0 = r0;
    long long tiles = 0, pairs = 0;
    for (int e = v.e0; e < v.e0 + v.ne; ++e) {
      const long long nt = (cnt[e] + kTileRows - 1) / kTileRows, prim = nt < cap ? nt : cap;
      tiles += nt;
      pairs += (prim + 1) / 2 + (nt - prim + 1) / 2;
    }
    v.rows = tiles * kTileRows;
    if (nw > 1) {
      int32_t* rows0 = view + 7 * mt + v.e0 + w;
      int32_t* header = view + 7 * mt + 2ll * E + 8ll * w;
      v.s.max_tiles = static_cast<int>(tiles);
      v.s.tile_expert = view + tile_off;
      v.s.tile_row0 = view + mt + tile_off;
      v.s.tile_rows = view + 2 * mt + tile_off;
      v.s.pair_tile = view + 3 * mt + 2 * pair_off;
      v.s.unit_group = view + 5 * mt + 2 * tile_off;   // the window's tile groups, then its pair groups
      v.s.row0 = rows0;
      v.s.header = header;
      v.s.cnt = s->cnt + v.e0;
      v.s.row_src = s->row_src + r0;
      v.s.scratch = nullptr;
      MOK_CUDA(launch_window_view(s->cnt, s->row0, s->header, v.e0, v.ne, v.s.tile_expert, v.s.tile_row0,
                                  v.s.tile_rows, v.s.pair_tile, v.s.unit_group, rows0, header, cs));
    }
    out->push_back(v);
    r0 += v.rows;
    tile_off += tiles;
    pair_off += pairs;
  }
  return MOK_OK;
}

// NVTX ranges (host timeline; they cost nothing unless a tool is attached):
// one per C-ABI call and one per stage inside it, so that a profiler can pick
// a call's or a stage's kernels (e.g. ncu --nvtx --nvtx-include "mok_backward/").
const char* const kStageNames[MOK_NUM_STAGES] = {
    "fwd_prep", "fwd_shared_gateup", "fwd_shared_down", "fwd_gateup", "fwd_down", "fwd_combine",
    "bwd_down", "bwd_wgrad_down", "bwd_wgrad_gateup", "bwd_dgrad_gateup", "bwd_shared_down",
    "bwd_shared_wgrad_down", "bwd_shared_wgrad_gateup", "bwd_shared_dgrad", "bwd_reduce",
    "fwd_dispatch", "bwd_dispatch"};
thread_local int g_nvtx_depth = 0;

// The call's range; on the way out it also closes stage ranges an early
// (error) return left open.
struct NvtxCall {
  int base;
  explicit NvtxCall(const char* name) : base(g_nvtx_depth) {
    nvtxRangePushA(name);
    ++g_nvtx_depth;
  }
  ~NvtxCall() {
    while (g_nvtx_depth > base) {
      nvtxRangePop();
      --g_nvtx_depth;
    }
  }
};

// Records the caller's timing event for the start (end = 0) or end of a stage
// (a NULL entry, or event = false: nothing), and opens or closes the stage's
// NVTX range.  With a macrobatch ring a routed stage runs once per window: its
// NVTX range opens and closes each time, its events are recorded at the start
// in the first window and the end in the last.
cudaError_t mark(const mok_config_t* cfg, int stage, int end, cudaStream_t st, bool event = true) {
  if (!end) {
    nvtxRangePushA(kStageNames[stage]);
    ++g_nvtx_depth;
  } else if (g_nvtx_depth > 0) {
    nvtxRangePop();
    --g_nvtx_depth;
  }
  if (event && cfg->events && cfg->num_events >= 2 * MOK_NUM_STAGES && cfg->events[2 * stage + end])
    return cudaEventRecord(static_cast<cudaEvent_t>(cfg->events[2 * stage + end]), st);
  return cudaSuccess;
}

mok_status_t check_config(const mok_config_t* cfg) {
  if (cfg->mode != MOK_MODE_BF16 && cfg->mode != MOK_MODE_MXFP8_FWD && cfg->mode != MOK_MODE_MXFP8)
    return fail(MOK_ERR_INVALID_ARG, "unknown mode %d", cfg->mode);
  if (cfg->events && cfg->num_events != 2 * MOK_NUM_STAGES)
    return fail(MOK_ERR_INVALID_ARG, "events needs 2 * MOK_NUM_STAGES entries");
  if (cfg->minibatch_size < 0) return fail(MOK_ERR_INVALID_ARG, "minibatch_size < 0");
  if (cfg->macrobatch_size < 0) return fail(MOK_ERR_INVALID_ARG, "macrobatch_size < 0");
  if (cfg->dispatch < MOK_DISPATCH_AUTO || cfg->dispatch > MOK_DISPATCH_FUSED)
    return fail(MOK_ERR_INVALID_ARG, "unknown dispatch %d", cfg->dispatch);
  if (!std::isfinite(cfg->swiglu_limit) || cfg->swiglu_limit < 0.f)
    return fail(MOK_ERR_INVALID_ARG, "swiglu_limit must be finite and >= 0");
  return MOK_OK;
}

int resolve_dispatch(const mok_config_t* cfg) {
  return cfg->dispatch == MOK_DISPATCH_FUSED ? MOK_DISPATCH_FUSED : MOK_DISPATCH_PERMUTE;
}

__global__ void propagate_status_kernel(const int* header, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  if (header[2] != 0) atomicCAS(status, 0, header[2]);
}

}  // namespace

namespace {

// ---------------------------------------------------------------------------
// Side stream for work that overlaps the caller's stream inside one call (the
// dispatch permutes): one per host thread and device, created on first use.
// Every call forks it from the caller's stream with an event and joins it back
// before the work that reads its results, so all of the call's work stays
// ordered after what precedes it on the caller's stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
  cudaEvent_t join2 = nullptr;   // a second hand-back point within one call
};
thread_local SideStream g_side[64];

// The work-item counters of the calling thread's current forward or backward
// call (zeroed at its start), handed out one per TMA-fed GEMM launch in
// launch order; the scope ends with the call.
struct TicketPool {
  int32_t* base = nullptr;
  int n = 0;
  int used = 0;
};
thread_local TicketPool g_tickets;
struct TicketScope {
  TicketScope(int32_t* base, int n) { g_tickets = TicketPool{base, n, 0}; }
  ~TicketScope() { g_tickets = TicketPool{}; }
};

mok_status_t side_stream(SideStream** out) {
  int dev = 0;
  MOK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOK_ERR_UNSUPPORTED, "device ordinal %d", dev);
  SideStream& sd = g_side[dev];
  if (!sd.s) {
    MOK_CUDA(cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking));
    MOK_CUDA(cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming));
    MOK_CUDA(cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming));
    MOK_CUDA(cudaEventCreateWithFlags(&sd.join2, cudaEventDisableTiming));
  }
  *out = &sd;
  return MOK_OK;
}

}  // namespace

int* mok::next_ticket() {
  if (!g_tickets.base || g_tickets.used >= g_tickets.n) return nullptr;
  return g_tickets.base + g_tickets.used++;
}


// ---------------------------------------------------------------------------
// Scratch for mok_schedule_noalloc: per-chunk expert histograms live in this
// file-scope device array instead of the caller's buffer.  Every GPU that
// loads the library holds it until the process exits.
constexpr long long kStaticSchedScratchInts = 1ll << 20;  // 4 MiB
static __device__ __align__(256) int32_t g_sched_scratch[kStaticSchedScratchInts];

namespace {
int32_t* g_sched_scratch_dev[64] = {};
std::mutex g_sched_scratch_mu;

// Device address of g_sched_scratch on the current device, looked up once per
// device (host code may not use the symbol itself as a device pointer).
mok_status_t static_sched_scratch(int32_t** out) {
  int dev = 0;
  MOK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOK_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_sched_scratch_mu);
  if (!g_sched_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_sched_scratch);
    if (e != cudaSuccess || !p)
      return fail(MOK_ERR_CUDA, "cudaGetSymbolAddress(schedule scratch) failed: %s", cudaGetErrorString(e));
    g_sched_scratch_dev[dev] = static_cast<int32_t*>(p);
  }
  *out = g_sched_scratch_dev[dev];
  return MOK_OK;
}
}  // namespace

namespace {

// Events for the routed stages of a forward or backward that found no window
// (a failed schedule under a ring): each recorded back to back.
cudaError_t mark_skipped(const mok_config_t* cfg, std::initializer_list<int> stages, cudaStream_t cs) {
  for (int sg : stages) {
    cudaError_t e = mark(cfg, sg, 0, cs);
    if (e == cudaSuccess) e = mark(cfg, sg, 1, cs);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// BF16 forward: shared expert, then the routed experts window by window (token
// rows of x permuted into schedule order, or gathered inside the GEMM).
mok_status_t forward_bf16(const mok_config_t* cfg, const uint16_t* x, const float* router_w, const mok_schedule_t* s,
                          const std::vector<Win>& wins, const mok_weights_t* w, mok_ctx_t* ctx, int sms, bool g4,
                          cudaStream_t cs) {
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  const size_t nw = wins.size();
  mok_status_t st;
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_PREP, 1, cs));
  const int disp = resolve_dispatch(cfg);
  ctx->dispatch = disp;
  const bool perm = disp == MOK_DISPATCH_PERMUTE;
  auto permute = [&](const Win& v, cudaStream_t st2) {
    return launch_permute_rows(x, T, H, k, s->slot_row, s->row_src, s->header, v.r0, v.rows, ctx->x_perm, sms, st2);
  };
  // token rows of x in schedule order (read by the routed gate/up GEMM as
  // dense tiles); the first window's are written on a side stream while the
  // shared expert runs
  SideStream* side = nullptr;
  if (perm && nw > 0) {
    if ((st = side_stream(&side))) return st;
    MOK_CUDA(cudaEventRecord(side->fork, cs));
    MOK_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 0, side->s));
    MOK_CUDA(permute(wins[0], side->s));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 1, side->s, nw == 1));
    MOK_CUDA(cudaEventRecord(side->join, side->s));
  } else {
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_FWD_DISPATCH}, cs));
  }

  // ---- shared expert: gate/up + SwiGLU over all T tokens, then down
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 0, cs));
  if (Is > 0) {
    GemmMaps m;
    if ((st = make_map(&m.a, x, H, T, 128, kTileBK)) || (st = make_map(&m.b0, w->ws_gate, H, Is, 128, kTileBK)) ||
        (st = make_map(&m.b1, w->ws_up, H, Is, 128, kTileBK)))
      return st;
    if ((st = make_map_out(&m.o0, ctx->gu_s, 2ull * Is, T)) || (st = make_map_out(&m.o1, ctx->h_s, Is, T))) return st;
    GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
    p.rows = T; p.K = H; p.N = Is; p.n_tiles = Is / 128; p.b_rows_per_expert = 0;
    p.out0 = ctx->gu_s; p.out1 = ctx->h_s;
    p.swiglu_limit = cfg->swiglu_limit;
    const long long items = ((T + 127) / 128) * static_cast<long long>(p.n_tiles);
    MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 256, EPI_SWIGLU>(m, p, items, row_pairs(T) * p.n_tiles,
                                                                     pair_on(cfg, 256), sms, cs)));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 1, cs));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 0, cs));
    GemmMaps m2;
    const int bn = tile_n(H);
    const bool pr = pair_on(cfg, bn);
    if ((st = make_map(&m2.a, ctx->h_s, Is, T, 128, kTileBK)) ||
        (st = make_map(&m2.b0, w->ws_down, Is, H, pr ? bn / 2 : bn, kTileBK)) ||
        (st = make_map_out(&m2.o0, ctx->shared_out, H, T)))
      return st;
    m2.b1 = m2.b0;
    GemmParams q = base_params(cfg, nullptr, ctx->status, 0);
    q.rows = T; q.K = Is; q.N = H; q.n_tiles = H / bn; q.out0 = ctx->shared_out; q.ld = H;
    const long long items2 = ((T + 127) / 128) * static_cast<long long>(q.n_tiles);
    if (bn == 256)
      MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 256, EPI_STORE_ROWS>(m2, q, items2, row_pairs(T) * q.n_tiles, pr,
                                                                          sms, cs)));
    else
      MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 128, EPI_STORE_ROWS>(m2, q, items2, 0, false, sms, cs)));
  } else {
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 1, cs));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 0, cs));
  }
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 1, cs));

  // ---- routed experts, window by window: gate/up + SwiGLU, then down +
  // scale + scatter (h and the token rows span the window; gu and the slots
  // every row)
  if (side) MOK_CUDA(cudaStreamWaitEvent(cs, side->join, 0));
  if (nw == 0) MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_FWD_GATEUP, MOK_STAGE_FWD_DOWN}, cs));
  for (size_t i = 0; i < nw; ++i) {
    const Win& v = wins[i];
    const bool first = i == 0, last = i + 1 == nw;
    if (perm && !first) {
      MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 0, cs, false));
      MOK_CUDA(permute(v, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 1, cs, last));
    }
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_GATEUP, 0, cs, first));
    uint16_t* gu = ctx->gu + v.r0 * 2 * I;
    GemmMaps m;
    const int bk = perm ? kTileBK : kGatherBK;
    if ((st = perm ? make_map(&m.a, ctx->x_perm, H, v.rows, 128, bk) : make_map(&m.a, x, H, T, 1, bk)) ||
        (st = make_map(&m.b0, w->w_gate, H, static_cast<uint64_t>(E) * I, 128, bk)) ||
        (st = make_map(&m.b1, w->w_up, H, static_cast<uint64_t>(E) * I, 128, bk)) ||
        (st = make_map_out(&m.o0, gu, 2ull * I, v.rows)) || (st = make_map_out(&m.o1, ctx->h, I, v.rows)))
      return st;
    GemmParams p = base_params(cfg, &v.s, ctx->status, cfg->debug_flags);
    p.grouped = 1; p.K = H; p.N = I; p.n_tiles = I / 128; p.b_rows_per_expert = I;
    p.out0 = gu; p.out1 = ctx->h; p.ga = x; p.ga_ld = H;
    p.swiglu_limit = cfg->swiglu_limit;
    const long long items = static_cast<long long>(v.s.max_tiles) * p.n_tiles;
    const int grid = items < sms ? static_cast<int>(items) : sms;
    if (perm)
      MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 256, EPI_SWIGLU>(m, p, items, items, pair_on(cfg, 256), sms, cs)));
    else if (g4)
      MOK_CUDA((launch_gemm<SRC_K_GATHER, SRC_K_TILE, 256, EPI_SWIGLU>(m, p, grid, cs)));
    else
      MOK_CUDA((launch_gemm<SRC_K_GATHER_LSU, SRC_K_TILE, 256, EPI_SWIGLU>(m, p, grid, cs)));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_GATEUP, 1, cs, last));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DOWN, 0, cs, first));
    uint16_t* slots = ctx->slots + v.r0 * H;
    GemmMaps m2;
    const int bn = tile_n(H);
    const bool pr = pair_on(cfg, bn);
    if ((st = make_map(&m2.a, ctx->h, I, v.rows, 128, kTileBK)) ||
        (st = make_map(&m2.b0, w->w_down, I, static_cast<uint64_t>(E) * H, pr ? bn / 2 : bn, kTileBK)) ||
        (st = make_map_out(&m2.o0, slots, H, v.rows)))
      return st;
    m2.b1 = m2.b0;
    GemmParams q = base_params(cfg, &v.s, ctx->status, 0);
    q.grouped = 1; q.K = I; q.N = H; q.n_tiles = H / bn; q.b_rows_per_expert = H;
    q.out0 = slots; q.ld = H; q.rw = router_w;
    const long long items2 = static_cast<long long>(v.s.max_tiles) * q.n_tiles;
    if (bn == 256)
      MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 256, EPI_SCALE_ROWS>(m2, q, items2, items2, pr, sms, cs)));
    else
      MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_K_TILE, 128, EPI_SCALE_ROWS>(m2, q, items2, 0, false, sms, cs)));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DOWN, 1, cs, last));
  }
  return MOK_OK;
}

// MXFP8 forward: x quantised straight into token order (shared expert) and
// schedule order (routed experts, one window at a time), weight scales
// rearranged for the tensor core, then the same four GEMMs on the
// block-scaled MMA; h is requantised in the SwiGLU epilogue.
mok_status_t forward_mxfp8(const mok_config_t* cfg, const uint16_t* x, const float* router_w,
                           const mok_schedule_t* s, const std::vector<Win>& wins, const mok_weights_t* w,
                           mok_ctx_t* ctx, const CtxExtra& X, int sms, cudaStream_t cs) {
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  const size_t nw = wins.size();
  mok_status_t st;
  // Tiling of the block-scaled GEMMs: single CTAs with 256-wide tiles (the
  // accumulator single-buffered beside the scale ring), or CTA pairs (M = 256)
  // with 256-wide tiles (single-buffered) or 128-wide tiles (double-buffered;
  // the gate/up weights' scales then go into the interleaved gate|up layout).
  const int tiling = (cfg->debug_flags & MOK_DEBUG_MX_CTA_PAIR) ? 1 : (cfg->debug_flags & MOK_DEBUG_MX_PAIR128) ? 2 : 0;
  // weight scales into the tensor-core layout on a side stream, while x is
  // quantised once per token into token order and schedule order
  SideStream* side = nullptr;
  if ((st = side_stream(&side))) return st;
  MOK_CUDA(cudaEventRecord(side->fork, cs));
  MOK_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
  {
    const long long sr = Is > 0 ? 1 : 0;   // the shared expert's jobs are skipped without one
    const int gu = tiling == 2 ? 1 : 0;    // interleaved gate|up scales for the 128-wide pairs
    const MxTileScaleJob jobs[] = {
        {w->mx_gate_sc, static_cast<long long>(E) * I, H, X.wg_sc, gu, I},
        {w->mx_up_sc, static_cast<long long>(E) * I, H, gu ? X.wg_sc : X.wu_sc, 2 * gu, I},
        {w->mx_down_sc, static_cast<long long>(E) * H, I, X.wd_sc, 0, 0},
        {w->mxs_gate_sc, sr * Is, H, X.wsg_sc, gu, Is},
        {w->mxs_up_sc, sr * Is, H, gu ? X.wsg_sc : X.wsu_sc, 2 * gu, Is},
        {w->mxs_down_sc, sr * H, Is, X.wsd_sc, 0, 0}};
    MOK_CUDA(launch_mx_tile_scales(jobs, 6, side->s));
  }
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_PREP, 1, side->s));
  MOK_CUDA(cudaEventRecord(side->join, side->s));
  ctx->dispatch = MOK_DISPATCH_PERMUTE;
  // MXFP8 forward / bf16 backward without a ring: the same pass also writes
  // x's bf16 rows in schedule order, which the backward's gate/up weight
  // gradient reads (a separate copy would contend for HBM with whichever GEMM
  // it overlapped).  Later windows skip the token-order copy.
  auto dispatch = [&](const Win& v, bool tokens) {
    cudaError_t e = launch_mx_dispatch(x, T, H, k, s->slot_row, s->row_src, s->header, v.r0, v.rows,
                                       tokens ? ctx->xq : nullptr, X.xs, ctx->xq_perm, ctx->x_perm, sms, cs);
    if (e != cudaSuccess) return e;
    return launch_mx_scale_gather(X.xs, T, H, k, s->row_src, s->header, v.r0, v.rows, ctx->xq_perm_sc,
                                  tokens ? ctx->xq_sc : nullptr, cs);
  };
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 0, cs));
  if (nw > 0) MOK_CUDA(dispatch(wins[0], true));
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 1, cs, nw <= 1));
  MOK_CUDA(cudaStreamWaitEvent(cs, side->join, 0));

  const int bn = tile_n(H);
  // per-CTA B rows of a gate/up tile (gate rows, then up rows, for single
  // CTAs; one CTA of a pair holds the gate rows, the other the up rows)
  const int gu_box = tiling == 2 ? 64 : 128;
  const int gu_cols = tiling == 2 ? 64 : 128;          // h columns per gate/up tile
  // down tiles: width and per-CTA B rows
  const int dn_bn = tiling == 2 ? 128 : bn;
  const bool dn_pair = tiling == 2 || (tiling == 1 && bn == 256);
  const int dn_box = dn_pair ? dn_bn / 2 : dn_bn;
  const long long t_atoms = (T + 127) / 128;   // 128-row blocks
  // gate|up scale maps: two tensors, or one interleaved tensor of 2 * rows
  auto gu_sf_maps = [&](MxMaps& m, const uint8_t* g_sc, const uint8_t* u_sc, long long rows) -> mok_status_t {
    mok_status_t r;
    if (tiling == 2) {
      if ((r = make_map_sf(&m.sfb0, g_sc, (2 * rows / 128) * (H / 128)))) return r;
      m.sfb1 = m.sfb0;
      return MOK_OK;
    }
    if ((r = make_map_sf(&m.sfb0, g_sc, (rows / 128) * (H / 128)))) return r;
    return make_map_sf(&m.sfb1, u_sc, (rows / 128) * (H / 128));
  };
  auto launch_gu = [&](const MxMaps& m, const GemmParams& p, long long items, long long pair_items) -> cudaError_t {
    if (tiling == 2) return launch_gemm_mx_pair<128, EPI_SWIGLU_MX>(m, p, pair_items, cs);
    if (tiling == 1) return launch_gemm_mx_pair<256, EPI_SWIGLU_MX>(m, p, pair_items, cs);
    return launch_gemm_mx<256, EPI_SWIGLU_MX>(m, p, items < sms ? static_cast<int>(items) : sms, cs);
  };
  auto launch_dn = [&](int EPI_tag, const MxMaps& m, const GemmParams& p, long long items,
                       long long pair_items) -> cudaError_t {
    const int grid = items < sms ? static_cast<int>(items) : sms;
    if (EPI_tag == EPI_SCALE_ROWS) {
      if (dn_pair) return dn_bn == 128 ? launch_gemm_mx_pair<128, EPI_SCALE_ROWS>(m, p, pair_items, cs)
                                       : launch_gemm_mx_pair<256, EPI_SCALE_ROWS>(m, p, pair_items, cs);
      return bn == 256 ? launch_gemm_mx<256, EPI_SCALE_ROWS>(m, p, grid, cs)
                       : launch_gemm_mx<128, EPI_SCALE_ROWS>(m, p, grid, cs);
    }
    if (dn_pair) return dn_bn == 128 ? launch_gemm_mx_pair<128, EPI_STORE_ROWS>(m, p, pair_items, cs)
                                     : launch_gemm_mx_pair<256, EPI_STORE_ROWS>(m, p, pair_items, cs);
    return bn == 256 ? launch_gemm_mx<256, EPI_STORE_ROWS>(m, p, grid, cs)
                     : launch_gemm_mx<128, EPI_STORE_ROWS>(m, p, grid, cs);
  };
  // ---- shared expert
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 0, cs));
  if (Is > 0) {
    MxMaps m;
    if ((st = make_map_u8(&m.a, ctx->xq, H, T, 128)) || (st = make_map_u8(&m.b0, w->mxs_gate, H, Is, gu_box)) ||
        (st = make_map_u8(&m.b1, w->mxs_up, H, Is, gu_box)) ||
        (st = make_map_sf(&m.sfa, ctx->xq_sc, t_atoms * (H / 128))) || (st = gu_sf_maps(m, X.wsg_sc, X.wsu_sc, Is)) ||
        (st = make_map_out(&m.o0, ctx->gu_s, 2ull * Is, T)) || (st = make_map_codes_out(&m.o1, ctx->hq_s, Is, T)))
      return st;
    GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
    p.rows = T; p.K = H; p.N = Is; p.n_tiles = Is / gu_cols; p.b_rows_per_expert = 0;
    p.out0 = ctx->gu_s; p.out1 = ctx->hq_s; p.sf_out = ctx->hq_s_sc;
    p.swiglu_limit = cfg->swiglu_limit;
    p.sfa = ctx->xq_sc; p.sfb0 = X.wsg_sc; p.sfb1 = X.wsu_sc;
    const long long items = ((T + 127) / 128) * static_cast<long long>(p.n_tiles);
    MOK_CUDA(launch_gu(m, p, items, row_pairs(T) * p.n_tiles));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 1, cs));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 0, cs));
    MxMaps m2;
    if ((st = make_map_u8(&m2.a, ctx->hq_s, Is, T, 128)) || (st = make_map_u8(&m2.b0, w->mxs_down, Is, H, dn_box)) ||
        (st = make_map_sf(&m2.sfa, ctx->hq_s_sc, t_atoms * (Is / 128))) ||
        (st = make_map_sf(&m2.sfb0, X.wsd_sc, (H / 128) * (Is / 128))) ||
        (st = make_map_out(&m2.o0, ctx->shared_out, H, T)))
      return st;
    m2.b1 = m2.b0;
    m2.sfb1 = m2.sfb0;
    GemmParams q = base_params(cfg, nullptr, ctx->status, 0);
    q.rows = T; q.K = Is; q.N = H; q.n_tiles = H / dn_bn; q.out0 = ctx->shared_out; q.ld = H;
    q.sfa = ctx->hq_s_sc; q.sfb0 = X.wsd_sc;
    const long long items2 = ((T + 127) / 128) * static_cast<long long>(q.n_tiles);
    MOK_CUDA(launch_dn(EPI_STORE_ROWS, m2, q, items2, row_pairs(T) * q.n_tiles));
  } else {
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_GATEUP, 1, cs));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 0, cs));
  }
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_SHARED_DOWN, 1, cs));

  // ---- routed experts, window by window (the codes of x and h span the
  // window; gu and the slots every row)
  if (nw == 0) MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_FWD_GATEUP, MOK_STAGE_FWD_DOWN}, cs));
  for (size_t i = 0; i < nw; ++i) {
    const Win& v = wins[i];
    const bool first = i == 0, last = i + 1 == nw;
    const long long r_atoms = v.rows / 128;
    if (!first) {
      MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 0, cs, false));
      MOK_CUDA(dispatch(v, false));
      MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DISPATCH, 1, cs, last));
    }
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_GATEUP, 0, cs, first));
    uint16_t* gu = ctx->gu + v.r0 * 2 * I;
    MxMaps m;
    if ((st = make_map_u8(&m.a, ctx->xq_perm, H, v.rows, 128)) ||
        (st = make_map_u8(&m.b0, w->mx_gate, H, static_cast<uint64_t>(E) * I, gu_box)) ||
        (st = make_map_u8(&m.b1, w->mx_up, H, static_cast<uint64_t>(E) * I, gu_box)) ||
        (st = make_map_sf(&m.sfa, ctx->xq_perm_sc, r_atoms * (H / 128))) ||
        (st = gu_sf_maps(m, X.wg_sc, X.wu_sc, static_cast<long long>(E) * I)) ||
        (st = make_map_out(&m.o0, gu, 2ull * I, v.rows)) || (st = make_map_codes_out(&m.o1, ctx->hq, I, v.rows)))
      return st;
    GemmParams p = base_params(cfg, &v.s, ctx->status, cfg->debug_flags);
    p.grouped = 1; p.K = H; p.N = I; p.n_tiles = I / gu_cols; p.b_rows_per_expert = I;
    p.out0 = gu; p.out1 = ctx->hq; p.sf_out = ctx->hq_sc;
    p.swiglu_limit = cfg->swiglu_limit;
    p.sfa = ctx->xq_perm_sc; p.sfb0 = X.wg_sc; p.sfb1 = X.wu_sc;
    const long long items = static_cast<long long>(v.s.max_tiles) * p.n_tiles;
    MOK_CUDA(launch_gu(m, p, items, items));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_GATEUP, 1, cs, last));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DOWN, 0, cs, first));
    uint16_t* slots = ctx->slots + v.r0 * H;
    MxMaps m2;
    if ((st = make_map_u8(&m2.a, ctx->hq, I, v.rows, 128)) ||
        (st = make_map_u8(&m2.b0, w->mx_down, I, static_cast<uint64_t>(E) * H, dn_box)) ||
        (st = make_map_sf(&m2.sfa, ctx->hq_sc, r_atoms * (I / 128))) ||
        (st = make_map_sf(&m2.sfb0, X.wd_sc, (static_cast<long long>(E) * H / 128) * (I / 128))) ||
        (st = make_map_out(&m2.o0, slots, H, v.rows)))
      return st;
    m2.b1 = m2.b0;
    m2.sfb1 = m2.sfb0;
    GemmParams q = base_params(cfg, &v.s, ctx->status, 0);
    q.grouped = 1; q.K = I; q.N = H; q.n_tiles = H / dn_bn; q.b_rows_per_expert = H;
    q.out0 = slots; q.ld = H; q.rw = router_w;
    q.sfa = ctx->hq_sc; q.sfb0 = X.wd_sc;
    const long long items2 = static_cast<long long>(v.s.max_tiles) * q.n_tiles;
    MOK_CUDA(launch_dn(EPI_SCALE_ROWS, m2, q, items2, items2));
    MOK_CUDA(mark(cfg, MOK_STAGE_FWD_DOWN, 1, cs, last));
  }
  return MOK_OK;
}

// One block-scaled GEMM on single CTAs: BN = 256 when the output width allows.
template <int EPI>
cudaError_t launch_mx_tiles(const MxMaps& m, const GemmParams& p, int bn, long long items, int sms,
                            cudaStream_t st) {
  const int grid = items < sms ? static_cast<int>(items) : sms;
  if (bn == 256) return launch_gemm_mx<256, EPI>(m, p, grid, st);
  return launch_gemm_mx<128, EPI>(m, p, grid, st);
}

// MXFP8 backward (MOK_MODE_MXFP8): the eight backward GEMMs on the
// block-scaled MMA, each operand quantised along that GEMM's contraction axis.
//   dgrad through down    A = dy rows (along H)            B = W_down^T (along H)
//   weight gradients      A, B = transposes of the row operands (along rows)
//   dgrad through gate/up A = dG|dU rows (along I)          B = W_gate^T | W_up^T (along I)
// dy and x are quantised here (rows, and transposed through the schedule);
// the SwiGLU backward's epilogue writes dG|dU (rows and transposed) and w h
// (transposed) straight as E4M3 codes, quantised from their bf16 values.
mok_status_t backward_mxfp8(const mok_config_t* cfg, const uint16_t* dy, const uint16_t* x, const float* router_w,
                            const mok_schedule_t* s, const std::vector<Win>& wins, const mok_ctx_t* ctx,
                            const mok_weights_t* w, uint16_t* dx, float* d_router_w, const mok_weight_grads_t* g,
                            const BwdLayout& L, int sms, cudaStream_t cs) {
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  const long long mr = static_cast<long long>(s->max_tiles) * kTileRows;
  const int Tp = (T + 127) / 128 * 128;
  const size_t nw = wins.size();
  mok_status_t st;
  // a window's x (transposed) and dy (rows and transposed), through the
  // schedule: its rows from 0 of the workspace's codes
  auto quant_x = [&](const Win& v, cudaStream_t st2) {
    const int rows = static_cast<int>(v.rows);
    return launch_mx_quantize_t(x, H, 1, rows, H, rows, v.s.row_src, k, s->header, L.xT, L.xT_sc, 1, sms, st2);
  };
  auto quant_dy = [&](const Win& v) {
    const int rows = static_cast<int>(v.rows);
    return launch_mx_quantize_t(dy, H, 1, rows, H, rows, v.s.row_src, k, s->header, L.dyT, L.dyT_sc, 1, sms, cs,
                                L.dyq, L.dyq_sc, 1);
  };
  // ---- on the side stream: weight scales into the tensor-core layout (one
  // launch, handed back at `join`), then the transposed x,
  // which only the gate/up weight gradients read (handed back at `join2`)
  SideStream* side = nullptr;
  if ((st = side_stream(&side))) return st;
  MOK_CUDA(cudaEventRecord(side->fork, cs));
  MOK_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
  {
    const long long sr = Is > 0 ? 1 : 0;   // the shared expert's jobs are skipped without one
    const MxTileScaleJob jobs[] = {
        {w->mxts_gate_sc, sr * H, Is, L.wtsg_sc},
        {w->mxts_up_sc, sr * H, Is, L.wtsu_sc},
        {w->mxts_down_sc, sr * Is, H, L.wtsd_sc},
        {w->mxt_gate_sc, static_cast<long long>(E) * H, I, L.wtg_sc},
        {w->mxt_up_sc, static_cast<long long>(E) * H, I, L.wtu_sc},
        {w->mxt_down_sc, static_cast<long long>(E) * I, H, L.wtd_sc}};
    MOK_CUDA(launch_mx_tile_scales(jobs, 6, side->s));
  }
  MOK_CUDA(cudaEventRecord(side->join, side->s));
  if (Is > 0)
    MOK_CUDA(launch_mx_quantize_t(x, H, 1, Tp, H, T, nullptr, 1, nullptr, L.xT_tok, L.xT_tok_sc, 1, sms, side->s));
  if (nw > 0) MOK_CUDA(quant_x(wins[0], side->s));
  MOK_CUDA(cudaEventRecord(side->join2, side->s));
  // ---- dy, rows and transposed from one read: in schedule order (routed,
  // the first window) and in token order (shared expert)
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 0, cs));
  if (nw > 0) MOK_CUDA(quant_dy(wins[0]));
  if (Is > 0)
    MOK_CUDA(launch_mx_quantize_t(dy, H, 1, Tp, H, T, nullptr, 1, nullptr, L.dyT_tok, L.dyT_tok_sc, 1, sms, cs,
                                  L.dyq_tok, L.dyq_tok_sc, 1));
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 1, cs, nw <= 1));
  MOK_CUDA(cudaStreamWaitEvent(cs, side->join, 0));
  const int bnH = tile_n(H);

  // ---- shared expert (dense rows, w = 1)
  if (Is > 0) {
    const int bnS = tile_n(Is);
    {  // dgrad through down + SwiGLU backward
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DOWN, 0, cs));
      // its epilogue writes dG|dU by rows (for the dgrad) and transposed (weight
      // gradient), and h transposed, all as E4M3 codes
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dyq_tok, H, T, 128)) || (st = make_map_u8(&m.b0, w->mxts_down, H, Is, 128)) ||
          (st = make_map_codes_out(&m.o0, L.dgusq, 2ull * Is, T)) ||
          (st = make_map_codes_out(&m.o1, L.dgusT, Tp, 2ull * Is)) || (st = make_map_codes_out(&m.o2, L.hsT, Tp, Is)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.rows = T; p.K = H; p.N = Is; p.n_tiles = Is / 128; p.b_rows_per_expert = 0;
      p.aux0 = ctx->gu_s; p.swiglu_limit = ctx->swiglu_limit;
      p.sf_out = L.dgusq_sc; p.out2 = L.dgusT_sc; p.sf_out2 = L.hsT_sc; p.ld = Tp;   // codes: maps o0..o2
      p.sfa = L.dyq_tok_sc; p.sfb0 = L.wtsd_sc;
      const long long items = static_cast<long long>(Tp / 128) * p.n_tiles;
      MOK_CUDA((launch_gemm_mx<128, EPI_DOWN_BWD_MX>(m, p, items < sms ? static_cast<int>(items) : sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DOWN, 1, cs));
    }
    {  // dW_s_down = dy^T h_s
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_DOWN, 0, cs));
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dyT_tok, Tp, H, 128)) || (st = make_map_u8(&m.b0, L.hsT, Tp, Is, bnS)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.wgrad = 1; p.rows = T; p.K = Tp; p.E = 1; p.m_tiles = H / 128; p.n_tiles = Is / bnS;
      p.out0 = g->d_ws_down; p.out1 = g->d_ws_down; p.ld = Is; p.split = H;
      p.sfa = L.dyT_tok_sc; p.sfb0 = L.hsT_sc;
      MOK_CUDA(launch_mx_tiles<EPI_WGRAD>(m, p, bnS, static_cast<long long>(p.m_tiles) * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_DOWN, 1, cs));
    }
    MOK_CUDA(cudaStreamWaitEvent(cs, side->join2, 0));   // the transposed x is ready
    {  // dW_s_gate|up = (dG_s|dU_s)^T x
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_GATEUP, 0, cs));
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dgusT, Tp, 2ull * Is, 128)) || (st = make_map_u8(&m.b0, L.xT_tok, Tp, H, bnH)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.wgrad = 1; p.rows = T; p.K = Tp; p.E = 1; p.m_tiles = 2 * Is / 128; p.n_tiles = H / bnH;
      p.out0 = g->d_ws_gate; p.out1 = g->d_ws_up; p.ld = H; p.split = Is;
      p.sfa = L.dgusT_sc; p.sfb0 = L.xT_tok_sc;
      MOK_CUDA(launch_mx_tiles<EPI_WGRAD>(m, p, bnH, static_cast<long long>(p.m_tiles) * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_GATEUP, 1, cs));
    }
    {  // dx_s = dG_s W_s_gate + dU_s W_s_up
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DGRAD, 0, cs));
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dgusq, 2ull * Is, T, 128)) || (st = make_map_u8(&m.b0, w->mxts_gate, Is, H, bnH)) ||
          (st = make_map_u8(&m.b1, w->mxts_up, Is, H, bnH)) || (st = make_map_out(&m.o0, L.dx_s, H, T)))
        return st;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.rows = T; p.K = 2 * Is; p.N = H; p.n_tiles = H / bnH; p.b_rows_per_expert = 0; p.b_split = Is;
      p.out0 = L.dx_s; p.ld = H;
      p.sfa = L.dgusq_sc; p.sfb0 = L.wtsg_sc; p.sfb1 = L.wtsu_sc; p.sf_kgb = Is / 128;
      MOK_CUDA(launch_mx_tiles<EPI_STORE_ROWS>(m, p, bnH, static_cast<long long>(Tp / 128) * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DGRAD, 1, cs));
    }
  } else {
    for (int sg = MOK_STAGE_BWD_SHARED_DOWN; sg <= MOK_STAGE_BWD_SHARED_DGRAD; ++sg) {
      MOK_CUDA(mark(cfg, sg, 0, cs));
      MOK_CUDA(mark(cfg, sg, 1, cs));
    }
    MOK_CUDA(cudaStreamWaitEvent(cs, side->join2, 0));   // the transposed x is ready
  }

  // ---- routed, window by window (the codes span the window; the dx rows
  // and the router-weight partials every row)
  if (nw == 0)
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_BWD_DOWN, MOK_STAGE_BWD_WGRAD_DOWN, MOK_STAGE_BWD_WGRAD_GATEUP,
                                MOK_STAGE_BWD_DGRAD_GATEUP}, cs));
  for (size_t i = 0; i < nw; ++i) {
    const Win& v = wins[i];
    const bool first = i == 0, last = i + 1 == nw;
    const int rows = static_cast<int>(v.rows);
    if (!first) {
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 0, cs, false));
      MOK_CUDA(quant_dy(v));
      MOK_CUDA(quant_x(v, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 1, cs, last));
    }
    {  // dgrad through down + SwiGLU backward + router-weight partials
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DOWN, 0, cs, first));
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dyq, H, v.rows, 128)) ||
          (st = make_map_u8(&m.b0, w->mxt_down, H, static_cast<uint64_t>(E) * I, 128)) ||
          (st = make_map_codes_out(&m.o0, L.dguq, 2ull * I, v.rows)) ||
          (st = make_map_codes_out(&m.o1, L.dguT, v.rows, 2ull * I)) ||
          (st = make_map_codes_out(&m.o2, L.hwT, v.rows, I)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.grouped = 1; p.K = H; p.N = I; p.n_tiles = I / 128; p.b_rows_per_expert = I;
      p.aux0 = ctx->gu + v.r0 * 2 * I; p.rw = router_w; p.dw_part = L.dw_part; p.swiglu_limit = ctx->swiglu_limit;
      p.sf_out = L.dguq_sc; p.out2 = L.dguT_sc; p.sf_out2 = L.hwT_sc; p.ld = v.rows;   // codes: maps o0..o2
      p.sfa = L.dyq_sc; p.sfb0 = L.wtd_sc;
      const long long items = static_cast<long long>(v.s.max_tiles) * p.n_tiles;
      MOK_CUDA((launch_gemm_mx<128, EPI_DOWN_BWD_MX>(m, p, items < sms ? static_cast<int>(items) : sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DOWN, 1, cs, last));
    }
    {  // dW_down[e] = sum over e's rows of dy[t(r)]^T (w h)[r]
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_DOWN, 0, cs, first));
      const int bn = tile_n(I);
      uint16_t* out = g->d_w_down + static_cast<long long>(v.e0) * H * I;
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dyT, v.rows, H, 128)) || (st = make_map_u8(&m.b0, L.hwT, v.rows, I, bn)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.wgrad = 1; p.grouped = 1; p.K = rows; p.E = v.ne; p.m_tiles = H / 128; p.n_tiles = I / bn;
      p.out0 = out; p.out1 = out; p.ld = I; p.split = H;
      p.sfa = L.dyT_sc; p.sfb0 = L.hwT_sc;
      MOK_CUDA(launch_mx_tiles<EPI_WGRAD>(m, p, bn, static_cast<long long>(v.ne) * p.m_tiles * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_DOWN, 1, cs, last));
    }
    {  // dW_gate|up[e] = sum over e's rows of (dG|dU)[r]^T x[t(r)]
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_GATEUP, 0, cs, first));
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dguT, v.rows, 2ull * I, 128)) || (st = make_map_u8(&m.b0, L.xT, v.rows, H, bnH)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.wgrad = 1; p.grouped = 1; p.K = rows; p.E = v.ne; p.m_tiles = 2 * I / 128; p.n_tiles = H / bnH;
      p.out0 = g->d_w_gate + static_cast<long long>(v.e0) * I * H;
      p.out1 = g->d_w_up + static_cast<long long>(v.e0) * I * H;
      p.ld = H; p.split = I;
      p.sfa = L.dguT_sc; p.sfb0 = L.xT_sc;
      MOK_CUDA(launch_mx_tiles<EPI_WGRAD>(m, p, bnH, static_cast<long long>(v.ne) * p.m_tiles * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_GATEUP, 1, cs, last));
    }
    {  // dx rows = dG W_gate[e] + dU W_up[e], in schedule order
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DGRAD_GATEUP, 0, cs, first));
      uint16_t* out = ctx->slots + v.r0 * H;
      MxMaps m;
      if ((st = make_map_u8(&m.a, L.dguq, 2ull * I, v.rows, 128)) ||
          (st = make_map_u8(&m.b0, w->mxt_gate, I, static_cast<uint64_t>(E) * H, bnH)) ||
          (st = make_map_u8(&m.b1, w->mxt_up, I, static_cast<uint64_t>(E) * H, bnH)) ||
          (st = make_map_out(&m.o0, out, H, v.rows)))
        return st;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.grouped = 1; p.K = 2 * I; p.N = H; p.n_tiles = H / bnH; p.b_rows_per_expert = H; p.b_split = I;
      p.out0 = out; p.ld = H;
      p.sfa = L.dguq_sc; p.sfb0 = L.wtg_sc; p.sfb1 = L.wtu_sc; p.sf_kgb = I / 128;
      MOK_CUDA(launch_mx_tiles<EPI_STORE_ROWS>(m, p, bnH, static_cast<long long>(v.s.max_tiles) * p.n_tiles, sms, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DGRAD_GATEUP, 1, cs, last));
    }
  }
  // ---- fixed-order reductions: dx and the router-weight gradient
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_REDUCE, 0, cs));
  MOK_CUDA(launch_combine(ctx->slots, s->slot_row, s->header, mr, Is > 0 ? L.dx_s : nullptr, T, k, H, dx, sms, cs));
  MOK_CUDA(launch_dw_reduce(L.dw_part, T * k, 2 * (I / 128), d_router_w, cs));
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_REDUCE, 1, cs));
  return MOK_OK;
}

// BF16 backward (after MOK_MODE_BF16 and MOK_MODE_MXFP8_FWD forwards): the
// shared expert's SwiGLU backward and dgrad, the routed experts window by
// window, the shared weight gradients, then the fixed-order reductions.
mok_status_t backward_bf16(const mok_config_t* cfg, const uint16_t* dy, const uint16_t* x, const float* router_w,
                           const mok_schedule_t* s, const std::vector<Win>& wins, const mok_ctx_t* ctx, const mok_weights_t* w, uint16_t* dx, float* d_router_w,
                           const mok_weight_grads_t* g, const BwdLayout& L, int sms, bool g4, cudaStream_t cs) {
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  const long long mr = static_cast<long long>(s->max_tiles) * kTileRows;
  const size_t nw = wins.size();
  mok_status_t st;
  const int bn1 = tile_n(I);
  const bool perm = resolve_dispatch(cfg) == MOK_DISPATCH_PERMUTE;
  // ---- permuted dispatch: token rows of dy, and of x (unquantised, for the
  // gate/up weight gradient), in schedule order.  x's rows: the forward's copy
  // where it spans the whole schedule (a one-pass forward with the permuted
  // dispatch), else permuted here window by window, else (a one-pass MXFP8
  // forward workspace after a forward with a ring) gathered by that GEMM.  The
  // first window's permutes run on a side stream, overlapping the shared
  // expert's backward, which reads token-order rows only.
  const bool reuse_x = perm && ctx->ring_rows == 0 && ctx->dispatch == MOK_DISPATCH_PERMUTE && ctx->x_perm &&
                       (ctx->mode == MOK_MODE_BF16 || ctx->mode == MOK_MODE_MXFP8_FWD);
  uint16_t* x_ws = (perm && !reuse_x) ? L.xb_perm : nullptr;
  auto x_rows = [&](const Win& v) -> const uint16_t* {
    if (reuse_x) return ctx->x_perm + v.r0 * H;
    return x_ws;   // NULL: gathered
  };
  auto dispatch = [&](const Win& v, cudaStream_t st2) -> cudaError_t {
    cudaError_t e = cudaSuccess;
    if (x_ws) e = launch_permute_rows(x, T, H, k, s->slot_row, s->row_src, s->header, v.r0, v.rows, x_ws, sms, st2);
    if (e == cudaSuccess)
      e = launch_permute_rows(dy, T, H, k, s->slot_row, s->row_src, s->header, v.r0, v.rows, L.dy_perm, sms, st2);
    return e;
  };
  SideStream* side = nullptr;
  if (perm && nw > 0) {
    if ((st = side_stream(&side))) return st;
    MOK_CUDA(cudaEventRecord(side->fork, cs));
    MOK_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 0, side->s));
    MOK_CUDA(dispatch(wins[0], side->s));
    MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 1, side->s, nw == 1));
    MOK_CUDA(cudaEventRecord(side->join, side->s));
  } else {
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_BWD_DISPATCH}, cs));
  }
  // ---- shared expert backward, first part (dense rows, w = 1): the SwiGLU
  // backward, which reads dy in token order while the side stream writes dy's
  // rows in schedule order, and the dgrad.  A GEMM that shares HBM with that
  // copy slows by more than the copy takes alone, so only this first GEMM
  // overlaps it; the shared weight gradients run after the routed GEMMs.
  if (Is > 0) {
    const int bns = tile_n(Is);
    {
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DOWN, 0, cs));
      GemmMaps m;
      const bool pr = pair_on(cfg, bns);
      if ((st = make_map(&m.a, dy, H, T, 128, kTileBK)) ||
          (st = make_map_mn(&m.b0, w->ws_down, Is, H, pr ? bns / 2 : bns, kTileBK)) ||
          (st = make_map_out(&m.o0, L.dgu_s, 2ull * Is, T)) || (st = make_map_out(&m.o1, L.hs, Is, T)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.rows = T; p.K = H; p.N = Is; p.n_tiles = Is / bns; p.b_rows_per_expert = 0;
      p.aux0 = ctx->gu_s; p.out0 = L.dgu_s; p.out1 = L.hs;
      p.swiglu_limit = ctx->swiglu_limit;
      const long long items = ((T + 127) / 128) * static_cast<long long>(p.n_tiles);
      if (bns == 256)
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 256, EPI_DOWN_BWD>(m, p, items, row_pairs(T) * p.n_tiles, pr,
                                                                           sms, cs)));
      else
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 128, EPI_DOWN_BWD>(m, p, items, 0, false, sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DOWN, 1, cs));
    }
    if (side) MOK_CUDA(cudaStreamWaitEvent(cs, side->join, 0));   // dy's schedule-order rows are written
    {  // dx_s = dG_s W_s_gate + dU_s W_s_up
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DGRAD, 0, cs));
      GemmMaps m;
      const int bn = tile_n(H);
      const bool pr = pair_on(cfg, bn);
      if ((st = make_map(&m.a, L.dgu_s, 2 * Is, T, 128, kTileBK)) ||
          (st = make_map_mn(&m.b0, w->ws_gate, H, Is, pr ? bn / 2 : bn, kTileBK)) ||
          (st = make_map_mn(&m.b1, w->ws_up, H, Is, pr ? bn / 2 : bn, kTileBK)) ||
          (st = make_map_out(&m.o0, L.dx_s, H, T)))
        return st;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.rows = T; p.K = 2 * Is; p.N = H; p.n_tiles = H / bn; p.b_rows_per_expert = 0; p.b_split = Is;
      p.out0 = L.dx_s; p.ld = H;
      const long long items = ((T + 127) / 128) * static_cast<long long>(p.n_tiles);
      if (bn == 256)
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 256, EPI_STORE_ROWS>(m, p, items, row_pairs(T) * p.n_tiles, pr,
                                                                             sms, cs)));
      else
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 128, EPI_STORE_ROWS>(m, p, items, 0, false, sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_DGRAD, 1, cs));
    }
  } else {
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_BWD_SHARED_DOWN, MOK_STAGE_BWD_SHARED_DGRAD}, cs));
  }
  if (side) MOK_CUDA(cudaStreamWaitEvent(cs, side->join, 0));
  // ---- routed experts, window by window (the token rows, dG|dU and w h span
  // the window; the dx rows and the router-weight partials every row)
  if (nw == 0)
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_BWD_DOWN, MOK_STAGE_BWD_WGRAD_DOWN, MOK_STAGE_BWD_WGRAD_GATEUP,
                                MOK_STAGE_BWD_DGRAD_GATEUP}, cs));
  for (size_t i = 0; i < nw; ++i) {
    const Win& v = wins[i];
    const bool first = i == 0, last = i + 1 == nw;
    if (perm && !first) {
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 0, cs, false));
      MOK_CUDA(dispatch(v, cs));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DISPATCH, 1, cs, last));
    }
    {  // down dgrad + SwiGLU backward + router-weight partials
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DOWN, 0, cs, first));
      GemmMaps m;
      const int bk = perm ? kTileBK : kGatherBK;
      const bool pr = perm && pair_on(cfg, bn1);
      if ((st = perm ? make_map(&m.a, L.dy_perm, H, v.rows, 128, bk) : make_map(&m.a, dy, H, T, 1, bk)) ||
          (st = make_map_mn(&m.b0, w->w_down, I, static_cast<uint64_t>(E) * H, pr ? bn1 / 2 : bn1, bk)) ||
          (st = make_map_out(&m.o0, L.dgu, 2ull * I, v.rows)) || (st = make_map_out(&m.o1, L.hw, I, v.rows)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.grouped = 1; p.K = H; p.N = I; p.n_tiles = I / bn1; p.b_rows_per_expert = H;
      p.aux0 = ctx->gu + v.r0 * 2 * I; p.out0 = L.dgu; p.out1 = L.hw; p.rw = router_w; p.dw_part = L.dw_part;
      p.swiglu_limit = ctx->swiglu_limit;
      p.ga = dy; p.ga_ld = H;
      const long long items = static_cast<long long>(v.s.max_tiles) * p.n_tiles;
      const int grid = items < sms ? static_cast<int>(items) : sms;
      if (perm && bn1 == 256)
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 256, EPI_DOWN_BWD>(m, p, items, items, pr, sms, cs)));
      else if (perm)
        MOK_CUDA((launch_gemm<SRC_K_TILE, SRC_MN_TILE, 128, EPI_DOWN_BWD>(m, p, grid, cs)));
      else if (g4 && bn1 == 256)
        MOK_CUDA((launch_gemm<SRC_K_GATHER, SRC_MN_TILE, 256, EPI_DOWN_BWD>(m, p, grid, cs)));
      else if (g4)
        MOK_CUDA((launch_gemm<SRC_K_GATHER, SRC_MN_TILE, 128, EPI_DOWN_BWD>(m, p, grid, cs)));
      else if (bn1 == 256)
        MOK_CUDA((launch_gemm<SRC_K_GATHER_LSU, SRC_MN_TILE, 256, EPI_DOWN_BWD>(m, p, grid, cs)));
      else
        MOK_CUDA((launch_gemm<SRC_K_GATHER_LSU, SRC_MN_TILE, 128, EPI_DOWN_BWD>(m, p, grid, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DOWN, 1, cs, last));
    }
    {  // dW_down[e] = sum over e's rows of dy[t(r)]^T (w h)[r]
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_DOWN, 0, cs, first));
      uint16_t* out = g->d_w_down + static_cast<long long>(v.e0) * H * I;
      GemmMaps m;
      const int bk = perm ? kTileBK : kGatherBK;
      const int bn = tile_n(I);
      const bool pr = perm && pair_on(cfg, bn);
      if ((st = perm ? make_map_mn(&m.a, L.dy_perm, H, v.rows, 128, bk) : make_map(&m.a, dy, H, T, 1, bk)) ||
          (st = make_map_mn(&m.b0, L.hw, I, v.rows, pr ? bn / 2 : bn, bk)) ||
          (st = make_map_out(&m.o0, out, I, static_cast<uint64_t>(v.ne) * H)))
        return st;
      m.o1 = m.o0;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.wgrad = 1; p.grouped = 1; p.E = v.ne; p.m_tiles = H / 128; p.n_tiles = I / bn;
      p.out0 = out; p.out1 = out; p.ld = I; p.split = H;
      p.estride = static_cast<long long>(H) * I;
      p.ga = dy; p.ga_ld = H;
      const long long items = static_cast<long long>(v.ne) * p.m_tiles * p.n_tiles;
      const long long pitems = static_cast<long long>(v.ne) * ((p.m_tiles + 1) / 2) * p.n_tiles;
      const int grid = items < sms ? static_cast<int>(items) : sms;
      if (perm && bn == 256)
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, items, pitems, pr, sms, cs)));
      else if (perm)
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, grid, cs)));
      else if (g4 && bn == 256)
        MOK_CUDA((launch_gemm<SRC_MN_GATHER, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, grid, cs)));
      else if (g4)
        MOK_CUDA((launch_gemm<SRC_MN_GATHER, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, grid, cs)));
      else if (bn == 256)
        MOK_CUDA((launch_gemm<SRC_MN_GATHER_LSU, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, grid, cs)));
      else
        MOK_CUDA((launch_gemm<SRC_MN_GATHER_LSU, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, grid, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_DOWN, 1, cs, last));
    }
    {  // dW_gate|up[e] = sum over e's rows of (dG|dU)[r]^T x[t(r)]
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_GATEUP, 0, cs, first));
      uint16_t* out_g = g->d_w_gate + static_cast<long long>(v.e0) * I * H;
      uint16_t* out_u = g->d_w_up + static_cast<long long>(v.e0) * I * H;
      const uint16_t* xr = x_rows(v);
      GemmMaps m;
      const int bk = xr ? kTileBK : kGatherBK;
      const int bn = tile_n(H);
      const bool pr = xr && pair_on(cfg, bn);
      if ((st = make_map_mn(&m.a, L.dgu, 2 * I, v.rows, 128, bk)) ||
          (st = xr ? make_map_mn(&m.b0, xr, H, v.rows, pr ? bn / 2 : bn, bk) : make_map(&m.b0, x, H, T, 1, bk)) ||
          (st = make_map_out(&m.o0, out_g, H, static_cast<uint64_t>(v.ne) * I)) ||
          (st = make_map_out(&m.o1, out_u, H, static_cast<uint64_t>(v.ne) * I)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.wgrad = 1; p.grouped = 1; p.E = v.ne; p.m_tiles = 2 * I / 128; p.n_tiles = H / bn;
      p.out0 = out_g; p.out1 = out_u; p.ld = H; p.split = I;
      p.estride = static_cast<long long>(I) * H;
      p.gb = x; p.gb_ld = H;
      const long long items = static_cast<long long>(v.ne) * p.m_tiles * p.n_tiles;
      const long long pitems = static_cast<long long>(v.ne) * ((p.m_tiles + 1) / 2) * p.n_tiles;
      const int grid = items < sms ? static_cast<int>(items) : sms;
      if (xr && bn == 256)
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, items, pitems, pr, sms, cs)));
      else if (xr)
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, grid, cs)));
      else if (g4 && bn == 256)
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_GATHER, 256, EPI_WGRAD>(m, p, grid, cs)));
      else if (g4)
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_GATHER, 128, EPI_WGRAD>(m, p, grid, cs)));
      else if (bn == 256)
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_GATHER_LSU, 256, EPI_WGRAD>(m, p, grid, cs)));
      else
        MOK_CUDA((launch_gemm<SRC_MN_TILE, SRC_MN_GATHER_LSU, 128, EPI_WGRAD>(m, p, grid, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_WGRAD_GATEUP, 1, cs, last));
    }
    {  // dx rows = dG W_gate[e] + dU W_up[e], in schedule order
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DGRAD_GATEUP, 0, cs, first));
      uint16_t* out = ctx->slots + v.r0 * H;
      GemmMaps m;
      const int bn = tile_n(H);
      const bool pr = pair_on(cfg, bn);
      const int bw = pr ? bn / 2 : bn;
      if ((st = make_map(&m.a, L.dgu, 2 * I, v.rows, 128, kTileBK)) ||
          (st = make_map_mn(&m.b0, w->w_gate, H, static_cast<uint64_t>(E) * I, bw, kTileBK)) ||
          (st = make_map_mn(&m.b1, w->w_up, H, static_cast<uint64_t>(E) * I, bw, kTileBK)) ||
          (st = make_map_out(&m.o0, out, H, v.rows)))
        return st;
      GemmParams p = base_params(cfg, &v.s, ctx->status, 0);
      p.grouped = 1; p.K = 2 * I; p.N = H; p.n_tiles = H / bn; p.b_rows_per_expert = I; p.b_split = I;
      p.out0 = out; p.ld = H;
      const long long items = static_cast<long long>(v.s.max_tiles) * p.n_tiles;
      if (bn == 256)
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 256, EPI_STORE_ROWS>(m, p, items, items, pr, sms, cs)));
      else
        MOK_CUDA((launch_tiles<SRC_K_TILE, SRC_MN_TILE, 128, EPI_STORE_ROWS>(m, p, items, 0, false, sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_DGRAD_GATEUP, 1, cs, last));
    }
  }
  // ---- shared expert backward, second part: the weight gradients
  if (Is > 0) {
    const int bns = tile_n(Is);
    {  // dW_s_down = dy^T h_s
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_DOWN, 0, cs));
      GemmMaps m;
      const bool pr = pair_on(cfg, bns);
      if ((st = make_map_mn(&m.a, dy, H, T, 128, kTileBK)) ||
          (st = make_map_mn(&m.b0, L.hs, Is, T, pr ? bns / 2 : bns, kTileBK)) ||
          (st = make_map_out(&m.o0, g->d_ws_down, Is, H)))
        return st;
      m.o1 = m.o0;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.wgrad = 1; p.rows = T; p.E = 1; p.m_tiles = H / 128; p.n_tiles = Is / bns;
      p.out0 = g->d_ws_down; p.out1 = g->d_ws_down; p.ld = Is; p.split = H; p.estride = 0;
      const long long items = static_cast<long long>(p.m_tiles) * p.n_tiles;
      const long long pitems = static_cast<long long>((p.m_tiles + 1) / 2) * p.n_tiles;
      if (bns == 256)
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, items, pitems, pr, sms, cs)));
      else
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, items, 0, false, sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_DOWN, 1, cs));
    }
    {  // dW_s_gate|up = (dG_s|dU_s)^T x
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_GATEUP, 0, cs));
      GemmMaps m;
      const int bn = tile_n(H);
      const bool pr = pair_on(cfg, bn);
      if ((st = make_map_mn(&m.a, L.dgu_s, 2 * Is, T, 128, kTileBK)) ||
          (st = make_map_mn(&m.b0, x, H, T, pr ? bn / 2 : bn, kTileBK)) ||
          (st = make_map_out(&m.o0, g->d_ws_gate, H, Is)) || (st = make_map_out(&m.o1, g->d_ws_up, H, Is)))
        return st;
      m.b1 = m.b0;
      GemmParams p = base_params(cfg, nullptr, ctx->status, 0);
      p.wgrad = 1; p.rows = T; p.E = 1; p.m_tiles = 2 * Is / 128; p.n_tiles = H / bn;
      p.out0 = g->d_ws_gate; p.out1 = g->d_ws_up; p.ld = H; p.split = Is; p.estride = 0;
      const long long items = static_cast<long long>(p.m_tiles) * p.n_tiles;
      const long long pitems = static_cast<long long>((p.m_tiles + 1) / 2) * p.n_tiles;
      if (bn == 256)
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 256, EPI_WGRAD>(m, p, items, pitems, pr, sms, cs)));
      else
        MOK_CUDA((launch_tiles<SRC_MN_TILE, SRC_MN_TILE, 128, EPI_WGRAD>(m, p, items, 0, false, sms, cs)));
      MOK_CUDA(mark(cfg, MOK_STAGE_BWD_SHARED_WGRAD_GATEUP, 1, cs));
    }
  } else {
    MOK_CUDA(mark_skipped(cfg, {MOK_STAGE_BWD_SHARED_WGRAD_DOWN, MOK_STAGE_BWD_SHARED_WGRAD_GATEUP}, cs));
  }
  // ---- fixed-order reductions: dx and the router-weight gradient
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_REDUCE, 0, cs));
  MOK_CUDA(launch_combine(ctx->slots, s->slot_row, s->header, mr, Is > 0 ? L.dx_s : nullptr, T, k, H, dx, sms,
                          cs));
  MOK_CUDA(launch_dw_reduce(L.dw_part, T * k, 2 * (I / bn1), d_router_w, cs));
  MOK_CUDA(mark(cfg, MOK_STAGE_BWD_REDUCE, 1, cs));
  return MOK_OK;
}

}  // namespace

// ===========================================================================
extern "C" {

int mok_version(void) { return 1; }

const char* mok_last_error(void) { return g_err; }

size_t mok_schedule_bytes(int T, int k, int E) {
  if (T < 1 || k < 1 || E < 1) return 0;
  SchedLayout L;
  return carve_schedule(nullptr, T, k, E, &L);
}

mok_status_t mok_schedule(const int64_t* top_experts, int T, int k, int E, double capacity_multiplier,
                          void* buf, size_t bytes, mok_schedule_t* out, void* stream) {
  NvtxCall nvtx("mok_schedule");
  if (!top_experts || !buf || !out) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (T < 1 || k < 1 || k > 64 || E < 1 || E > 1024)
    return fail(MOK_ERR_INVALID_ARG, "need T >= 1, 1 <= k <= 64, 1 <= E <= 1024");
  if (static_cast<long long>(T) * k >= (1ll << 31) - 128ll * E)
    return fail(MOK_ERR_INVALID_ARG, "T*k too large");
  if (!std::isfinite(capacity_multiplier) || capacity_multiplier < 0.0)
    return fail(MOK_ERR_INVALID_ARG, "capacity_multiplier must be finite and >= 0");
  if (!aligned16(top_experts) || !aligned16(buf)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  if (bytes < mok_schedule_bytes(T, k, E)) return fail(MOK_ERR_INVALID_ARG, "schedule buffer too small");
  int sms = 0;
  mok_status_t st = device_info(&sms);
  if (st) return st;
  SchedLayout L;
  carve_schedule(buf, T, k, E, &L);
  const long long mt = max_tiles_of(T, k, E);
  // per-expert tile budget, decided in double precision on the caller's value
  const double rows = std::ceil(capacity_multiplier * static_cast<double>(T));
  double capd = std::ceil(rows / kTileRows);
  if (capd > static_cast<double>(mt)) capd = static_cast<double>(mt);
  const int cap = static_cast<int>(capd);
  MOK_CUDA(launch_schedule(top_experts, T, k, E, cap, static_cast<int>(mt), L.hist, L.cnt, L.row0,
                           L.row_src, L.slot_row, L.tile_expert, L.tile_row0, L.tile_rows, L.pair_tile,
                           L.unit_group, L.header, static_cast<cudaStream_t>(stream)));
  out->T = T; out->k = k; out->E = E; out->max_tiles = static_cast<int>(mt);
  out->cnt = L.cnt; out->row0 = L.row0; out->row_src = L.row_src; out->slot_row = L.slot_row;
  out->tile_expert = L.tile_expert; out->tile_row0 = L.tile_row0; out->tile_rows = L.tile_rows;
  out->header = L.header; out->scratch = L.hist; out->pair_tile = L.pair_tile; out->unit_group = L.unit_group;
  return MOK_OK;
}

mok_status_t mok_schedule_status(const mok_schedule_t* s, int* status, int* num_tiles, int* P) {
  if (!s || !s->header) return fail(MOK_ERR_INVALID_ARG, "NULL schedule");
  int h[8];
  MOK_CUDA(cudaDeviceSynchronize());
  MOK_CUDA(cudaMemcpy(h, s->header, sizeof(h), cudaMemcpyDeviceToHost));
  if (status) *status = h[2];
  if (num_tiles) *num_tiles = h[0];
  if (P) *P = h[1];
  return MOK_OK;
}

mok_status_t mok_mxfp8_quantize(const uint16_t* x, int64_t rows, int K, uint8_t* codes,
                                uint8_t* scales, void* stream) {
  NvtxCall nvtx("mok_mxfp8_quantize");
  if (rows < 0 || K <= 0 || K % 32) return fail(MOK_ERR_INVALID_ARG, "need rows >= 0 and K % 32 == 0");
  if (rows == 0) return MOK_OK;
  if (!x || !codes || !scales) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(x) || !aligned16(codes)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  int sms = 0;
  mok_status_t st = device_info(&sms);
  if (st) return st;
  MOK_CUDA(launch_mx_quantize(x, rows * (K / 32), codes, scales, sms, static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status_t mok_mxfp8_quantize_t(const uint16_t* x, int64_t batch, int rows, int cols, uint8_t* codes,
                                  uint8_t* scales, void* stream) {
  NvtxCall nvtx("mok_mxfp8_quantize_t");
  if (batch < 0 || rows < 0 || cols < 0 || rows % 32 || cols % 64)
    return fail(MOK_ERR_INVALID_ARG, "need batch, rows, cols >= 0, rows %% 32 == 0 and cols %% 64 == 0");
  if (batch == 0 || rows == 0 || cols == 0) return MOK_OK;
  if (batch > (1ll << 30) / 64) return fail(MOK_ERR_INVALID_ARG, "batch too large");
  if (!x || !codes || !scales) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(x) || !aligned16(codes)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  int sms = 0;
  mok_status_t st = device_info(&sms);
  if (st) return st;
  MOK_CUDA(launch_mx_quantize_t(x, cols, static_cast<int>(batch), rows, cols, rows, nullptr, 1, nullptr, codes, scales,
                                0, sms, static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status_t mok_mxfp8_quantize_dual(const uint16_t* x, int64_t batch, int rows, int cols, uint8_t* codes,
                                     uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, void* stream) {
  NvtxCall nvtx("mok_mxfp8_quantize_dual");
  if (batch < 0 || rows < 0 || cols < 0 || rows % 32 || cols % 64)
    return fail(MOK_ERR_INVALID_ARG, "need batch, rows, cols >= 0, rows %% 32 == 0 and cols %% 64 == 0");
  if (batch == 0 || rows == 0 || cols == 0) return MOK_OK;
  if (batch > (1ll << 30) / 64) return fail(MOK_ERR_INVALID_ARG, "batch too large");
  if (!x || !codes || !scales || !codes_t || !scales_t) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(x) || !aligned16(codes) || !aligned16(codes_t)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  int sms = 0;
  mok_status_t st = device_info(&sms);
  if (st) return st;
  MOK_CUDA(launch_mx_quantize_t(x, cols, static_cast<int>(batch), rows, cols, rows, nullptr, 1, nullptr, codes_t,
                                scales_t, 0, sms, static_cast<cudaStream_t>(stream), codes, scales, 0));
  return MOK_OK;
}

size_t mok_ctx_bytes(int T, int k, int E, int H, int I, int I_s, int mode) {
  return mok_ctx_bytes_ring(T, k, E, H, I, I_s, mode, 0);
}

size_t mok_ctx_bytes_ring(int T, int k, int E, int H, int I, int I_s, int mode, int64_t macrobatch_size) {
  if (check_shapes(T, k, E, H, I, I_s) != MOK_OK || macrobatch_size < 0) return 0;
  mok_ctx_t c;
  CtxExtra X;
  return carve_ctx(nullptr, T, k, E, H, I, I_s, mode,
                   ring_rows_of(macrobatch_size, max_tiles_of(T, k, E) * kTileRows), &c, &X);
}

mok_status_t mok_macrobatch_plan(const int32_t* cnt, int E, int64_t macrobatch_size, int32_t* first_expert,
                                 int* num_windows) {
  if (!cnt || !first_expert || !num_windows) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (E < 1 || E > 1024) return fail(MOK_ERR_INVALID_ARG, "need 1 <= E <= 1024 (E=%d)", E);
  if (macrobatch_size < 0) return fail(MOK_ERR_INVALID_ARG, "macrobatch_size < 0");
  const long long ring = macrobatch_size == 0 ? 0 : (macrobatch_size + kTileRows - 1) / kTileRows * kTileRows;
  std::vector<int> first;
  const mok_status_t st = plan_windows(cnt, E, ring, &first);
  if (st) return st;
  for (size_t i = 0; i < first.size(); ++i) first_expert[i] = first[i];
  *num_windows = static_cast<int>(first.size()) - 1;
  return MOK_OK;
}

mok_status_t mok_ctx_status(const mok_ctx_t* ctx, int* status) {
  if (!ctx || !ctx->status || !status) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  MOK_CUDA(cudaDeviceSynchronize());
  MOK_CUDA(cudaMemcpy(status, ctx->status, sizeof(int), cudaMemcpyDeviceToHost));
  return MOK_OK;
}

mok_status_t mok_forward(const mok_config_t* cfg, const uint16_t* x, const float* router_w,
                         const mok_schedule_t* s, const mok_weights_t* w, uint16_t* y, void* ctx_buf,
                         size_t ctx_bytes, mok_ctx_t* ctx, void* stream) {
  NvtxCall nvtx("mok_forward");
  if (!cfg || !x || !router_w || !s || !w || !y || !ctx_buf || !ctx)
    return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  mok_status_t st = check_config(cfg);
  if (st) return st;
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  if (w->E != E) return fail(MOK_ERR_INVALID_ARG, "weights have E=%d, schedule E=%d", w->E, E);
  st = check_shapes(T, k, E, H, I, Is);
  if (st) return st;
  if (!w->w_gate || !w->w_up || !w->w_down) return fail(MOK_ERR_INVALID_ARG, "NULL routed weight");
  if (Is > 0 && (!w->ws_gate || !w->ws_up || !w->ws_down))
    return fail(MOK_ERR_INVALID_ARG, "NULL shared weight");
  const bool mx = cfg->mode == MOK_MODE_MXFP8_FWD || cfg->mode == MOK_MODE_MXFP8;
  if (mx && (!w->mx_gate || !w->mx_gate_sc || !w->mx_up || !w->mx_up_sc || !w->mx_down || !w->mx_down_sc ||
             (Is > 0 && (!w->mxs_gate || !w->mxs_gate_sc || !w->mxs_up || !w->mxs_up_sc || !w->mxs_down ||
                         !w->mxs_down_sc))))
    return fail(MOK_ERR_INVALID_ARG, "MXFP8 mode needs the prequantised weights");
  if (mx) {
    const void* mp[] = {w->mx_gate, w->mx_gate_sc, w->mx_up, w->mx_up_sc, w->mx_down, w->mx_down_sc,
                        w->mxs_gate, w->mxs_gate_sc, w->mxs_up, w->mxs_up_sc, w->mxs_down, w->mxs_down_sc};
    for (const void* q : mp)
      if (!aligned16(q)) return fail(MOK_ERR_INVALID_ARG, "misaligned MXFP8 weight pointer");
  }
  const void* ptrs[] = {x, router_w, y, ctx_buf, w->w_gate, w->w_up, w->w_down};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  if (Is > 0 && (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down)))
    return fail(MOK_ERR_INVALID_ARG, "misaligned shared weight pointer");
  if (ctx_bytes < mok_ctx_bytes_ring(T, k, E, H, I, Is, cfg->mode, cfg->macrobatch_size))
    return fail(MOK_ERR_INVALID_ARG, "context buffer too small");
  int sms = 0;
  st = device_info(&sms);
  if (st) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool g4 = (cfg->debug_flags & MOK_DEBUG_TMA_GATHER4) != 0;
  const long long mr = static_cast<long long>(s->max_tiles) * kTileRows;
  const long long ring = ring_rows_of(cfg->macrobatch_size, mr);
  CtxExtra X;
  mok_ctx_t c;
  carve_ctx(ctx_buf, T, k, E, H, I, Is, cfg->mode, ring, &c, &X);
  // the windows are planned (a ring reads the expert counts back) before any
  // layer work is enqueued
  std::vector<Win> wins;
  if ((st = make_windows(s, ring, X.view, cs, &wins))) return st;
  *ctx = c;
  ctx->swiglu_limit = cfg->swiglu_limit;
  MOK_CUDA(cudaMemsetAsync(X.tickets, 0, fwd_tickets(E) * sizeof(int32_t), cs));
  TicketScope tickets(X.tickets, fwd_tickets(E));
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_PREP, 0, cs));
  MOK_CUDA(cudaMemsetAsync(ctx->status, 0, 8 * sizeof(int), cs));
  MOK_CUDA(launch_dependent(propagate_status_kernel, dim3(1), dim3(1), 0, cs, static_cast<const int*>(s->header),
                            ctx->status));

  if (mx) {
    st = forward_mxfp8(cfg, x, router_w, s, wins, w, ctx, X, sms, cs);
    if (st) return st;
  } else {
    st = forward_bf16(cfg, x, router_w, s, wins, w, ctx, sms, g4, cs);
    if (st) return st;
  }

  // ---- combine: y[t] = shared[t] + sum_j slots[t, j] in fixed order
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_COMBINE, 0, cs));
  MOK_CUDA(launch_combine(ctx->slots, s->slot_row, s->header, mr, Is > 0 ? ctx->shared_out : nullptr, T, k, H, y,
                          sms, cs));
  MOK_CUDA(mark(cfg, MOK_STAGE_FWD_COMBINE, 1, cs));
  return MOK_OK;
}

size_t mok_bwd_workspace_bytes(int T, int k, int E, int H, int I, int I_s, int mode) {
  return mok_bwd_workspace_bytes_ring(T, k, E, H, I, I_s, mode, 0);
}

size_t mok_bwd_workspace_bytes_ring(int T, int k, int E, int H, int I, int I_s, int mode, int64_t macrobatch_size) {
  if (check_shapes(T, k, E, H, I, I_s) != MOK_OK || macrobatch_size < 0) return 0;
  if (mode != MOK_MODE_BF16 && mode != MOK_MODE_MXFP8_FWD && mode != MOK_MODE_MXFP8) return 0;
  BwdLayout L;
  return carve_bwd(nullptr, T, k, E, H, I, I_s, mode,
                   ring_rows_of(macrobatch_size, max_tiles_of(T, k, E) * kTileRows), &L);
}

mok_status_t mok_backward(const mok_config_t* cfg, const uint16_t* dy, const uint16_t* x,
                          const float* router_w, const mok_schedule_t* s, const mok_ctx_t* ctx,
                          const mok_weights_t* w, uint16_t* dx, float* d_router_w,
                          const mok_weight_grads_t* g, void* ws, size_t ws_bytes, void* stream) {
  NvtxCall nvtx("mok_backward");
  if (!cfg || !dy || !x || !router_w || !s || !ctx || !w || !dx || !d_router_w || !g || !ws)
    return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  mok_status_t st = check_config(cfg);
  if (st) return st;
  const int T = s->T, k = s->k, E = s->E, H = w->H, I = w->I, Is = w->I_s;
  st = check_shapes(T, k, E, H, I, Is);
  if (st) return st;
  if (w->E != E) return fail(MOK_ERR_INVALID_ARG, "weights have E=%d, schedule E=%d", w->E, E);
  if (ctx->T != T || ctx->k != k || ctx->E != E || ctx->H != H || ctx->I != I || ctx->I_s != Is)
    return fail(MOK_ERR_INVALID_ARG, "context does not match the schedule / weights");
  if (ctx->mode != MOK_MODE_BF16 && ctx->mode != MOK_MODE_MXFP8_FWD && ctx->mode != MOK_MODE_MXFP8)
    return fail(MOK_ERR_INVALID_ARG, "context mode %d is not one a forward records", ctx->mode);
  if (!g->d_w_gate || !g->d_w_up || !g->d_w_down) return fail(MOK_ERR_INVALID_ARG, "NULL routed grad");
  if (Is > 0 && (!g->d_ws_gate || !g->d_ws_up || !g->d_ws_down || !w->ws_gate || !w->ws_up || !w->ws_down))
    return fail(MOK_ERR_INVALID_ARG, "NULL shared weight or grad");
  const void* ptrs[] = {dy, x, router_w, dx, d_router_w, ws, g->d_w_gate, g->d_w_up, g->d_w_down};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  if (Is > 0) {
    const void* sp[] = {w->ws_gate, w->ws_up, w->ws_down, g->d_ws_gate, g->d_ws_up, g->d_ws_down};
    for (const void* q : sp)
      if (!aligned16(q)) return fail(MOK_ERR_INVALID_ARG, "misaligned shared weight or grad pointer");
  }
  const bool mxb = ctx->mode == MOK_MODE_MXFP8;
  if (mxb) {
    const void* mp[] = {w->mxt_gate, w->mxt_gate_sc, w->mxt_up, w->mxt_up_sc, w->mxt_down, w->mxt_down_sc};
    const void* ms[] = {w->mxts_gate, w->mxts_gate_sc, w->mxts_up, w->mxts_up_sc, w->mxts_down, w->mxts_down_sc};
    for (const void* q : mp)
      if (!q || !aligned16(q)) return fail(MOK_ERR_INVALID_ARG, "MXFP8 backward needs the transposed weight copies");
    for (const void* q : ms)
      if (Is > 0 && (!q || !aligned16(q)))
        return fail(MOK_ERR_INVALID_ARG, "MXFP8 backward needs the transposed shared weight copies");
  }
  if (ws_bytes < mok_bwd_workspace_bytes_ring(T, k, E, H, I, Is, ctx->mode, cfg->macrobatch_size))
    return fail(MOK_ERR_INVALID_ARG, "backward workspace too small");
  int sms = 0;
  st = device_info(&sms);
  if (st) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool g4 = (cfg->debug_flags & MOK_DEBUG_TMA_GATHER4) != 0;
  const long long ring = ring_rows_of(cfg->macrobatch_size, max_tiles_of(T, k, E) * kTileRows);
  BwdLayout L;
  carve_bwd(ws, T, k, E, H, I, Is, ctx->mode, ring, &L);
  std::vector<Win> wins;
  if ((st = make_windows(s, ring, L.view, cs, &wins))) return st;
  MOK_CUDA(cudaMemsetAsync(L.tickets, 0, bwd_tickets(E) * sizeof(int32_t), cs));
  TicketScope tickets(L.tickets, bwd_tickets(E));
  if (mxb) return backward_mxfp8(cfg, dy, x, router_w, s, wins, ctx, w, dx, d_router_w, g, L, sms, cs);
  return backward_bf16(cfg, dy, x, router_w, s, wins, ctx, w, dx, d_router_w, g, L, sms, g4, cs);
}

mok_status_t mok_schedule_noalloc(const int64_t* top_experts, int T, int k, int E,
                                  double capacity_multiplier, void* buf, size_t bytes,
                                  mok_schedule_t* out, void* stream) {
  NvtxCall nvtx("mok_schedule_noalloc");
  if (!top_experts || !buf || !out) return fail(MOK_ERR_INVALID_ARG, "NULL argument");
  if (T < 1 || k < 1 || k > 64 || E < 1 || E > 1024)
    return fail(MOK_ERR_INVALID_ARG, "need T >= 1, 1 <= k <= 64, 1 <= E <= 1024");
  if (static_cast<long long>(T) * k >= (1ll << 31) - 128ll * E)
    return fail(MOK_ERR_INVALID_ARG, "T*k too large");
  const long long nchunks = (static_cast<long long>(T) * k + kSchedChunk - 1) / kSchedChunk;
  if (nchunks * E > kStaticSchedScratchInts)
    return fail(MOK_ERR_INVALID_ARG,
                "mok_schedule_noalloc: ceil(T*k/%d) * E = %lld exceeds its fixed scratch of %lld ints",
                kSchedChunk, nchunks * E, kStaticSchedScratchInts);
  if (!std::isfinite(capacity_multiplier) || capacity_multiplier < 0.0)
    return fail(MOK_ERR_INVALID_ARG, "capacity_multiplier must be finite and >= 0");
  if (!aligned16(top_experts) || !aligned16(buf)) return fail(MOK_ERR_INVALID_ARG, "misaligned pointer");
  SchedLayout L;
  carve_schedule(buf, T, k, E, &L);
  // only the output arrays (everything before the histogram region) live in buf
  const size_t need = static_cast<size_t>(reinterpret_cast<uint8_t*>(L.hist) - static_cast<uint8_t*>(buf));
  if (bytes < need) return fail(MOK_ERR_INVALID_ARG, "schedule buffer too small (%zu < %zu)", bytes, need);
  int sms = 0;
  mok_status_t st = device_info(&sms);
  if (st) return st;
  int32_t* scratch = nullptr;
  if ((st = static_sched_scratch(&scratch))) return st;
  const long long mt = max_tiles_of(T, k, E);
  const double rows = std::ceil(capacity_multiplier * static_cast<double>(T));
  double capd = std::ceil(rows / kTileRows);
  if (capd > static_cast<double>(mt)) capd = static_cast<double>(mt);
  // every histogram entry the build reads is first written by it, so the
  // array needs no clearing between calls
  MOK_CUDA(launch_schedule(top_experts, T, k, E, static_cast<int>(capd), static_cast<int>(mt), scratch, L.cnt,
                           L.row0, L.row_src, L.slot_row, L.tile_expert, L.tile_row0, L.tile_rows, L.pair_tile,
                           L.unit_group, L.header, static_cast<cudaStream_t>(stream)));
  out->T = T; out->k = k; out->E = E; out->max_tiles = static_cast<int>(mt);
  out->cnt = L.cnt; out->row0 = L.row0; out->row_src = L.row_src; out->slot_row = L.slot_row;
  out->tile_expert = L.tile_expert; out->tile_row0 = L.tile_row0; out->tile_rows = L.tile_rows;
  out->header = L.header; out->scratch = scratch; out->pair_tile = L.pair_tile; out->unit_group = L.unit_group;
  return MOK_OK;
}

}  // extern "C"

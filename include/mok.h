/*
 * mok.h — C ABI of libmok: a single-GPU (GB300, sm_103a) implementation of
 * the deterministic routed-plus-shared SwiGLU mixture-of-experts layer that
 * the Mixture-of-Kittens (MoK) pages describe.
 *
 * Sources (page title, section):
 *   [MoKEd]  "Mixture-of-Kittens: a deterministic MoE megakernel for NVL72
 *            racks" — "The two API layers and the schedule object": the
 *            schedule is built once from the routing, before any kernel runs,
 *            and the same object feeds forward and backward; a workspace holds
 *            scratch.  "Tuning the five hyperparameters before production":
 *            minibatch_size, schedule_capacity_multiplier, MXFP8 weights
 *            prequantised by a separate mxfp8_quantize.  "Where MoK is the
 *            wrong tool": top-k experts int64 [tokens, topk], router weights
 *            float32, the router is outside the library.
 *   [MoKDoc] "nemo_automodel.components.moe.mok_experts" — _MoKRuntime.forward
 *            (x bf16 [tokens, hidden], router weights fp32 [tokens, topk],
 *            top experts int64, shared gate/up [I_s, H], shared down [H, I_s],
 *            routed gate/up [E, I, H], routed down [E, H, I], all contiguous
 *            bf16; returns y bf16 [tokens, hidden] plus an opaque schedule and
 *            context) and _MoKRuntime.backward (gradients for x, the router
 *            weights, the three routed and the three shared weights).
 *
 * Conventions for every call:
 *   - Every pointer is a DEVICE pointer unless stated otherwise; every buffer
 *     is contiguous, row-major and 16-byte aligned.  bf16 values are passed as
 *     uint16_t bit patterns.
 *   - The library allocates nothing.  The caller owns every buffer; the
 *     *_bytes() queries say how large each caller-provided region must be.
 *   - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and returns without synchronising.  Only mok_schedule_status()
 *     and mok_ctx_status() synchronise.
 *   - Host-visible argument errors return a status code and enqueue nothing.
 *     Errors found on the device (an expert id out of range, a bounded wait
 *     that gave up) are recorded in a device status word and read back with
 *     mok_schedule_status() / mok_ctx_status(); kernels that follow a failed
 *     schedule do no work.
 *   - mok_last_error() returns a message for the last failing call of the
 *     calling thread.
 *   - Loading the library creates no CUDA context.
 *   - Only sm_103a devices are supported (MOK_ERR_UNSUPPORTED otherwise).
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mok_status_t;

#define MOK_OK               0
#define MOK_ERR_INVALID_ARG  1  /* bad size, NULL or misaligned pointer, short buffer */
#define MOK_ERR_INDEX        2  /* an expert id outside [0, E) */
#define MOK_ERR_CAPACITY     3  /* one expert's rows do not fit the macrobatch ring (the
                                   capacity split itself never drops rows) */
#define MOK_ERR_UNSUPPORTED  4  /* not an sm_103a device, or a shape outside the kernels' contract */
#define MOK_ERR_TIMEOUT      5  /* a bounded device-side wait gave up */
#define MOK_ERR_CUDA         6  /* a CUDA runtime call failed */

#define MOK_TILE_ROWS 128       /* each expert's row range is padded to this */
#define MOK_MX_BLOCK  32        /* MXFP8: one E8M0 scale per 1x32 block along K */

#define MOK_MODE_BF16       0   /* forward and backward in bf16, fp32 accumulate */
#define MOK_MODE_MXFP8_FWD  1   /* forward GEMMs on MXFP8 operands, backward in bf16 */
#define MOK_MODE_MXFP8      2   /* forward and backward GEMMs on MXFP8 operands: each
                                   backward GEMM quantises both operands along its own
                                   contraction axis (dgrad: dy and dG|dU by rows, the
                                   weights along H or I; weight gradients: both
                                   operands over 32 consecutive rows of an expert in
                                   schedule order, or 32 consecutive tokens for the
                                   shared expert); fp32 accumulate, bf16 outputs */

/* Debug flags (mok_config_t.debug_flags). */
#define MOK_DEBUG_DROP_ACC_SIGNAL 1  /* the first forward GEMM withholds one
                                        accumulator-ready signal, so a bounded
                                        wait must expire and the context must
                                        report MOK_ERR_TIMEOUT (tests only) */
#define MOK_DEBUG_TMA_GATHER4     2  /* fetch gathered token rows with TMA
                                        tile::gather4 loads instead of the
                                        gather warps' cp.async copies (same
                                        results, slower; kept for comparison) */
#define MOK_DEBUG_NO_CTA_PAIR     4  /* run every bf16 GEMM on single CTAs instead
                                        of CTA pairs (M = 256 over two SMs
                                        sharing B; same results; for comparison) */
#define MOK_DEBUG_MX_CTA_PAIR     8  /* run the block-scaled MXFP8 forward GEMMs as
                                        CTA pairs with 256-wide tiles (same results;
                                        measured slower on one GB300: their
                                        accumulator is single-buffered, so each
                                        tile waits for both CTAs' epilogues) */
#define MOK_DEBUG_MX_PAIR128     16  /* run the block-scaled MXFP8 forward GEMMs as
                                        CTA pairs with 128-wide tiles and a
                                        double-buffered accumulator (same results;
                                        measured slower on one GB300) */
#define MOK_DEBUG_PLAIN_ORDER    32  /* visit each GEMM's output tiles row unit by
                                        row unit, all column tiles of one before
                                        the next (same results; for comparison with
                                        the default, which walks a group of row
                                        units inside each column tile so that the
                                        larger operand streams through L2 once) */
#define MOK_DEBUG_STATIC_ORDER   64  /* give each CTA of the bf16 GEMMs the work
                                        items idx, idx + grid, ... (same results).
                                        By default the row GEMMs of long launches
                                        (at least 200 work items per SM) hand out
                                        the next item in line as a CTA starts one,
                                        which keeps every CTA on neighbouring items
                                        so that shared operands stay in L2 */
#define MOK_DEBUG_TICKET_ORDER  128  /* hand out every TMA-fed bf16 GEMM's items
                                        in line, whatever the launch's size (same
                                        results; tests and comparison) */

/* Stages of the layer, for optional per-stage timing events. */
#define MOK_STAGE_FWD_PREP                 0  /* status hand-over; MXFP8: weight scales into the tensor-core layout */
#define MOK_STAGE_FWD_SHARED_GATEUP        1  /* shared gate/up GEMM + SwiGLU */
#define MOK_STAGE_FWD_SHARED_DOWN          2  /* shared down GEMM */
#define MOK_STAGE_FWD_GATEUP               3  /* routed gate/up GEMM + SwiGLU */
#define MOK_STAGE_FWD_DOWN                 4  /* routed down GEMM + router scale + scatter */
#define MOK_STAGE_FWD_COMBINE              5  /* fixed-order combine into y */
#define MOK_STAGE_BWD_DOWN                 6  /* routed dgrad through down + SwiGLU bwd + router-grad partials */
#define MOK_STAGE_BWD_WGRAD_DOWN           7  /* routed dW_down */
#define MOK_STAGE_BWD_WGRAD_GATEUP         8  /* routed dW_gate, dW_up */
#define MOK_STAGE_BWD_DGRAD_GATEUP         9  /* routed dgrad through gate/up -> dx rows in schedule order */
#define MOK_STAGE_BWD_SHARED_DOWN         10
#define MOK_STAGE_BWD_SHARED_WGRAD_DOWN   11
#define MOK_STAGE_BWD_SHARED_WGRAD_GATEUP 12
#define MOK_STAGE_BWD_SHARED_DGRAD        13
#define MOK_STAGE_BWD_REDUCE              14  /* fixed-order dx combine + router-grad reduce */
#define MOK_STAGE_FWD_DISPATCH            15  /* token rows of x into schedule order (MXFP8: quantised on the way) */
#define MOK_STAGE_BWD_DISPATCH            16  /* token rows of dy (and x) into schedule order */
#define MOK_NUM_STAGES                    17

/* Per-call knobs ([MoKEd] "Tuning the five hyperparameters before
 * production").  minibatch_size (0 = T) is accepted and checked; on one GPU
 * the GEMMs visit work expert by expert for every size (there is no exchange
 * to overlap, and wave order would re-read every expert's weights once per
 * wave), so it never changes a result bit.  `events`, when not NULL, holds
 * 2 * MOK_NUM_STAGES cudaEvent_t handles (owned by the caller); the call
 * records events[2s] before and events[2s+1] after stage s on the stream the
 * stage runs on (the caller's, or for the dispatch stages the library's side
 * stream; a stage that does not run records both back to back), so a caller
 * can time each kernel.  A NULL entry records nothing: each record costs the
 * device a few microseconds, so a timing run can watch one stage alone. */
/* How the routed GEMMs receive the token rows of each expert tile (the
 * on-chip form of MoK's dispatch exchange).  Every choice moves the same bytes
 * into the same shared-memory layout, so results are bitwise identical. */
#define MOK_DISPATCH_AUTO     0  /* the library's choice: MOK_DISPATCH_PERMUTE */
#define MOK_DISPATCH_PERMUTE  1  /* a bandwidth-bound kernel writes the token rows in
                                    schedule order once (x in the forward, dy and,
                                    when needed, x in the backward); the GEMMs then
                                    read dense TMA tiles */
#define MOK_DISPATCH_FUSED    2  /* the GEMMs gather the token rows themselves
                                    (gather warps; TMA tile::gather4 with
                                    MOK_DEBUG_TMA_GATHER4) */

typedef struct {
  int mode;            /* MOK_MODE_* */
  int minibatch_size;  /* tokens per wave of the persistent pipeline; 0 = T */
  int debug_flags;     /* MOK_DEBUG_*; 0 in production */
  int dispatch;        /* MOK_DISPATCH_*: the bf16 GEMMs' choice (the bf16
                          forward, and every bf16 backward).  The MXFP8 GEMMs
                          always read rows that a quantiser wrote in schedule
                          order. */
  int num_events;      /* 0, or 2 * MOK_NUM_STAGES when events is set */
  void* const* events; /* optional cudaEvent_t[2 * MOK_NUM_STAGES], NULL = off */
  float swiglu_limit;  /* forward: 0 = plain SwiGLU; L > 0 clamps the gate
                          pre-activation to <= L and the up pre-activation to
                          [-L, L] before the SwiGLU ([MoKDoc] _MoKRuntime names
                          swiglu_limit without defining it; this is the usual
                          clamped SwiGLU).  The backward takes the value the
                          forward recorded in the context and differentiates
                          the clamp (gate gradient where G <= L, up gradient
                          where |U| <= L).  Negative or non-finite:
                          MOK_ERR_INVALID_ARG. */
  int64_t macrobatch_size; /* rows of the token ring ([MoKEd] "Tuning the five
                          hyperparameters before production": macrobatch_size
                          is the token ring buffer size; a value that holds
                          every row means the ring is used once).  A routed
                          row is one token's copy for one expert.  0, or a
                          size of at least max_tiles * 128 rows, runs the
                          routed experts in one pass over buffers for the
                          whole schedule.  A smaller size, rounded up to a
                          multiple of 128, bounds every schedule-order scratch
                          buffer of the call (the token rows, h, dG|dU, w*h
                          and their MXFP8 codes): the routed experts then run
                          window by window, each window a run of whole
                          experts in expert order whose padded rows fit the
                          ring (mok_macrobatch_plan), so no contraction is
                          split and every result bit equals the single pass.
                          The saved gate|up pre-activations and the per-row
                          outputs the fixed-order combines read (y's and dx's
                          schedule-order rows) stay full size.  Such a call
                          reads the expert counts back to the host once
                          (it synchronises `stream`, so it cannot be captured
                          in a CUDA graph), and fails with MOK_ERR_CAPACITY,
                          enqueueing no layer work, when one expert's padded
                          rows exceed the ring.  Size the buffers with
                          mok_ctx_bytes_ring / mok_bwd_workspace_bytes_ring.
                          With a ring, per-stage events of the routed stages
                          bracket all windows (from the stage's start in the
                          first window to its end in the last), so their
                          intervals overlap.  Negative: MOK_ERR_INVALID_ARG. */
} mok_config_t;

/* The dispatch/combine schedule ([MoKEd] "The two API layers and the
 * schedule object").  All arrays live in the caller's schedule buffer.
 * Flat routed row f = t*k + j.  Rows of expert e occupy schedule rows
 * [row0[e], row0[e] + cnt[e]) in ascending f; each expert's range is padded
 * to a multiple of 128 rows; padding rows and unused entries hold -1. */
typedef struct {
  int T, k, E;
  int max_tiles;          /* floor((T*k + 127*E) / 128): bound on tiles */
  int32_t* cnt;           /* [E]   rows per expert */
  int32_t* row0;          /* [E+1] exclusive scan of the padded counts; row0[E] = P */
  int32_t* row_src;       /* [max_tiles*128] schedule row -> f, or -1 */
  int32_t* slot_row;      /* [T*k] f -> schedule row */
  int32_t* tile_expert;   /* [max_tiles] expert of each 128-row tile, or -1 */
  int32_t* tile_row0;     /* [max_tiles] first schedule row of the tile, or -1 */
  int32_t* tile_rows;     /* [max_tiles] valid rows in the tile (1..128), or -1 */
  int32_t* header;        /* [8] num_tiles, P, status, num_primary, num_pairs, cap_tiles
                             (the per-expert budget of the primary list), 0, 0 */
  int32_t* scratch;       /* internal: per-chunk histograms */
  int32_t* pair_tile;     /* [max_tiles][2] tile pairs for CTA-pair GEMMs: two consecutive
                             tiles of one expert (within the primary list, then within the
                             overflow list), second -1 for an odd tile; unused pairs -1 */
  int32_t* unit_group;    /* [2][max_tiles] the GEMMs' work groups: entry t of the first
                             half for tile t, entry p of the second for pair p.  Each run of
                             one expert's tiles (pairs) in the primary list, and in the
                             overflow list, is cut evenly into groups of at most 32 tiles
                             (16 pairs); an entry holds the unit's position in its group in
                             bits 0..7 and the group's length in bits 8..15.  Unused -1 */
} mok_schedule_t;

/* Layer weights, [MoKDoc] _MoKRuntime.forward layouts.  The shared expert is
 * optional (I_s == 0 and NULL pointers).  In MOK_MODE_MXFP8_FWD the MXFP8
 * copies (codes uint8 row-major like the bf16 tensor, scales uint8 E8M0
 * [rows][K/32]) made by mok_mxfp8_quantize along each tensor's K axis
 * (gate/up: H; down: I or I_s) are required as well; the backward always
 * uses the bf16 tensors. */
typedef struct {
  int E, H, I, I_s;
  const uint16_t* w_gate;    /* [E][I][H] */
  const uint16_t* w_up;      /* [E][I][H] */
  const uint16_t* w_down;    /* [E][H][I] */
  const uint16_t* ws_gate;   /* [I_s][H] or NULL */
  const uint16_t* ws_up;     /* [I_s][H] or NULL */
  const uint16_t* ws_down;   /* [H][I_s] or NULL */
  const uint8_t* mx_gate;  const uint8_t* mx_gate_sc;   /* [E][I][H], [E][I][H/32] */
  const uint8_t* mx_up;    const uint8_t* mx_up_sc;     /* [E][I][H], [E][I][H/32] */
  const uint8_t* mx_down;  const uint8_t* mx_down_sc;   /* [E][H][I], [E][H][I/32] */
  const uint8_t* mxs_gate; const uint8_t* mxs_gate_sc;  /* [I_s][H], [I_s][H/32] */
  const uint8_t* mxs_up;   const uint8_t* mxs_up_sc;    /* [I_s][H], [I_s][H/32] */
  const uint8_t* mxs_down; const uint8_t* mxs_down_sc;  /* [H][I_s], [H][I_s/32] */
  /* MOK_MODE_MXFP8 only: each weight quantised along its leading axis (the
   * axis the backward's dgrad GEMMs contract over), as made by
   * mok_mxfp8_quantize_t: codes of the transpose, scales [..][leading/32]. */
  const uint8_t* mxt_gate;  const uint8_t* mxt_gate_sc;   /* [E][H][I], [E][H][I/32] */
  const uint8_t* mxt_up;    const uint8_t* mxt_up_sc;     /* [E][H][I], [E][H][I/32] */
  const uint8_t* mxt_down;  const uint8_t* mxt_down_sc;   /* [E][I][H], [E][I][H/32] */
  const uint8_t* mxts_gate; const uint8_t* mxts_gate_sc;  /* [H][I_s], [H][I_s/32] */
  const uint8_t* mxts_up;   const uint8_t* mxts_up_sc;    /* [H][I_s], [H][I_s/32] */
  const uint8_t* mxts_down; const uint8_t* mxts_down_sc;  /* [I_s][H], [I_s][H/32] */
} mok_weights_t;

/* Forward context: activations saved for the backward plus forward scratch,
 * all inside the caller's context buffer ([MoKDoc] _MoKRuntime.forward
 * returns an opaque context that _MoKRuntime.backward consumes). */
typedef struct {
  int T, k, E, H, I, I_s, mode, max_tiles;
  uint16_t* gu;       /* [max_tiles*128][2I] gate | up pre-activations per schedule row (saved) */
  uint16_t* h;        /* [max_tiles*128][I]  SwiGLU output, bf16 mode (scratch) */
  uint8_t*  hq;       /* [max_tiles*128][I]  SwiGLU output E4M3 codes, MXFP8 mode (scratch) */
  uint8_t*  hq_sc;    /* its E8M0 scales, tensor-core scale layout (below) */
  uint16_t* slots;    /* [max_tiles*128][H] router-weighted expert outputs in schedule order
                         (scratch; the combine reads row slot_row[t*k + j] for (t, j)).
                         The backward reuses it for its dx rows in schedule order. */
  uint16_t* gu_s;     /* [T][2 I_s] shared gate | up (saved) */
  uint16_t* h_s;      /* [T][I_s] shared SwiGLU output, bf16 mode (scratch) */
  uint8_t*  hq_s;     /* [T][I_s] shared SwiGLU output codes, MXFP8 mode */
  uint8_t*  hq_s_sc;  /* its scales, tensor-core scale layout (rows padded to 128) */
  uint16_t* shared_out; /* [T][H] shared expert output (scratch) */
  uint8_t*  xq;       /* [T][H] x codes in token order, MXFP8 mode (scratch) */
  uint8_t*  xq_sc;    /* their scales, tensor-core scale layout (rows padded to 128) */
  int32_t*  status;   /* device status word: MOK_OK or the first device error */
  uint16_t* x_perm;   /* [max_tiles*128][H] token rows of x in schedule order: the bf16 forward's
                         GEMM operand (MOK_DISPATCH_PERMUTE), or, in MOK_MODE_MXFP8_FWD, the bf16
                         backward's (written on the library's side stream during the forward) */
  int dispatch;       /* the dispatch the forward used */
  uint8_t*  xq_perm;  /* [max_tiles*128][H] x codes in schedule order, MXFP8 mode (scratch) */
  uint8_t*  xq_perm_sc; /* their scales, tensor-core scale layout */
  float swiglu_limit; /* the forward's mok_config_t.swiglu_limit */
  int64_t ring_rows;  /* 0: the forward ran in one pass and its schedule-order
                         scratch (x_perm, h, hq, xq_perm) spans the whole
                         schedule; else the rows of its macrobatch ring: that
                         scratch holds one window, and x_perm is NULL in
                         MOK_MODE_MXFP8_FWD */
} mok_ctx_t;
/* Tensor-core scale layout (MXFP8 context scratch): the E8M0 scales of a
 * [R][K] code tensor as 512-byte atoms, one per (128-row block rb, 128-column
 * group g), atom index rb * (K/128) + g; inside an atom, row r's scales of
 * the group's four 32-column blocks are the bytes of one 32-bit word at byte
 * (r % 32) * 16 + (r / 32) * 4, block b at byte b % 4 of it. */

/* Weight gradients (bf16, same layouts as the weights; shared ones NULL when
 * the layer has no shared expert). */
typedef struct {
  uint16_t* d_w_gate;   /* [E][I][H] */
  uint16_t* d_w_up;     /* [E][I][H] */
  uint16_t* d_w_down;   /* [E][H][I] */
  uint16_t* d_ws_gate;  /* [I_s][H] or NULL */
  uint16_t* d_ws_up;    /* [I_s][H] or NULL */
  uint16_t* d_ws_down;  /* [H][I_s] or NULL */
} mok_weight_grads_t;

/* ---- version / errors --------------------------------------------------- */
int mok_version(void);
const char* mok_last_error(void);

/* ---- schedule ([MoKEd] "The two API layers and the schedule object") ----
 * Bytes of the device buffer mok_schedule() carves its arrays from. */
size_t mok_schedule_bytes(int T, int k, int E);

/* Build the schedule for top_experts (device int64 [T][k]) over E experts.
 * capacity_multiplier (>= 0, finite) sets the per-expert tile budget
 * ceil(ceil(c*T)/128) of the static work table, with c*T rounded up in
 * double precision on exactly the caller's value ([MoKEd] "Tuning the five
 * hyperparameters before production": the worst-case fraction of tokens on
 * one expert); tiles beyond it go to an overflow list that follows the
 * primary list.  It changes the order of the tile list only, never a row or a
 * result.  `out` (host struct) receives pointers into `buf`.  An id outside
 * [0, E) sets status MOK_ERR_INDEX in header[2] and num_tiles = 0.
 * Limits: 1 <= k <= 64, 1 <= E <= 1024, T*k < 2^31. */
mok_status_t mok_schedule(const int64_t* top_experts, int T, int k, int E,
                          double capacity_multiplier, void* buf, size_t bytes,
                          mok_schedule_t* out, void* stream);

/* Synchronise `stream`'s work on the schedule and read its header.  Any of the
 * host output pointers may be NULL. */
mok_status_t mok_schedule_status(const mok_schedule_t* sched, int* status,
                                 int* num_tiles, int* P);

/* Schedule build for callers that cannot allocate device memory.  Some
 * callers own no device allocator of their own: code that runs inside
 * another framework's fixed memory pool, or a latency-bound loop that must
 * not call cudaMalloc because it can synchronise the device.  This call
 * builds the same schedule as mok_schedule(), bit for bit, but takes its
 * per-chunk histogram scratch from an array of fixed size that the library
 * itself holds in device memory, so `buf` holds only the output arrays
 * (mok_schedule_bytes(T, k, E) always suffices; the exact need is checked).
 * The pages have no counterpart to this call.
 *   - Limit: ceil(T*k / 1024) * E must not exceed 1048576 (a 4 MiB array);
 *     larger problems return MOK_ERR_INVALID_ARG with a message.  The array
 *     is held by every GPU that loads the library, until the process exits.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Every entry a build reads is first written by it, so nothing needs
 *     clearing, but calls that overlap on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 *   - No allocation of any kind happens in this call.
 * Arguments, outputs and errors are those of mok_schedule(). */
mok_status_t mok_schedule_noalloc(const int64_t* top_experts, int T, int k, int E,
                                  double capacity_multiplier, void* buf, size_t bytes,
                                  mok_schedule_t* out, void* stream);

/* ---- MXFP8 quantiser ([MoKEd] "Tuning the five hyperparameters before
 * production": weights are prequantised by a separate mxfp8_quantize) ----
 * x bf16 [rows][K] -> codes E4M3 [rows][K], scales E8M0 [rows][K/32].  Per
 * 1x32 block: s = smallest integer with amax <= 448 * 2^s (clamped to
 * [-127, 127]; s = 0 for an all-zero block), scale code s + 127, element code
 * = E4M3 round-to-nearest-even of v / 2^s with saturation; a value that
 * rounds to zero keeps its sign.  Inputs must be finite.  K % 32 == 0. */
mok_status_t mok_mxfp8_quantize(const uint16_t* x, int64_t rows, int K,
                                uint8_t* codes, uint8_t* scales, void* stream);

/* Transposing MXFP8 quantiser for the MOK_MODE_MXFP8 backward (the weights'
 * copies quantised along their leading axis, [MoKEd] "Tuning the five
 * hyperparameters before production": weights are prequantised by the
 * caller).  x bf16 [batch][rows][cols] -> codes E4M3 [batch][cols][rows] (the
 * transpose) and scales E8M0 [batch][cols][rows/32]: one scale per 32
 * consecutive rows of each column, with the block rule of
 * mok_mxfp8_quantize.  Needs rows % 32 == 0 and cols % 64 == 0; inputs
 * finite; x and codes 16-byte aligned. */
mok_status_t mok_mxfp8_quantize_t(const uint16_t* x, int64_t batch, int rows, int cols,
                                  uint8_t* codes, uint8_t* scales, void* stream);

/* Both orientations from one read of x: the output of mok_mxfp8_quantize
 * (codes [batch][rows][cols], scales [batch][rows][cols/32]) and that of
 * mok_mxfp8_quantize_t (codes_t [batch][cols][rows], scales_t
 * [batch][cols][rows/32]), bit for bit.  This is the MOK_MODE_MXFP8 weight
 * prequantisation: a weight needs its forward copy (blocks along K) and its
 * backward copy (blocks along the leading axis).  Same conditions as
 * mok_mxfp8_quantize_t; codes and codes_t 16-byte aligned. */
mok_status_t mok_mxfp8_quantize_dual(const uint16_t* x, int64_t batch, int rows, int cols,
                                     uint8_t* codes, uint8_t* scales, uint8_t* codes_t,
                                     uint8_t* scales_t, void* stream);

/* ---- forward ([MoKDoc] _MoKRuntime.forward) -----------------------------
 * y[t] = S(x[t]) + sum_j w[t,j] * F_{e[t,j]}(x[t]),
 * F_e(v) = W_down[e] (silu(W_gate[e] v) * (W_up[e] v)), S the same with the
 * shared weights.  Deterministic: every output element is summed in a fixed
 * order (shared term, then j ascending) with no floating-point atomics.
 * Shape contract: H % 128 == 0, I % 128 == 0, I_s % 128 == 0, T >= 1.
 * x bf16 [T][H]; router_w fp32 [T][k]; y bf16 [T][H].  The context buffer
 * (mok_ctx_bytes) must stay alive and unmodified until mok_backward. */
size_t mok_ctx_bytes(int T, int k, int E, int H, int I, int I_s, int mode);
/* The context bytes for mok_config_t.macrobatch_size (0: mok_ctx_bytes). */
size_t mok_ctx_bytes_ring(int T, int k, int E, int H, int I, int I_s, int mode, int64_t macrobatch_size);
mok_status_t mok_forward(const mok_config_t* cfg, const uint16_t* x,
                         const float* router_w, const mok_schedule_t* sched,
                         const mok_weights_t* w, uint16_t* y, void* ctx_buf,
                         size_t ctx_bytes, mok_ctx_t* ctx, void* stream);

/* Synchronise and read the context's device status word. */
mok_status_t mok_ctx_status(const mok_ctx_t* ctx, int* status);

/* ---- backward ([MoKDoc] _MoKRuntime.backward) ---------------------------
 * Exact gradients of the forward given dy = dL/dy (bf16 [T][H]); in the
 * MXFP8 modes the derivative treats the quantisers as the identity and is
 * taken at the saved gate/up pre-activations.  The backward runs in the mode
 * the forward recorded in the context: bf16 GEMMs after MOK_MODE_BF16 and
 * MOK_MODE_MXFP8_FWD, MXFP8 GEMMs after MOK_MODE_MXFP8 (which needs the
 * weights' mxt* copies).  In MOK_MODE_MXFP8 every backward GEMM quantises
 * both of its operands in blocks of 32 along its own contraction axis; for
 * the weight gradients that axis is the expert's rows in schedule order.
 * The quantisers see bf16 values: dy, x, the saved gate/up, and the bf16
 * roundings of dG, dU and w*h.  x and router_w are the forward's inputs.  Outputs:
 * dx bf16 [T][H], d_router_w fp32 [T][k] (= <dy[t], F_e(x[t])>), the six
 * weight gradients.  Scratch comes from `ws` (mok_bwd_workspace_bytes with
 * the context's mode) and from the context's slots, the forward's scratch,
 * which receive the dx rows in schedule order; the saved activations are only
 * read, so the backward may run again on the same context.  Device errors
 * land in ctx->status. */
size_t mok_bwd_workspace_bytes(int T, int k, int E, int H, int I, int I_s, int mode);
/* The workspace bytes for mok_config_t.macrobatch_size (0:
 * mok_bwd_workspace_bytes).  The backward's ring is its own: it need not
 * match the forward's. */
size_t mok_bwd_workspace_bytes_ring(int T, int k, int E, int H, int I, int I_s, int mode,
                                    int64_t macrobatch_size);

/* ---- macrobatch windows ([MoKEd] "Tuning the five hyperparameters before
 * production": macrobatch_size) ----------------------------------------
 * The windows a ring of macrobatch_size rows (rounded up to a multiple of
 * 128) runs the routed experts in, from the per-expert row counts cnt (a
 * HOST array of E counts, as the schedule's cnt): experts in order, each
 * padded to a multiple of 128 rows; a window takes the next expert while its
 * padded rows still fit the ring, else the next window starts there.
 * first_expert (HOST, E + 1 entries) receives each window's first expert and
 * then E; *num_windows their number (>= 1).  macrobatch_size 0 gives one
 * window.  An expert whose padded rows exceed the ring: MOK_ERR_CAPACITY.
 * Host only: needs no GPU. */
mok_status_t mok_macrobatch_plan(const int32_t* cnt, int E, int64_t macrobatch_size, int32_t* first_expert,
                                 int* num_windows);
mok_status_t mok_backward(const mok_config_t* cfg, const uint16_t* dy,
                          const uint16_t* x, const float* router_w,
                          const mok_schedule_t* sched, const mok_ctx_t* ctx,
                          const mok_weights_t* w, uint16_t* dx,
                          float* d_router_w, const mok_weight_grads_t* grads,
                          void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H */

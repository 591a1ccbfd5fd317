"""CPU oracle for the Mixture-of-Kittens (MoK) routed-plus-shared SwiGLU MoE layer.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously-correct
definition that the CUDA library is checked against.  It shares no code with
the CUDA path and must never be imported by it.  Floating point runs in
float64 (NumPy); contractions use ``numpy.matmul`` as a library step; the
schedule is a plain Python loop; the MXFP8 codec is the textbook definition.

Sources (page title, section):
  [MoKDoc]  "nemo_automodel.components.moe.mok_experts" (NVIDIA NeMo AutoModel
            API docs): ``GroupedExpertsMoK.forward`` ("Execute fused shared and
            routed SwiGLU experts", operand shapes/dtypes), ``_MoKRuntime.forward``
            / ``_MoKRuntime.backward`` (what forward returns, which gradients
            backward returns), ``down_proj_bias`` (no expert bias).
  [MoKEd]   "Mixture-of-Kittens: a deterministic MoE megakernel for NVL72
            racks": "The two API layers and the schedule object" (schedule is
            built once, before any kernel, and makes the layer deterministic),
            "Tuning the five hyperparameters before production"
            (schedule_capacity_multiplier, MXFP8 weights prequantised by
            mxfp8_quantize), "Where MoK is the wrong tool" (top-k experts int64
            [tokens, topk], router weights float32, router outside the library).
  [MoKBlog] "Mixture of Kittens" code review: "How It Is Wired" (schedule,
            mxfp8_quantize as primitive kernels).
  [OCP-MX]  OCP Microscaling Formats (MX) v1.0: E4M3 element encoding (bias 7,
            max normal 448, no infinities, one NaN pattern per sign) and E8M0
            scale encoding (2^(code-127)).  The pages only say "MXFP8"; the
            1x32 block, E8M0 scale and E4M3 element come from the workload
            definition of the MXFP8 configurations.

Readings where the pages are silent (each listed with its reasoning in the
design notes): the router weight scales the expert output; the shared expert
is added unweighted; rows of an expert are ordered by flat index f = t*k + j;
an out-of-range expert id is an error; the E8M0 scale is the smallest power
of two that brings the block amax to <= 448 (no clipping); an all-zero block
gets scale 2^0; a negative value that rounds to zero keeps its sign bit; the
MXFP8 backward is straight-through (quantisation treated as identity) and is
evaluated at the gate/up pre-activations of the quantised forward; in the
fully MXFP8 backward every backward contraction takes both operands quantised
in blocks of 32 along its own contraction axis (for the weight gradients, 32
consecutive rows of an expert in schedule order), from the bf16 values the
backward holds; ``swiglu_limit`` is the usual clamped SwiGLU (gate <= L, up
in [-L, L]).
"""
from __future__ import annotations

import math

import numpy as np

TILE_ROWS = 128  # rows per expert tile; each expert's row range is padded to it

# status words (same numeric meaning as the C library's)
STATUS_OK = 0
STATUS_INDEX = 2


# ---------------------------------------------------------------------------
# Schedule  ([MoKEd] "The two API layers and the schedule object";
#            [MoKEd] "Tuning the five hyperparameters before production")
# ---------------------------------------------------------------------------

def max_tiles(T: int, k: int, E: int) -> int:
    """Upper bound on the number of 128-row tiles: sum_e ceil(cnt_e/128) with
    sum_e cnt_e = T*k is at most floor((T*k + 127*E) / 128)."""
    return (T * k + (TILE_ROWS - 1) * E) // TILE_ROWS


def capacity_tiles(T: int, capacity_multiplier: float, mt: int) -> int:
    """Per-expert tile budget of the static work table: the multiplier is the
    worst-case fraction of the T tokens that land on one expert, rounded up to
    whole rows and then to whole 128-row tiles.  Decided in float64."""
    rows = math.ceil(float(capacity_multiplier) * float(T))
    return min((rows + TILE_ROWS - 1) // TILE_ROWS, mt)


def build_schedule(top_experts, E: int, capacity_multiplier: float = 0.5) -> dict:
    """Dispatch/combine schedule for one batch of routing decisions.

    ``top_experts`` is int64 [T, k].  Flat routed row index f = t*k + j.
    Rows of expert e occupy schedule rows [row0[e], row0[e] + cnt[e]) in
    ascending f (stable), and the range is padded to a multiple of 128.
    Padding rows and unused tail entries hold -1.

    Tile list: first every expert's first ``capacity_tiles`` tiles (expert
    ascending), then the tiles beyond that budget (the overflow list, expert
    ascending).  Tile membership never depends on the multiplier; only the
    order of the list does.

    Returns int32 arrays sized exactly like the device buffers.
    """
    te = np.asarray(top_experts, dtype=np.int64)
    T, k = te.shape
    n = T * k
    flat = te.reshape(-1)
    mt = max_tiles(T, k, E)
    out = {
        "cnt": np.zeros(E, np.int32),
        "row0": np.zeros(E + 1, np.int32),
        "row_src": np.full(mt * TILE_ROWS, -1, np.int32),
        "slot_row": np.full(n, -1, np.int32),
        "tile_expert": np.full(mt, -1, np.int32),
        "tile_row0": np.full(mt, -1, np.int32),
        "tile_rows": np.full(mt, -1, np.int32),
        "num_tiles": 0,
        "num_primary": 0,
        "P": 0,
        "status": STATUS_OK,
    }
    # validate: every id must name one of the E experts
    for f in range(n):
        if flat[f] < 0 or flat[f] >= E:
            out["status"] = STATUS_INDEX
            return out
    # histogram
    cnt = [0] * E
    for f in range(n):
        cnt[int(flat[f])] += 1
    # exclusive scan of the padded counts
    row0 = [0] * (E + 1)
    for e in range(E):
        padded = (cnt[e] + TILE_ROWS - 1) // TILE_ROWS * TILE_ROWS
        row0[e + 1] = row0[e] + padded
    # stable scatter in flat order
    fill = list(row0[:E])
    row_src = out["row_src"]
    slot_row = out["slot_row"]
    for f in range(n):
        e = int(flat[f])
        p = fill[e]
        fill[e] += 1
        row_src[p] = f
        slot_row[f] = p
    # tile list with the capacity split
    cap = capacity_tiles(T, capacity_multiplier, mt)
    tiles_primary, tiles_overflow = [], []
    for e in range(E):
        ntile = (cnt[e] + TILE_ROWS - 1) // TILE_ROWS
        for i in range(ntile):
            r0 = row0[e] + i * TILE_ROWS
            rows = min(TILE_ROWS, cnt[e] - i * TILE_ROWS)
            (tiles_primary if i < cap else tiles_overflow).append((e, r0, rows))
    tiles = tiles_primary + tiles_overflow
    for i, (e, r0, rows) in enumerate(tiles):
        out["tile_expert"][i] = e
        out["tile_row0"][i] = r0
        out["tile_rows"][i] = rows
    out["cnt"][:] = cnt
    out["row0"][:] = row0
    out["num_tiles"] = len(tiles)
    out["num_primary"] = len(tiles_primary)
    out["P"] = row0[E]
    return out


# ---------------------------------------------------------------------------
# MXFP8 codec  ([MoKEd] "Tuning the five hyperparameters before production":
#               weights are prequantised to MXFP8 by mxfp8_quantize; [OCP-MX])
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0
MX_BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 code bytes -> float64 values ([OCP-MX] E4M3: sign, 4-bit exponent
    with bias 7, 3-bit mantissa; exponent field 0 is subnormal with scale
    2^-6; 0x7F/0xFF are NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    mf = c & 0x7
    normal = np.ldexp(1.0 + mf / 8.0, (ef - 7).astype(np.int64))
    sub = np.ldexp(mf / 8.0, -6)
    v = sign * np.where(ef == 0, sub, normal)
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return v


def e4m3_encode(y) -> np.ndarray:
    """float64 -> E4M3 codes: round to nearest, ties to even, saturating at
    +-448.  A value whose magnitude rounds to zero keeps its sign bit."""
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.minimum(np.abs(y), E4M3_MAX)
    # quantum of the binade that holds a; binades below 2^-6 share 2^-9
    _, e = np.frexp(a)                      # a = m * 2^e, m in [0.5, 1)
    ex = np.maximum(e - 1, -6)              # a in [2^ex, 2^(ex+1)) or subnormal
    q = np.ldexp(1.0, (ex - 3).astype(np.int64))
    v = np.rint(a / q) * q                  # np.rint rounds half to even
    v = np.minimum(v, E4M3_MAX)
    # encode the rounded magnitude
    _, e2 = np.frexp(v)
    ex2 = e2 - 1
    is_sub = v < 2.0 ** -6
    sub_m = np.rint(v / 2.0 ** -9).astype(np.int64)          # 0..7
    ex2c = np.clip(ex2, -6, 8).astype(np.int64)
    nrm_m = np.rint((v / np.ldexp(1.0, ex2c) - 1.0) * 8.0).astype(np.int64)
    nrm_code = ((ex2c + 7) << 3) | nrm_m
    mag = np.where(is_sub, sub_m, nrm_code)
    return (mag | np.where(neg, 0x80, 0)).astype(np.uint8)


def e8m0_scale_exponent(amax) -> np.ndarray:
    """Shared block exponent s: the smallest integer with amax <= 448 * 2^s,
    clamped to [-127, 127]; s = 0 when amax == 0.  Decided exactly from the
    binary exponent and mantissa of amax (no floating-point log)."""
    amax = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(amax)                   # amax = m * 2^e, m in [0.5, 1)
    # amax/448 = (2m / 1.75) * 2^(e-1-8); 2m in [1, 2)
    s = (e - 1 - 8) + (2.0 * m > 1.75)
    s = np.clip(s, -127, 127)
    return np.where(amax == 0, 0, s).astype(np.int64)


def mxfp8_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """[R, K] values -> (E4M3 codes uint8 [R, K], E8M0 scale codes uint8
    [R, K/32]).  One scale per 1x32 block along the contiguous K axis."""
    x = np.asarray(x, dtype=np.float64)
    R, K = x.shape
    assert K % MX_BLOCK == 0
    blocks = x.reshape(R, K // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    s = e8m0_scale_exponent(amax)
    y = blocks * np.ldexp(1.0, -s)[:, :, None]   # exact power-of-two scaling
    codes = e4m3_encode(y).reshape(R, K)
    return codes, (s + 127).astype(np.uint8)


def mxfp8_dequantize(codes, scales) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    R, K = codes.shape
    s = np.asarray(scales, np.uint8).astype(np.int64) - 127
    v = e4m3_decode(codes).reshape(R, K // MX_BLOCK, MX_BLOCK)
    return (v * np.ldexp(1.0, s)[:, :, None]).reshape(R, K)


def mxfp8_roundtrip(x) -> np.ndarray:
    """Quantise then dequantise (the value the MXFP8 GEMMs actually see)."""
    return mxfp8_dequantize(*mxfp8_quantize(x))


# ---------------------------------------------------------------------------
# The layer  ([MoKDoc] GroupedExpertsMoK.forward, _MoKRuntime.forward/backward)
# ---------------------------------------------------------------------------

def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):          # torch tensor (bf16 widens exactly)
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), via float32: the top
    16 bits of the float32 pattern after round-to-nearest-even."""
    b = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def clamp_gate_up(g, u, limit):
    """The ``swiglu_limit`` of [MoKDoc] _MoKRuntime (named there, not
    defined), read as the usual clamped SwiGLU: with limit > 0 the gate
    pre-activation is clamped from above at limit and the up pre-activation
    to [-limit, limit] before the SwiGLU; limit <= 0 (the default) leaves
    both as they are."""
    if not limit or limit <= 0:
        return g, u
    return np.minimum(g, limit), np.clip(u, -limit, limit)


def _expert(v, wg, wu, wd, limit=0.0):
    """F(v) = W_down (silu(W_gate v) * (W_up v)) for a batch of rows v [n, H]
    (gate/up clamped by ``clamp_gate_up``).  Returns (output [n, H], g [n, I],
    u [n, I], h [n, I])."""
    g = v @ wg.T
    u = v @ wu.T
    gc, uc = clamp_gate_up(g, u, limit)
    h = silu(gc) * uc
    return h @ wd.T, g, u, h


def layer_forward(x, router_w, top_experts, w_gate, w_up, w_down,
                  ws_gate=None, ws_up=None, ws_down=None, swiglu_limit=0.0):
    """y[t] = S(x[t]) + sum_j w[t,j] * F_{e[t,j]}(x[t])   (float64).

    Shapes ([MoKDoc] _MoKAutogradFunction.forward): x [T, H]; router_w [T, k]
    float32; top_experts [T, k] int64; routed gate/up [E, I, H], down
    [E, H, I]; shared gate/up [I_s, H], down [H, I_s] (absent -> no shared
    expert).  No expert bias ([MoKDoc] down_proj_bias).  ``swiglu_limit``:
    see ``clamp_gate_up`` (routed and shared experts alike).
    """
    x, w = _f64(x), _f64(router_w)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    te = np.asarray(top_experts if not hasattr(top_experts, "numpy")
                    else top_experts.cpu().numpy(), np.int64)
    T, H = x.shape
    E = wg.shape[0]
    y = np.zeros((T, H))
    if ws_gate is not None:
        y += _expert(x, _f64(ws_gate), _f64(ws_up), _f64(ws_down), swiglu_limit)[0]
    for e in range(E):
        t_idx, j_idx = np.nonzero(te == e)
        if t_idx.size == 0:
            continue
        o = _expert(x[t_idx], wg[e], wu[e], wd[e], swiglu_limit)[0]
        np.add.at(y, t_idx, w[t_idx, j_idx][:, None] * o)
    return y


def layer_backward(x, router_w, top_experts, w_gate, w_up, w_down, dy,
                   ws_gate=None, ws_up=None, ws_down=None, gu_override=None, swiglu_limit=0.0):
    """Exact gradients of ``layer_forward`` given dL/dy = dy (float64).

    Returns dict: dx [T,H], d_router_w [T,k], d_w_gate/d_w_up [E,I,H],
    d_w_down [E,H,I], and d_ws_gate/d_ws_up [I_s,H], d_ws_down [H,I_s] when a
    shared expert is present ([MoKDoc] _MoKRuntime.backward: gradients for x,
    router weights, the three routed weights and the shared weights).

    ``gu_override`` (used by the MXFP8 straight-through backward) supplies the
    gate/up pre-activations to evaluate the derivative at: a callable
    (expert or None, v) -> (g, u).
    With ``swiglu_limit`` > 0 the clamp of ``clamp_gate_up`` is
    differentiated as the clamp itself: the gate gradient passes where
    g <= limit, the up gradient where |u| <= limit (the bounds included),
    decided on the float64 g and u.
    """
    x, w, dy = _f64(x), _f64(router_w), _f64(dy)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    te = np.asarray(top_experts if not hasattr(top_experts, "numpy")
                    else top_experts.cpu().numpy(), np.int64)
    T, H = x.shape
    k = te.shape[1]
    E = wg.shape[0]
    dx = np.zeros_like(x)
    dw = np.zeros((T, k))
    dwg, dwu, dwd = np.zeros_like(wg), np.zeros_like(wu), np.zeros_like(wd)

    def one(e, v, scale, dyv, Wg, Wu, Wd):
        if gu_override is None:
            g, u = v @ Wg.T, v @ Wu.T
        else:
            g, u = gu_override(e, v)
        gc, uc = clamp_gate_up(g, u, swiglu_limit)
        sg = sigmoid(gc)
        h = gc * sg * uc
        o = h @ Wd.T
        d_scale = np.sum(dyv * o, axis=1)            # <dy, F(x)>
        dh = scale[:, None] * (dyv @ Wd)              # w * W_down^T dy
        dWd = (scale[:, None] * dyv).T @ h            # dy (w h)^T
        dg = dh * uc * sg * (1.0 + gc * (1.0 - sg))   # silu'(g) = s (1 + g (1 - s))
        du = dh * gc * sg
        if swiglu_limit and swiglu_limit > 0:         # the clamp's own derivative
            lim = float(np.float32(swiglu_limit))
            dg = dg * (g <= lim)
            du = du * (np.abs(u) <= lim)
        dWg = dg.T @ v
        dWu = du.T @ v
        dv = dg @ Wg + du @ Wu
        return d_scale, dv, dWg, dWu, dWd

    out = {}
    if ws_gate is not None:
        sg_, su_, sd_ = _f64(ws_gate), _f64(ws_up), _f64(ws_down)
        _, dv, dWg, dWu, dWd = one(None, x, np.ones(T), dy, sg_, su_, sd_)
        dx += dv
        out["d_ws_gate"], out["d_ws_up"], out["d_ws_down"] = dWg, dWu, dWd
    for e in range(E):
        t_idx, j_idx = np.nonzero(te == e)
        if t_idx.size == 0:
            continue
        d_scale, dv, dWg, dWu, dWd = one(e, x[t_idx], w[t_idx, j_idx], dy[t_idx],
                                         wg[e], wu[e], wd[e])
        dw[t_idx, j_idx] = d_scale
        np.add.at(dx, t_idx, dv)
        dwg[e] += dWg
        dwu[e] += dWu
        dwd[e] += dWd
    out.update(dx=dx, d_router_w=dw, d_w_gate=dwg, d_w_up=dwu, d_w_down=dwd)
    return out


def layer_forward_mxfp8(x, router_w, top_experts, w_gate, w_up, w_down,
                        ws_gate=None, ws_up=None, ws_down=None, swiglu_limit=0.0):
    """MXFP8 forward with the quantisation the MXFP8 configurations define:
    x (along H), every weight (along its K axis: H for gate/up, I for down)
    and the intermediate activation h (along I) are quantised to E4M3 with one
    E8M0 scale per 1x32 block; products are exact and accumulate in float64
    here.  Routed and shared experts are treated alike.
    """
    x, w = _f64(x), _f64(router_w)
    te = np.asarray(top_experts if not hasattr(top_experts, "numpy")
                    else top_experts.cpu().numpy(), np.int64)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    T, H = x.shape
    E = wg.shape[0]
    xq = mxfp8_roundtrip(x)

    def expert_q(v, Wg, Wu, Wd):
        g = v @ mxfp8_roundtrip(Wg).T
        u = v @ mxfp8_roundtrip(Wu).T
        g, u = clamp_gate_up(g, u, swiglu_limit)
        h = mxfp8_roundtrip(silu(g) * u)
        return h @ mxfp8_roundtrip(Wd).T

    y = np.zeros((T, H))
    if ws_gate is not None:
        y += expert_q(xq, _f64(ws_gate), _f64(ws_up), _f64(ws_down))
    for e in range(E):
        t_idx, j_idx = np.nonzero(te == e)
        if t_idx.size == 0:
            continue
        o = expert_q(xq[t_idx], wg[e], wu[e], wd[e])
        np.add.at(y, t_idx, w[t_idx, j_idx][:, None] * o)
    return y


def layer_backward_mxfp8(x, router_w, top_experts, w_gate, w_up, w_down, dy,
                         ws_gate=None, ws_up=None, ws_down=None, swiglu_limit=0.0):
    """Backward of the MXFP8 forward in BF16 weights, straight-through: the
    derivative treats every quantiser as the identity and is evaluated at the
    gate/up pre-activations g, u that the quantised forward produced.
    Weight gradients contract against the unquantised x."""
    xq = mxfp8_roundtrip(_f64(x))
    wg, wu = _f64(w_gate), _f64(w_up)
    shared = (None if ws_gate is None else
              (mxfp8_roundtrip(_f64(ws_gate)), mxfp8_roundtrip(_f64(ws_up))))
    routed_q = {}

    def gu(e, v):
        # v is a block of rows of the unquantised x; recover their quantised
        # version row-for-row (quantisation is per row, so it commutes).
        vq = mxfp8_roundtrip(v)
        if e is None:
            qg, qu = shared
        else:
            if e not in routed_q:
                routed_q[e] = (mxfp8_roundtrip(wg[e]), mxfp8_roundtrip(wu[e]))
            qg, qu = routed_q[e]
        return vq @ qg.T, vq @ qu.T

    del xq
    return layer_backward(x, router_w, top_experts, w_gate, w_up, w_down, dy,
                          ws_gate, ws_up, ws_down, gu_override=gu, swiglu_limit=swiglu_limit)


# ---------------------------------------------------------------------------
# MXFP8 backward  ([MoKEd] "Where MoK is the wrong tool": the MXFP8 backward
#                  is one of the two measured layer passes; [OCP-MX])
# ---------------------------------------------------------------------------

def mxfp8_roundtrip_cols(m) -> np.ndarray:
    """Quantise then dequantise along axis 0: every column is cut into blocks
    of 32 consecutive rows (rows past the end count as zeros, which leave the
    block amax unchanged), each block with its own E8M0 scale."""
    m = np.asarray(m, dtype=np.float64)
    R, C = m.shape
    pad = (-R) % MX_BLOCK
    mp = np.vstack([m, np.zeros((pad, C))]) if pad else m
    return mxfp8_roundtrip(mp.T).T[:R]


def layer_backward_mxfp8_full(x, router_w, top_experts, w_gate, w_up, w_down, dy,
                              ws_gate=None, ws_up=None, ws_down=None, swiglu_limit=0.0):
    """Backward of the MXFP8 forward with every backward GEMM on MXFP8
    operands too (E4M3 values, one E8M0 scale per 32 elements along that
    GEMM's contraction axis, exact products, float64 sums here):

      dgrad through down     Z = dy . W_down[e]      dy rows along H;
                                                     W_down[e] [H, I] along H
      dgrad through gate/up  dx = dG W_gate + dU W_up  dG|dU rows along I;
                                                     W_gate[e], W_up[e] [I, H] along I
      weight gradients       dW_down = dy^T (w h), dW_gate = dG^T x, dW_up = dU^T x:
                             both operands along the expert's rows, in
                             schedule order (ascending f = t*k + j), 32
                             consecutive rows per block; the shared expert
                             takes 32 consecutive tokens per block.

    The quantisers see the values the backward holds in bf16: the inputs dy
    and x and the bf16 weights; the gate/up pre-activations of the quantised
    forward as the forward saves them (rounded to bf16); dG, dU and w h
    rounded to bf16.  The derivative is straight-through (quantisers count as
    the identity); the router-weight gradient is <Z, h>; the clamp of
    ``clamp_gate_up`` is differentiated as in ``layer_backward``.
    Returns the dict of ``layer_backward``.
    """
    x, w, dy = _f64(x), _f64(router_w), _f64(dy)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    te = np.asarray(top_experts if not hasattr(top_experts, "numpy")
                    else top_experts.cpu().numpy(), np.int64)
    T, H = x.shape
    k = te.shape[1]
    E = wg.shape[0]
    xq = mxfp8_roundtrip(x)
    rows_q = mxfp8_roundtrip
    cols_q = mxfp8_roundtrip_cols
    lim = float(np.float32(swiglu_limit)) if swiglu_limit and swiglu_limit > 0 else 0.0

    def one(v, vq, scale, dyv, Wg, Wu, Wd):
        # the forward's pre-activations (quantised operands), kept as bf16
        g = round_bf16(vq @ rows_q(Wg).T)
        u = round_bf16(vq @ rows_q(Wu).T)
        gc, uc = clamp_gate_up(g, u, lim)
        sg = sigmoid(gc)
        h = gc * sg * uc
        z = rows_q(dyv) @ cols_q(Wd)                   # [n, I]
        d_scale = np.sum(z * h, axis=1)
        dh = scale[:, None] * z
        dg = dh * uc * sg * (1.0 + gc * (1.0 - sg))
        du = dh * gc * sg
        if lim > 0:
            dg = dg * (g <= lim)
            du = du * (np.abs(u) <= lim)
        dg, du = round_bf16(dg), round_bf16(du)
        hw = round_bf16(scale[:, None] * h)
        dWd = cols_q(dyv).T @ cols_q(hw)
        vc = cols_q(v)
        dWg = cols_q(dg).T @ vc
        dWu = cols_q(du).T @ vc
        dv = rows_q(dg) @ cols_q(Wg) + rows_q(du) @ cols_q(Wu)
        return d_scale, dv, dWg, dWu, dWd

    dx = np.zeros_like(x)
    dw = np.zeros((T, k))
    dwg, dwu, dwd = np.zeros_like(wg), np.zeros_like(wu), np.zeros_like(wd)
    out = {}
    if ws_gate is not None:
        _, dv, dWg, dWu, dWd = one(x, xq, np.ones(T), dy, _f64(ws_gate), _f64(ws_up), _f64(ws_down))
        dx += dv
        out["d_ws_gate"], out["d_ws_up"], out["d_ws_down"] = dWg, dWu, dWd
    for e in range(E):
        t_idx, j_idx = np.nonzero(te == e)            # row-major: ascending f
        if t_idx.size == 0:
            continue
        d_scale, dv, dWg, dWu, dWd = one(x[t_idx], xq[t_idx], w[t_idx, j_idx], dy[t_idx],
                                         wg[e], wu[e], wd[e])
        dw[t_idx, j_idx] = d_scale
        np.add.at(dx, t_idx, dv)
        dwg[e] += dWg
        dwu[e] += dWu
        dwd[e] += dWd
    out.update(dx=dx, d_router_w=dw, d_w_gate=dwg, d_w_up=dwu, d_w_down=dwd)
    return out

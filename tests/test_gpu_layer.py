"""GPU parity of the layer forward and backward against the CPU oracle, plus
determinism, invariance and device-error checks."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import (BF16_TOL, MX_UNQ_TOL, clamp_limit, compare_all, mok, oracle_args, oracle_fwd_bwd,
                            rel_l2, run_layer, subset_inputs, weights_of)

pytestmark = pytest.mark.gpu

# (T, H, I, E, k, I_s, skew): the tiny layer, a ragged-T layer with a shared
# expert whose I is not a multiple of 256, a skewed layer with empty and hot
# experts (several tiles), and a 2-tile-wide H with a 1-expert layer.
SHAPES = {
    "tiny": (128, 128, 256, 8, 2, 0, None),
    "ragged_shared": (200, 256, 384, 5, 3, 256, None),
    "skewed": (333, 128, 128, 16, 4, 0, 1.2),
    "one_expert": (300, 384, 128, 1, 1, 128, None),
    "wide": (520, 512, 256, 12, 6, 384, 1.2),
}
# a deep H for the MXFP8 paths: 132 blocks of 32 a row (not a whole number of
# 32-block chunks) in 33 column groups of the scale layout (more than one pass
# of the scale layouts' 16- and 32-group loops)
EXTRA_SHAPES = {"deep_h": (300, 4224, 128, 4, 2, 128, None)}


def _inputs(name, seed=0):
    T, H, I, E, k, I_s, skew = SHAPES[name] if name in SHAPES else EXTRA_SHAPES[name]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=seed)
    inp.meta.update(name=name)
    return inp


@pytest.mark.parametrize("name", list(SHAPES))
def test_bf16_forward_backward_matches_oracle(name):
    inp = _inputs(name)
    y, grads, sched, ctx = run_layer(inp, "bf16")
    assert ctx.status() == 0
    y_ref, g_ref = oracle_fwd_bwd(inp, "bf16")
    errs, bad = compare_all(y, grads, y_ref, g_ref, BF16_TOL)
    assert not bad, errs


@pytest.mark.parametrize("name", list(SHAPES) + ["deep_h"])
def test_mxfp8_forward_matches_same_quantisation_oracle(name):
    inp = _inputs(name, seed=1)
    y, grads, sched, ctx = run_layer(inp, "mxfp8")
    assert ctx.status() == 0
    y_ref, g_ref = oracle_fwd_bwd(inp, "mxfp8")
    errs, bad = compare_all(y, grads, y_ref, g_ref, BF16_TOL)
    assert not bad, errs
    # Against the unquantised layer: quantising x, W_gate, W_up, h and W_down to
    # E4M3 (3 mantissa bits) puts the oracle's own MXFP8 forward about 6.5e-2
    # (rel-L2) away from the unquantised one, above a 3e-2 bound.  The GPU may add
    # no more than the same-quantisation tolerance to that intrinsic gap.
    y_unq = oracle.layer_forward(*oracle_args(inp))
    intrinsic = rel_l2(y_ref, y_unq)
    assert rel_l2(y, y_unq) <= max(MX_UNQ_TOL, intrinsic + BF16_TOL), (rel_l2(y, y_unq), intrinsic)


@pytest.mark.parametrize("name", list(SHAPES) + ["deep_h"])
def test_mxfp8_full_backward_matches_same_quantisation_oracle(name):
    """MXFP8 forward and backward: every backward GEMM on block-scaled E4M3
    operands, against the oracle that quantises the same operands along the
    same axes."""
    inp = _inputs(name, seed=9)
    y, grads, sched, ctx = run_layer(inp, "mxfp8_full")
    assert ctx.status() == 0
    y_ref, g_ref = oracle_fwd_bwd(inp, "mxfp8_full")
    errs, bad = compare_all(y, grads, y_ref, g_ref, BF16_TOL)
    assert not bad, errs


@pytest.mark.parametrize("mode,seed", [("bf16", 2), ("mxfp8", 11), ("mxfp8_full", 10)])
def test_repeated_runs_bitwise_identical(mode, seed):
    inp = _inputs("wide", seed=seed)
    a = run_layer(inp, mode)
    b = run_layer(inp, mode)
    assert torch.equal(a[0], b[0])
    for key in a[1]:
        assert torch.equal(a[1][key], b[1][key]), key


@pytest.mark.parametrize("mode", ["bf16", "mxfp8", "mxfp8_full"])
def test_capacity_and_minibatch_change_no_bit(mode):
    inp = _inputs("skewed", seed=3)
    base = run_layer(inp, mode, capacity=1.0, minibatch=0)
    for c, mb in ((0.0, 0), (0.05, 64), (0.5, 128), (3.0, 1)):
        other = run_layer(inp, mode, capacity=c, minibatch=mb)
        assert torch.equal(base[0], other[0]), (c, mb)
        for key in base[1]:
            assert torch.equal(base[1][key], other[1][key]), (c, mb, key)


def test_zero_router_weights_give_shared_expert_only():
    inp = _inputs("ragged_shared", seed=4)
    inp.router_w.zero_()
    y, grads, _, _ = run_layer(inp, "bf16")
    y_ref, g_ref = oracle_fwd_bwd(inp, "bf16")
    assert rel_l2(y, y_ref) <= BF16_TOL
    assert grads["d_w_down"].abs().max().item() == 0.0
    assert rel_l2(grads["d_router_w"], g_ref["d_router_w"]) <= BF16_TOL


def test_bounded_wait_reports_timeout_and_context_survives():
    m = mok()
    inp = _inputs("tiny", seed=5)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    y, ctx = m.forward(g.x, g.router_w, sched, w, debug=1)   # withholds one accumulator signal
    assert ctx.status() == 5                                  # MOK_ERR_TIMEOUT
    # the context is still usable: a normal call afterwards is correct
    y2, ctx2 = m.forward(g.x, g.router_w, sched, w)
    assert ctx2.status() == 0
    y_ref = oracle.layer_forward(*oracle_args(inp))
    assert rel_l2(y2, y_ref) <= BF16_TOL


def test_bad_expert_id_blocks_the_layer_and_reports():
    m = mok()
    inp = _inputs("tiny", seed=6)
    inp.top_experts[7, 1] = 99
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    y, ctx = m.forward(g.x, g.router_w, sched, w)
    assert ctx.status() == 2                                  # MOK_ERR_INDEX


def test_host_argument_errors():
    m = mok()
    inp = _inputs("tiny")
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    with pytest.raises(ValueError):
        m.forward(g.x.float(), g.router_w, sched, w)            # wrong dtype
    bad = m.Weights(g.w_gate[:, :, :96].contiguous(), g.w_up[:, :, :96].contiguous(),
                    g.w_down[:, :96].contiguous())
    with pytest.raises(ValueError):
        m.forward(g.x[:, :96].contiguous(), g.router_w, sched, bad)   # H outside the contract
    with pytest.raises(m.MokError) as ei:
        m.forward(g.x, g.router_w, sched, w, mode="mxfp8")     # no prequantised weights
    assert ei.value.code == 1
    # the MXFP8 backward needs the weights' transposed copies as well
    wq = m.quantize_weights(w)
    y, ctx = m.forward(g.x, g.router_w, sched, wq, mode="mxfp8_full")
    with pytest.raises(m.MokError) as ei:
        m.backward(g.dy, g.x, g.router_w, sched, ctx, wq)
    assert ei.value.code == 1
    with pytest.raises(ValueError):
        m.forward(g.x, g.router_w, sched, wq, mode="fp4")


@pytest.mark.parametrize("mode", ["bf16", "mxfp8", "mxfp8_full"])
def test_full_size_T4096_sampled(mode):
    """The T=4096 layers (H=2048, I=1024, E=64, k=8, I_s=2048; bf16, MXFP8 forward,
    MXFP8 forward and backward) at full
    size, in the launch configuration the benchmark times: y, dx and d_router_w
    on 48 sampled tokens, and the full weight gradients of the hottest and the
    coldest expert, against the oracle."""
    wl = {"bf16": "bf16_T4096", "mxfp8": "mxfp8_T4096", "mxfp8_full": "mxfp8full_T4096"}[mode]
    inp = gen.make_workload(wl, seed=0)
    y, grads, sched, ctx = run_layer(inp, mode, capacity=0.5, minibatch=2048)
    assert ctx.status() == 0
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(inp.meta["T"], 48, replace=False))
    sub = subset_inputs(inp, tok)
    y_ref, g_ref = oracle_fwd_bwd(sub, mode)
    assert rel_l2(y[tok], y_ref) <= BF16_TOL
    assert rel_l2(grads["dx"][tok], g_ref["dx"]) <= BF16_TOL
    assert rel_l2(grads["d_router_w"][tok], g_ref["d_router_w"]) <= BF16_TOL
    # full weight gradients of the hottest and the coldest expert: only the rows
    # routed to expert e reach dW[e], so a k = 1 layer over those rows gives it
    te = inp.top_experts.numpy()
    cnt = np.bincount(te.reshape(-1), minlength=inp.meta["E"])
    for e in (int(cnt.argmax()), int(cnt.argmin())):
        t_e, j_e = np.nonzero(te == e)
        idx = torch.as_tensor(t_e)
        sub_e = gen.LayerInputs(inp.x[idx], inp.router_w[idx, j_e].reshape(-1, 1).contiguous(),
                                torch.full((len(t_e), 1), e, dtype=torch.int64), inp.w_gate, inp.w_up,
                                inp.w_down, None, None, None, inp.dy[idx], dict(inp.meta))
        _, ge = oracle_fwd_bwd(sub_e, mode)
        for key in ("d_w_gate", "d_w_up", "d_w_down"):
            assert rel_l2(grads[key][e], ge[key][e]) <= BF16_TOL, (e, key)
    # shared expert gradients: a layer with no routed experts gives them alone
    if inp.ws_gate is not None:
        sub_s = gen.LayerInputs(inp.x, inp.router_w, inp.top_experts, inp.w_gate[:0], inp.w_up[:0],
                                inp.w_down[:0], inp.ws_gate, inp.ws_up, inp.ws_down, inp.dy, dict(inp.meta))
        _, gs = oracle_fwd_bwd(sub_s, mode)
        for key in ("d_ws_gate", "d_ws_up", "d_ws_down"):
            assert rel_l2(grads[key], gs[key]) <= BF16_TOL, key


def test_stage_events_time_each_stage():
    m = mok()
    from mixture_experts_layer_mok_gb300 import _lib

    inp = _inputs("ragged_shared", seed=7)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * _lib.MOK_NUM_STAGES)]
    y, ctx = m.forward(g.x, g.router_w, sched, w, events=ev)
    m.backward(g.dy, g.x, g.router_w, sched, ctx, w, events=ev)
    torch.cuda.synchronize()
    ms = [ev[2 * s].elapsed_time(ev[2 * s + 1]) for s in range(_lib.MOK_NUM_STAGES)]
    assert all(v >= 0 for v in ms)
    for name in ("fwd_gateup", "fwd_down", "bwd_down", "bwd_wgrad_gateup", "bwd_shared_dgrad"):
        assert ms[_lib.STAGE_NAMES.index(name)] > 0, name
    with pytest.raises(ValueError):
        m.forward(g.x, g.router_w, sched, w, events=ev[:3])


@pytest.mark.parametrize("name", ["skewed", "wide", "ragged_shared"])
@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_dispatch_paths_agree_bitwise(name, mode):
    """Permuted copies, the gather warps (cp.async) and TMA tile::gather4 move
    the same token rows into the same shared-memory layout, so every output of
    forward and backward must be bit-identical across the three."""
    m = mok()
    inp = _inputs(name, seed=8)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g, mode)
    outs = []
    for dispatch, flags in (("permute", 0), ("fused", 0), ("fused", 2)):
        y, ctx = m.forward(g.x, g.router_w, sched, w, mode=mode, debug=flags, dispatch=dispatch)
        grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, debug=flags, dispatch=dispatch)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        outs.append((y.clone(), {kk: v.clone() for kk, v in grads.items()}))
    for other in outs[1:]:
        assert torch.equal(outs[0][0], other[0])
        for key in outs[0][1]:
            assert torch.equal(outs[0][1][key], other[1][key]), key


@pytest.mark.parametrize("name,mode", [(n, "bf16") for n in SHAPES] + [(n, "mxfp8") for n in SHAPES])
def test_cta_pairs_match_single_ctas_bitwise(name, mode):
    """CTA pairs (M = 256 over two SMs, each holding half of B) and single CTAs
    run every output element's K loop in the same order, so forward and
    backward must be bit-identical between them (bf16 GEMMs: pairs by
    default, 4 = MOK_DEBUG_NO_CTA_PAIR; block-scaled forward GEMMs: single
    CTAs with 256-wide tiles, 8 = MOK_DEBUG_MX_CTA_PAIR (pairs, 256-wide
    tiles), 16 = MOK_DEBUG_MX_PAIR128 (pairs, 128-wide tiles, interleaved
    gate|up weight scales))."""
    m = mok()
    inp = _inputs(name, seed=9)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g, mode)
    outs = []
    for flags in ((0, 4) if mode == "bf16" else (0, 8, 16)):
        y, ctx = m.forward(g.x, g.router_w, sched, w, mode=mode, debug=flags)
        grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, debug=flags)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        outs.append((y.clone(), {kk: v.clone() for kk, v in grads.items()}))
    for other in outs[1:]:
        assert torch.equal(outs[0][0], other[0])
        for key in outs[0][1]:
            assert torch.equal(outs[0][1][key], other[1][key]), key


@pytest.mark.parametrize("name,mode", [("wide", "bf16"), ("skewed", "bf16"), ("wide", "mxfp8"),
                                       ("ragged_shared", "mxfp8_full")])
def test_item_order_changes_no_bit(name, mode):
    """Each GEMM output tile has one owner and a fixed K order, so the order in
    which the persistent CTAs visit the tiles changes no output bit: the
    default grouped order, 32 = MOK_DEBUG_PLAIN_ORDER, 64 =
    MOK_DEBUG_STATIC_ORDER, 128 = MOK_DEBUG_TICKET_ORDER (every CTA takes the
    next item in line through the work-item queue), and combinations."""
    m = mok()
    inp = _inputs(name, seed=13)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g, mode)
    outs = []
    for flags in (0, 32, 64, 128, 160):
        y, ctx = m.forward(g.x, g.router_w, sched, w, mode=mode, debug=flags)
        grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, debug=flags)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        outs.append((y.clone(), {kk: v.clone() for kk, v in grads.items()}))
    for other in outs[1:]:
        assert torch.equal(outs[0][0], other[0])
        for key in outs[0][1]:
            assert torch.equal(outs[0][1][key], other[1][key]), key


def test_fused_forward_permuted_backward_mix():
    """A backward may use another dispatch than its forward (it then makes its
    own copy of x's rows)."""
    m = mok()
    inp = _inputs("wide", seed=9)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    y, ctx = m.forward(g.x, g.router_w, sched, w, dispatch="fused")
    grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, dispatch="permute")
    torch.cuda.synchronize()
    y_ref, g_ref = oracle_fwd_bwd(inp, "bf16")
    errs, bad = compare_all(y, grads, y_ref, g_ref, BF16_TOL)
    assert not bad, errs


def _ctx_bytes(ctx, field, nbytes):
    """nbytes of the context buffer at the device pointer ctx.c.<field>."""
    off = getattr(ctx.c, field) - ctx.buf.data_ptr()
    assert 0 <= off and off + nbytes <= ctx.buf.numel()
    return ctx.buf[off:off + nbytes].cpu().numpy()


def _untile_scales(tiled, rows, K):
    """Row-major [rows][K/32] scales from the tensor-core scale layout (512-byte
    atoms per 128-row block and 128-column group; row r's four block scales of
    a group are one 32-bit word at byte (r % 32) * 16 + (r / 32) * 4)."""
    cg = K // 128
    out = np.empty((rows, K // 32), np.uint8)
    for row in range(rows):
        r = row % 128
        for b in range(K // 32):
            atom = (row // 128) * cg + b // 4
            out[row, b] = tiled[atom * 512 + (r % 32) * 16 + (r // 32) * 4 + b % 4]
    return out


@pytest.mark.parametrize("name", ["ragged_shared", "skewed", "deep_h"])
def test_mxfp8_dispatch_codes_and_scales_bit_exact(name):
    """The MXFP8 forward's quantise-and-dispatch step: x's E4M3 codes and E8M0
    scales in token order and in schedule order equal the oracle's quantiser,
    row for row; padding rows hold zero codes and unit scales.  The bf16 rows
    it copies into schedule order are x's rows, bit for bit."""
    m = mok()
    inp = _inputs(name, seed=3)
    T, H, k = inp.meta["T"], inp.meta["H"], inp.meta["k"]
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g, "mxfp8")
    _, ctx = m.forward(g.x, g.router_w, sched, w, mode="mxfp8")
    torch.cuda.synchronize()
    assert ctx.status() == 0
    codes, scales = oracle.mxfp8_quantize(inp.x.float().numpy())
    t_pad = (T + 127) // 128 * 128
    xq = _ctx_bytes(ctx, "xq", T * H).reshape(T, H)
    assert np.array_equal(xq, codes)
    xs = _untile_scales(_ctx_bytes(ctx, "xq_sc", t_pad * H // 32), t_pad, H)
    assert np.array_equal(xs[:T], scales)
    assert np.all(xs[T:] == 127)
    st, _, P = sched.status()
    assert st == 0
    row_src = sched.arrays()["row_src"][:P].cpu().numpy()
    xp = _ctx_bytes(ctx, "xq_perm", P * H).reshape(P, H)
    xps = _untile_scales(_ctx_bytes(ctx, "xq_perm_sc", (P + 127) // 128 * 128 * H // 32), P, H)
    tok = np.where(row_src >= 0, row_src // k, 0)
    valid = row_src >= 0
    assert np.array_equal(xp[valid], codes[tok[valid]])
    assert np.array_equal(xps[valid], scales[tok[valid]])
    assert np.all(xp[~valid] == 0) and np.all(xps[~valid] == 127)
    # the same pass writes x's bf16 rows in schedule order for the bf16 backward
    xb = _ctx_bytes(ctx, "x_perm", P * H * 2).view(np.uint16).reshape(P, H)
    x16 = inp.x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(xb[valid], x16[tok[valid]])
    assert np.all(xb[~valid] == 0)


@pytest.mark.parametrize("name,mode", [("ragged_shared", "bf16"), ("wide", "bf16"), ("skewed", "bf16"),
                                       ("ragged_shared", "mxfp8"), ("wide", "mxfp8"),
                                       ("ragged_shared", "mxfp8_full"), ("wide", "mxfp8_full")])
def test_swiglu_limit_matches_oracle(name, mode):
    """The clamped SwiGLU (swiglu_limit L: gate <= L, up in [-L, L]) against the
    oracle's clamped layer, forward and backward.  L lies in the 50-80%
    quantile range of the pre-activations (so a large share is clamped), on a
    bf16 midpoint as far as possible from every pre-activation: there the
    kernels' pass/stop decisions on bf16-rounded fp32 values and the oracle's
    on float64 values agree."""
    inp = _inputs(name, seed=12)
    L, gap = clamp_limit(inp, mode)
    assert gap > 0.0
    y, grads, sched, ctx = run_layer(inp, mode, swiglu_limit=L)
    assert ctx.status() == 0
    y_ref, g_ref = oracle_fwd_bwd(inp, mode, swiglu_limit=L)
    errs, bad = compare_all(y, grads, y_ref, g_ref, BF16_TOL)
    assert not bad, errs
    # the clamp changed the result: the plain layer is far from it
    y_plain, _ = oracle_fwd_bwd(inp, mode)
    assert rel_l2(y_ref, y_plain) > 10 * BF16_TOL


def test_swiglu_limit_rejects_bad_values():
    m = mok()
    inp = _inputs("tiny", seed=1)
    g = inp.to("cuda")
    sched = m.schedule(g.top_experts, inp.meta["E"], 0.5)
    w = weights_of(g)
    for bad in (-1.0, float("nan"), float("inf")):
        with pytest.raises(m.MokError):
            m.forward(g.x, g.router_w, sched, w, swiglu_limit=bad)

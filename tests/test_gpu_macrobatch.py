"""The macrobatch ring ("Mixture-of-Kittens: a deterministic MoE megakernel for
NVL72 racks", "Tuning the five hyperparameters before production":
macrobatch_size is the size of the token ring buffer).

With a ring smaller than the schedule, the routed experts run window by
window over ring-sized scratch, each window a run of whole experts.  No
contraction is split and every row is computed by the same tile with the same
K order, so every output bit must equal the single pass: y, dx, the router
weight gradient and all six weight gradients, in the three precisions, with
either dispatch form, with a forward ring and a backward ring of their own.
A ring smaller than one expert's padded rows is refused before any layer work.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import BF16_TOL, compare_all, mok, oracle_fwd_bwd, weights_of

pytestmark = pytest.mark.gpu

KEYS = ("dx", "d_router_w", "d_w_gate", "d_w_up", "d_w_down", "d_ws_gate", "d_ws_up", "d_ws_down")


def _run(g, E, w, mode, fwd_mb=0, bwd_mb=0, dispatch="auto", capacity=0.5, debug=0):
    m = mok()
    sched = m.schedule(g.top_experts, E, capacity)
    y, ctx = m.forward(g.x, g.router_w, sched, w, mode=mode, dispatch=dispatch, macrobatch=fwd_mb, debug=debug)
    grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, dispatch=dispatch, macrobatch=bwd_mb, debug=debug)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    return y, grads, sched, ctx


def _assert_same(a, b):
    assert torch.equal(a[0], b[0]), "y"
    for key in KEYS:
        if key in a[1]:
            assert torch.equal(a[1][key], b[1][key]), key


def _windows(sched, mb):
    cnt = sched.arrays()["cnt"].cpu().tolist()
    return mok().macrobatch_plan(cnt, mb)


def _largest_padded(sched):
    cnt = sched.arrays()["cnt"].cpu().numpy()
    return int(((cnt + 127) // 128 * 128).max())


@pytest.mark.parametrize("mb", [1024, 4096])
def test_bf16_T4096_ring_matches_single_pass_bitwise(mb):
    """The bf16 layer T=4096, H=2048, I=1024, E=64, k=8, I_s=2048 with rings of
    1024 and 4096 rows (forward and backward) against the single pass."""
    m = mok()
    inp = gen.make_workload("bf16_T4096", seed=0)
    g = inp.to("cuda")
    E = inp.meta["E"]
    w = weights_of(g, "bf16")
    ref = _run(g, E, w, "bf16")
    got = _run(g, E, w, "bf16", fwd_mb=mb, bwd_mb=mb)
    _assert_same(got, ref)
    wins = _windows(ref[2], mb)
    assert len(wins) >= 32768 // mb            # the ring really ran in windows
    assert got[3].c.ring_rows == mb and ref[3].c.ring_rows == 0
    dims = (inp.meta["T"], inp.meta["k"], E, inp.meta["H"], inp.meta["I"], inp.meta["I_s"], 0)
    lib = m._lib.load()
    assert lib.mok_ctx_bytes_ring(*dims, mb) < lib.mok_ctx_bytes(*dims)
    assert lib.mok_bwd_workspace_bytes_ring(*dims, mb) < lib.mok_bwd_workspace_bytes(*dims)


@pytest.mark.parametrize("fwd_mb,bwd_mb", [(4096, 4096), (4096, 0), (0, 4096)])
def test_mxfp8_T4096_ring_matches_single_pass_bitwise(fwd_mb, bwd_mb):
    """MXFP8 forward / bf16 backward at the T=4096 shapes: a ring in the
    forward, in the backward, or both (a one-pass backward after a forward with
    a ring gathers x's rows itself; a ring backward after a one-pass forward
    reads the forward's copy of them window by window)."""
    inp = gen.make_workload("mxfp8_T4096", seed=1)
    g = inp.to("cuda")
    w = weights_of(g, "mxfp8")
    ref = _run(g, inp.meta["E"], w, "mxfp8")
    got = _run(g, inp.meta["E"], w, "mxfp8", fwd_mb=fwd_mb, bwd_mb=bwd_mb)
    _assert_same(got, ref)
    if fwd_mb:
        assert got[3].c.x_perm is None           # no full-size copy of x's rows in the context


def test_mxfp8_full_T4096_ring_matches_single_pass_bitwise():
    """MXFP8 forward and backward at the T=4096 shapes with a 4096-row ring: the
    backward's 32-row quantisation blocks of the weight gradients stay whole."""
    inp = gen.make_workload("mxfp8full_T4096", seed=2)
    g = inp.to("cuda")
    w = weights_of(g, "mxfp8_full")
    ref = _run(g, inp.meta["E"], w, "mxfp8_full")
    got = _run(g, inp.meta["E"], w, "mxfp8_full", fwd_mb=4096, bwd_mb=4096)
    _assert_same(got, ref)


# (T, H, I, E, k, I_s, skew): skewed routing with hot and empty experts, and a
# layer with a shared expert whose I is not a multiple of 256
SMALL = {
    "skewed": (333, 128, 128, 16, 4, 0, 1.2),
    "wide": (520, 512, 256, 12, 6, 384, 1.2),
    "ragged_shared": (200, 256, 384, 5, 3, 256, None),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", ["bf16", "mxfp8", "mxfp8_full"])
def test_tightest_ring_and_overflow_list_match_single_pass(name, mode):
    """The smallest ring that holds the hottest expert (so that expert runs
    alone), with a capacity multiplier that sends most tiles to the overflow
    list: the windows keep the schedule's tile order, and every bit matches."""
    T, H, I, E, k, I_s, skew = SMALL[name]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=5)
    g = inp.to("cuda")
    w = weights_of(g, mode)
    ref = _run(g, E, w, mode, capacity=0.05)
    mb = _largest_padded(ref[2])
    got = _run(g, E, w, mode, fwd_mb=mb, bwd_mb=mb, capacity=0.05)
    _assert_same(got, ref)
    assert len(_windows(ref[2], mb)) > 1


@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_fused_dispatch_with_a_ring_matches_the_permuted_single_pass(mode):
    """Gathered token rows (no schedule-order copy of x or dy) with a ring."""
    T, H, I, E, k, I_s, skew = SMALL["wide"]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=6)
    g = inp.to("cuda")
    w = weights_of(g, mode)
    ref = _run(g, E, w, mode)
    mb = _largest_padded(ref[2])
    got = _run(g, E, w, mode, fwd_mb=mb, bwd_mb=mb, dispatch="fused")
    _assert_same(got, ref)


def test_single_cta_ring_matches_single_pass():
    """The ring with CTA pairs off (the pair lists of the windows unused)."""
    T, H, I, E, k, I_s, skew = SMALL["wide"]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=8)
    g = inp.to("cuda")
    w = weights_of(g, "bf16")
    ref = _run(g, E, w, "bf16")
    mb = _largest_padded(ref[2])
    got = _run(g, E, w, "bf16", fwd_mb=mb, bwd_mb=mb, debug=4)   # MOK_DEBUG_NO_CTA_PAIR
    _assert_same(got, ref)


def test_tiny_layer_one_tile_ring_against_oracle():
    """T=128, H=128, I=256, E=8, k=2 with a 1-row macrobatch (a ring of one
    128-row tile: one expert per window): against the oracle, and bitwise
    against the single pass."""
    inp = gen.make_layer_inputs(128, 128, 256, 8, 2, 0, seed=3)
    g = inp.to("cuda")
    w = weights_of(g, "bf16")
    ref = _run(g, 8, w, "bf16")
    got = _run(g, 8, w, "bf16", fwd_mb=1, bwd_mb=1)
    _assert_same(got, ref)
    assert len(_windows(ref[2], 1)) == int((ref[2].arrays()["cnt"] > 0).sum().item())
    y_ref, g_ref = oracle_fwd_bwd(inp, "bf16")
    _, bad = compare_all(got[0], got[1], y_ref, g_ref, BF16_TOL)
    assert not bad, bad


def test_ring_smaller_than_an_expert_is_refused_before_any_work():
    """MOK_ERR_CAPACITY from the forward and from the backward, with their
    outputs untouched."""
    m = mok()
    T, H, I, E, k, I_s, skew = SMALL["skewed"]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=4)
    g = inp.to("cuda")
    w = weights_of(g, "bf16")
    sched = m.schedule(g.top_experts, E, 0.5)
    mb = _largest_padded(sched) - 128
    assert mb > 0
    y = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MokError) as ei:
        m.forward(g.x, g.router_w, sched, w, macrobatch=mb, out=y)
    assert ei.value.code == 3
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    y, ctx = m.forward(g.x, g.router_w, sched, w)
    dx = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    grads = {"dx": dx, "d_router_w": torch.zeros((T, k), dtype=torch.float32, device="cuda"),
             "d_w_gate": torch.empty_like(g.w_gate), "d_w_up": torch.empty_like(g.w_up),
             "d_w_down": torch.empty_like(g.w_down)}
    with pytest.raises(m.MokError) as ei:
        m.backward(g.dy, g.x, g.router_w, sched, ctx, w, grads=grads, macrobatch=mb)
    assert ei.value.code == 3
    torch.cuda.synchronize()
    assert bool((dx == 7.0).all())
    with pytest.raises(ValueError):
        m.forward(g.x, g.router_w, sched, w, macrobatch=-1)


def test_ring_under_autograd_matches_single_pass():
    """MoKLayer with a ring: the same gradients as without."""
    from mixture_experts_layer_mok_gb300.autograd import MoKLayer

    T, H, I, E, k, I_s, skew = SMALL["wide"]
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=9)
    g = inp.to("cuda")
    mb_ring = _largest_padded(mok().schedule(g.top_experts, E, 0.5))
    out = []
    for mb in (0, mb_ring):
        layer = MoKLayer(E, H, I, I_s, macrobatch=mb, device="cuda")
        with torch.no_grad():
            for name in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
                getattr(layer, name).copy_(getattr(g, name))
        x = g.x.clone().requires_grad_(True)
        y = layer(x, g.router_w, g.top_experts)
        y.backward(g.dy)
        out.append((y.detach(), x.grad, layer.w_gate.grad, layer.ws_down.grad))
    for a, b in zip(*out):
        assert torch.equal(a, b)
    assert np.isfinite(out[0][1].float().cpu().numpy()).all()


@pytest.mark.parametrize("mode", ["bf16", "mxfp8_full"])
def test_ring_edge_layers_match_single_pass(mode):
    """A one-expert layer (its only expert fills the one window), and a layer
    where most experts are empty (the windows fold them in): bitwise equal to
    the single pass, the latter with a ring of one tile."""
    for (T, H, I, E, k, I_s, skew), mb in (((300, 384, 128, 1, 1, 128, None), None),
                                           ((96, 128, 128, 64, 1, 128, 2.0), 1)):
        inp = gen.make_layer_inputs(T, H, I, E, k, I_s, skew=skew, seed=12)
        g = inp.to("cuda")
        w = weights_of(g, mode)
        ref = _run(g, E, w, mode)
        ring = mb or _largest_padded(ref[2])
        if mb:
            cnt = ref[2].arrays()["cnt"].cpu().numpy()
            if ((cnt + 127) // 128 * 128).max() > 128:
                ring = _largest_padded(ref[2])
            assert (cnt == 0).sum() > E // 2          # the routing leaves most experts empty
        got = _run(g, E, w, mode, fwd_mb=ring, bwd_mb=ring)
        _assert_same(got, ref)

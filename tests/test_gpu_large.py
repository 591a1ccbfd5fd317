"""Full-size parity of the skewed (T=16384) and large (T=65536) layers.

Each runs at full size, in the launch configuration the benchmark uses, with
seeded inputs drawn on the GPU.  The oracle is evaluated on outputs it can
compute piece by piece:
- whole tokens (the layer is per token, so a token needs only its own k
  experts' weights);
- 128-column slices of the intermediate dimension for the weight gradients
  of chosen experts (a slice of h determines the same slice of every weight
  gradient, and an expert's gradient needs only the rows routed to it);
- slices of the shared expert's weight gradients, summed over blocks of
  tokens (those gradients are sums over tokens; blocks start at multiples of
  32 tokens, so the MXFP8 backward's 32-token quantisation blocks stay whole).
The oracle pieces run on a pool of host threads: NumPy releases the
interpreter lock inside its array operations.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import BF16_TOL, expert_slice_inputs, oracle_fwd_bwd, rel_l2, run_layer, token_inputs

pytestmark = pytest.mark.gpu


def _need_bytes(nbytes):
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.skip(f"needs {nbytes / 2**30:.0f} GiB of free device memory, {free / 2**30:.0f} GiB free")


def _threads(gib_per_task):
    """Host threads for the oracle pieces: at most the cores, and as many as
    the available host memory holds at gib_per_task each."""
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE") / 2**30
    except (ValueError, OSError):
        avail = 16.0
    return max(1, min(os.cpu_count() or 1, 16, int(avail * 0.6 / gib_per_task)))


def _check_tokens(inp, y, grads, mode, tokens, gib_per_task):
    def one(t):
        yt, gt = oracle_fwd_bwd(token_inputs(inp, int(t)), mode)
        return yt[0], gt["dx"][0], gt["d_router_w"][0]

    with ThreadPoolExecutor(_threads(gib_per_task)) as ex:
        ref = list(ex.map(one, tokens))
    idx = torch.as_tensor(np.asarray(tokens), device=y.device)
    assert rel_l2(y[idx], np.stack([r[0] for r in ref])) <= BF16_TOL
    assert rel_l2(grads["dx"][idx], np.stack([r[1] for r in ref])) <= BF16_TOL
    assert rel_l2(grads["d_router_w"][idx], np.stack([r[2] for r in ref])) <= BF16_TOL


def _check_expert_slice(inp, grads, mode, e, i0, i1):
    sub, _ = expert_slice_inputs(inp, e, i0, i1)
    _, ge = oracle_fwd_bwd(sub, mode)
    assert rel_l2(grads["d_w_gate"][e, i0:i1], ge["d_w_gate"][0]) <= BF16_TOL, (e, "gate")
    assert rel_l2(grads["d_w_up"][e, i0:i1], ge["d_w_up"][0]) <= BF16_TOL, (e, "up")
    assert rel_l2(grads["d_w_down"][e, :, i0:i1], ge["d_w_down"][0]) <= BF16_TOL, (e, "down")


def _check_shared_slice(inp, grads, mode, i0, i1, block=4096):
    """Columns [i0, i1) of the shared expert's weight gradients: the oracle's
    shared-expert-only layer over blocks of tokens, summed."""
    T = inp.x.shape[0]
    sg, su = inp.ws_gate[i0:i1].cpu(), inp.ws_up[i0:i1].cpu()
    sd = inp.ws_down[:, i0:i1].contiguous().cpu()
    e0, d0 = inp.w_gate[:0].cpu(), inp.w_down[:0].cpu()

    def part(a):
        b = min(T, a + block)
        sub = gen.LayerInputs(inp.x[a:b].cpu(), inp.router_w[a:b].cpu(), inp.top_experts[a:b].cpu(), e0, e0, d0,
                              sg, su, sd, inp.dy[a:b].cpu(), dict(inp.meta))
        g = oracle_fwd_bwd(sub, mode)[1]
        return g["d_ws_gate"], g["d_ws_up"], g["d_ws_down"]

    with ThreadPoolExecutor(_threads(4.0)) as ex:
        parts = list(ex.map(part, range(0, T, block)))
    ref = [sum(p[i] for p in parts) for i in range(3)]
    assert rel_l2(grads["d_ws_gate"][i0:i1], ref[0]) <= BF16_TOL
    assert rel_l2(grads["d_ws_up"][i0:i1], ref[1]) <= BF16_TOL
    assert rel_l2(grads["d_ws_down"][:, i0:i1], ref[2]) <= BF16_TOL


@pytest.mark.parametrize("capacity", [0.5, 1.0])
def test_skewed_T16384_full_size(capacity):
    """Zipf-skewed routing: T=16384, H=4096, I=1536, E=128, k=8, minibatch 4096."""
    _need_bytes(40 << 30)
    inp = gen.make_workload("skewed_T16384", seed=0, device="cuda")
    y, grads, sched, ctx = run_layer(inp, "bf16", capacity=capacity, minibatch=4096)
    assert ctx.status() == 0
    st, num_tiles, P = sched.status()
    assert st == 0
    rng = np.random.default_rng(1)
    _check_tokens(inp, y, grads, "bf16", np.sort(rng.choice(inp.meta["T"], 24, replace=False)), 1.0)
    cnt = torch.bincount(inp.top_experts.reshape(-1), minlength=inp.meta["E"]).cpu().numpy()
    hot, cold = int(cnt.argmax()), int(np.argmin(np.where(cnt > 0, cnt, 1 << 30)))
    assert cnt[hot] > 8 * cnt.mean()          # the skew is real: one expert holds many tiles
    _check_expert_slice(inp, grads, "bf16", hot, 1408, 1536)
    _check_expert_slice(inp, grads, "bf16", cold, 0, 128)
    for e in np.nonzero(cnt == 0)[0][:2]:     # experts nobody chose have zero gradients
        assert grads["d_w_down"][int(e)].abs().max().item() == 0.0


def test_skewed_T16384_ring_matches_single_pass_bitwise():
    """The skewed layer with a ring of 16384 rows (the hot experts alone in
    their windows, the cold ones many to a window): bitwise equal to the single
    pass."""
    from tests.gpu_util import mok, weights_of

    _need_bytes(40 << 30)
    m = mok()
    inp = gen.make_workload("skewed_T16384", seed=0, device="cuda")
    w = weights_of(inp, "bf16")
    E = inp.meta["E"]
    sched = m.schedule(inp.top_experts, E, 0.5)
    cnt = sched.arrays()["cnt"].cpu().numpy()
    ring = max(16384, int(((cnt + 127) // 128 * 128).max()))
    out = []
    for mb in (0, ring):
        y, ctx = m.forward(inp.x, inp.router_w, sched, w, minibatch=4096, macrobatch=mb)
        grads = m.backward(inp.dy, inp.x, inp.router_w, sched, ctx, w, minibatch=4096, macrobatch=mb)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        out.append((y, grads))
        del ctx
    assert torch.equal(out[0][0], out[1][0])
    for key in out[0][1]:
        assert torch.equal(out[0][1][key], out[1][1][key]), key
    assert len(m.macrobatch_plan(cnt.tolist(), ring)) > 2


def _large(mode, ntok, seed):
    """T=65536, H=7168, I=2048, E=256, k=8, one shared expert (I_s=2048)."""
    _need_bytes(150 << 30)
    inp = gen.make_workload("large_T65536", seed=0, device="cuda")
    y, grads, sched, ctx = run_layer(inp, mode, capacity=0.5, minibatch=4096)
    assert ctx.status() == 0
    rng = np.random.default_rng(seed)
    _check_tokens(inp, y, grads, mode, np.sort(rng.choice(inp.meta["T"], ntok, replace=False)), 7.0)
    cnt = torch.bincount(inp.top_experts.reshape(-1), minlength=inp.meta["E"]).cpu().numpy()
    _check_expert_slice(inp, grads, mode, int(cnt.argmax()), 0, 128)        # the hottest expert
    _check_expert_slice(inp, grads, mode, int(cnt.argmin()), 1920, 2048)    # the coldest
    _check_shared_slice(inp, grads, mode, 0, 64)


def test_large_T65536_full_size_mxfp8():
    """The large layer with MXFP8 forward / BF16 backward: 24 tokens, slices of
    the hottest and coldest experts' and the shared expert's weight gradients."""
    _large("mxfp8", 24, 2)


def test_large_T65536_full_size_mxfp8_full():
    """The large layer with MXFP8 forward and backward: 12 tokens, slices of the
    hottest and coldest experts' and the shared expert's weight gradients."""
    _large("mxfp8_full", 12, 3)


def test_large_T65536_ring_matches_single_pass_bitwise():
    """The large layer (MXFP8 forward / BF16 backward, the benchmark's default)
    with a 131072-row macrobatch ring in the forward and the backward: every
    bit of y, dx, the router-weight gradient and the six weight gradients
    equals the single pass (whose parity the tests above check), while the
    ring bounds the schedule-order scratch."""
    from tests.gpu_util import mok, weights_of

    _need_bytes(150 << 30)
    m = mok()
    inp = gen.make_workload("large_T65536", seed=0, device="cuda")
    w = weights_of(inp, "mxfp8")
    E, mb = inp.meta["E"], 131072
    sched = m.schedule(inp.top_experts, E, 0.5)
    out = []
    for ring in (0, mb):
        y, ctx = m.forward(inp.x, inp.router_w, sched, w, mode="mxfp8", minibatch=4096, macrobatch=ring)
        grads = m.backward(inp.dy, inp.x, inp.router_w, sched, ctx, w, minibatch=4096, macrobatch=ring)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        out.append((y, grads))
        del ctx
        torch.cuda.empty_cache()
    for key in out[0][1]:
        assert torch.equal(out[0][1][key], out[1][1][key]), key
    assert torch.equal(out[0][0], out[1][0])
    assert len(m.macrobatch_plan(sched.arrays()["cnt"].cpu().tolist(), mb)) >= 4
    dims = (inp.meta["T"], inp.meta["k"], E, inp.meta["H"], inp.meta["I"], inp.meta["I_s"], 1)
    lib = m._lib.load()
    full = lib.mok_ctx_bytes(*dims) + lib.mok_bwd_workspace_bytes(*dims)
    ringed = lib.mok_ctx_bytes_ring(*dims, mb) + lib.mok_bwd_workspace_bytes_ring(*dims, mb)
    assert ringed < 0.6 * full

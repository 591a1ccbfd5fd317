"""Full-size parity of the skewed (T=16384) and large (T=65536) layers.

Both run at full size, in the launch configuration the benchmark uses, with
seeded inputs drawn on the GPU. The oracle is evaluated on outputs it can
compute one by one:
- whole tokens (the layer is per-token, so a token needs only its own k
  experts' weights);
- 128-column slices of the intermediate dimension for the weight gradients of
  chosen experts and of the shared expert (a slice of h determines the same
  slice of every weight gradient).
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import (BF16_TOL, expert_slice_inputs, oracle_fwd_bwd, rel_l2, run_layer, shared_slice_inputs,
                            token_inputs)

pytestmark = pytest.mark.gpu


def _need_bytes(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.skip(f"needs {nbytes / 2**30:.0f} GiB of free device memory, {free / 2**30:.0f} GiB free")


def _check_tokens(inp, y, grads, mode, tokens):
    ys, yr, dxs, dxr, dws, dwr = [], [], [], [], [], []
    for t in tokens:
        yt, gt = oracle_fwd_bwd(token_inputs(inp, int(t)), mode)
        ys.append(y[t].float().cpu().numpy()); yr.append(yt[0])
        dxs.append(grads["dx"][t].float().cpu().numpy()); dxr.append(gt["dx"][0])
        dws.append(grads["d_router_w"][t].cpu().numpy()); dwr.append(gt["d_router_w"][0])
    assert rel_l2(np.stack(ys), np.stack(yr)) <= BF16_TOL
    assert rel_l2(np.stack(dxs), np.stack(dxr)) <= BF16_TOL
    assert rel_l2(np.stack(dws), np.stack(dwr)) <= BF16_TOL


def _check_expert_slice(inp, grads, mode, e, i0, i1):
    sub, _ = expert_slice_inputs(inp, e, i0, i1)
    _, ge = oracle_fwd_bwd(sub, mode)
    assert rel_l2(grads["d_w_gate"][e, i0:i1], ge["d_w_gate"][0]) <= BF16_TOL, (e, "gate")
    assert rel_l2(grads["d_w_up"][e, i0:i1], ge["d_w_up"][0]) <= BF16_TOL, (e, "up")
    assert rel_l2(grads["d_w_down"][e, :, i0:i1], ge["d_w_down"][0]) <= BF16_TOL, (e, "down")


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
    _check_tokens(inp, y, grads, "bf16", np.sort(rng.choice(inp.meta["T"], 24, replace=False)))
    cnt = torch.bincount(inp.top_experts.reshape(-1), minlength=inp.meta["E"]).cpu().numpy()
    hot, cold = int(cnt.argmax()), int(np.argmin(np.where(cnt > 0, cnt, 1 << 30)))
    assert cnt[hot] > 8 * cnt.mean()          # the skew is real: one expert holds many tiles
    _check_expert_slice(inp, grads, "bf16", hot, 1408, 1536)
    _check_expert_slice(inp, grads, "bf16", cold, 0, 128)
    for e in np.nonzero(cnt == 0)[0][:2]:     # experts nobody chose have zero gradients
        assert grads["d_w_down"][int(e)].abs().max().item() == 0.0


def test_large_T65536_full_size_mxfp8():
    """T=65536, H=7168, I=2048, E=256, k=8, one shared expert (I_s=2048), MXFP8
    forward / BF16 backward."""
    _need_bytes(170 << 30)
    inp = gen.make_workload("large_T65536", seed=0, device="cuda")
    y, grads, sched, ctx = run_layer(inp, "mxfp8", capacity=0.5, minibatch=4096)
    assert ctx.status() == 0
    rng = np.random.default_rng(2)
    _check_tokens(inp, y, grads, "mxfp8", np.sort(rng.choice(inp.meta["T"], 6, replace=False)))
    cnt = torch.bincount(inp.top_experts.reshape(-1), minlength=inp.meta["E"]).cpu().numpy()
    _check_expert_slice(inp, grads, "mxfp8", int(cnt.argmin()), 1920, 2048)
    gs = oracle_fwd_bwd(shared_slice_inputs(inp, 0, 64), "mxfp8")[1]
    assert rel_l2(grads["d_ws_gate"][0:64], gs["d_ws_gate"]) <= BF16_TOL
    assert rel_l2(grads["d_ws_up"][0:64], gs["d_ws_up"]) <= BF16_TOL
    assert rel_l2(grads["d_ws_down"][:, 0:64], gs["d_ws_down"]) <= BF16_TOL

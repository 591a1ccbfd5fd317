"""The torch.autograd face of the layer (MoKFunction / MoKLayer): gradients
that autograd delivers for a loss <y, dy> equal the oracle's gradients of the
same layer, in every mode."""
import pytest
import torch

from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import BF16_TOL, mok, oracle_fwd_bwd, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["bf16", "mxfp8", "mxfp8_full"])
@pytest.mark.parametrize("shape", [(200, 256, 384, 5, 3, 256), (333, 128, 128, 16, 4, 0)])
def test_autograd_gradients_match_oracle(mode, shape):
    mok()   # builds / loads the library
    from mixture_experts_layer_mok_gb300.autograd import MoKLayer

    T, H, I, E, k, I_s = shape
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, seed=11)
    layer = MoKLayer(E, H, I, I_s, mode=mode, device="cuda")
    with torch.no_grad():
        layer.w_gate.copy_(inp.w_gate); layer.w_up.copy_(inp.w_up); layer.w_down.copy_(inp.w_down)
        if I_s:
            layer.ws_gate.copy_(inp.ws_gate); layer.ws_up.copy_(inp.ws_up); layer.ws_down.copy_(inp.ws_down)
    x = inp.x.cuda().requires_grad_(True)
    rw = inp.router_w.cuda().requires_grad_(True)
    y = layer(x, rw, inp.top_experts.cuda())
    (y.float() * inp.dy.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    y_ref, g_ref = oracle_fwd_bwd(inp, mode)
    assert rel_l2(y, y_ref) <= BF16_TOL
    got = {"dx": x.grad, "d_router_w": rw.grad, "d_w_gate": layer.w_gate.grad, "d_w_up": layer.w_up.grad,
           "d_w_down": layer.w_down.grad}
    if I_s:
        got.update(d_ws_gate=layer.ws_gate.grad, d_ws_up=layer.ws_up.grad, d_ws_down=layer.ws_down.grad)
    for key, val in got.items():
        assert val is not None, key
        assert rel_l2(val, g_ref[key]) <= BF16_TOL, key


@pytest.mark.parametrize("mode", ["bf16", "mxfp8_full"])
def test_saved_schedule_and_context_survive_offload(mode):
    """The schedule and the forward context reach backward through
    save_for_backward, so saved-tensor hooks see them: under save_on_cpu they
    leave the device after the forward and come back at new addresses for the
    backward.  The gradients equal those of a run without offload, bit for bit."""
    mok()
    from mixture_experts_layer_mok_gb300.autograd import MoKLayer

    T, H, I, E, k, I_s = 200, 256, 384, 5, 3, 256
    inp = gen.make_layer_inputs(T, H, I, E, k, I_s, seed=13)

    def run(offload):
        layer = MoKLayer(E, H, I, I_s, mode=mode, device="cuda")
        with torch.no_grad():
            for name in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
                getattr(layer, name).copy_(getattr(inp, name))
        x = inp.x.cuda().requires_grad_(True)
        rw = inp.router_w.cuda().requires_grad_(True)
        if offload:
            with torch.autograd.graph.save_on_cpu(pin_memory=True):
                y = layer(x, rw, inp.top_experts.cuda())
        else:
            y = layer(x, rw, inp.top_experts.cuda())
        (y.float() * inp.dy.cuda().float()).sum().backward()
        torch.cuda.synchronize()
        return [y, x.grad, rw.grad] + [getattr(layer, n).grad for n in ("w_gate", "w_up", "w_down", "ws_gate",
                                                                        "ws_up", "ws_down")]

    for a, b in zip(run(False), run(True)):
        assert torch.equal(a, b)

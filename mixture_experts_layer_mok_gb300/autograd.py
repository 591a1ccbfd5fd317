"""torch.autograd face of the layer: ``MoKFunction`` and the ``MoKLayer`` module.

The pages' PyTorch-facing pieces are a runtime whose forward returns the
output plus an opaque context and whose backward consumes it, returning
"gradients matching every forward input" ("nemo_automodel.components.moe.
mok_experts": ``_MoKRuntime.forward`` / ``backward``, ``GroupedExpertsMoK``).
This module puts those two calls under torch.autograd, so that a model can
call the layer like any other module.  It only marshals arguments: the
schedule, forward and backward run in libmok's kernels through the binding.
"""
from __future__ import annotations

import torch

from . import Context, Schedule, Weights, backward, forward, quantize_weights, schedule


class MoKFunction(torch.autograd.Function):
    """y = MoK layer(x, router_w, top_experts; routed and optional shared
    SwiGLU weights).  Differentiable in x, router_w and every weight; the
    expert ids are integers and get no gradient."""

    @staticmethod
    def forward(ctx, x, router_w, top_experts, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, mode, capacity,
                minibatch, swiglu_limit=0.0, macrobatch=0):
        E = w_gate.shape[0]
        sched = schedule(top_experts, E, capacity)
        weights = Weights(w_gate, w_up, w_down, ws_gate, ws_up, ws_down)
        if mode in ("mxfp8", "mxfp8_full"):
            weights = quantize_weights(weights, backward=(mode == "mxfp8_full"))
        y, mctx = forward(x, router_w, sched, weights, mode=mode, minibatch=minibatch, swiglu_limit=swiglu_limit,
                          macrobatch=macrobatch)
        # the schedule and the context go through save_for_backward as their
        # buffers, so saved-tensor hooks (offload, checkpointing) see them
        sbuf, smeta = sched.flatten()
        cbuf, cmeta = mctx.flatten()
        ctx.save_for_backward(x, router_w, sbuf, cbuf)
        ctx.mok = (smeta, cmeta, weights, minibatch, macrobatch, ws_gate is not None)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, router_w, sbuf, cbuf = ctx.saved_tensors
        smeta, cmeta, weights, minibatch, macrobatch, shared = ctx.mok
        sched = Schedule.unflatten(sbuf, smeta)     # over wherever the hooks put the buffers
        mctx = Context.unflatten(cbuf, cmeta)
        g = backward(dy.to(torch.bfloat16).contiguous(), x, router_w, sched, mctx, weights, minibatch=minibatch,
                     macrobatch=macrobatch)
        ctx.mok = None
        return (g["dx"], g["d_router_w"], None, g["d_w_gate"], g["d_w_up"], g["d_w_down"],
                g["d_ws_gate"] if shared else None, g["d_ws_up"] if shared else None,
                g["d_ws_down"] if shared else None, None, None, None, None, None)


def mok_layer(x, router_w, top_experts, w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None,
              mode: str = "bf16", capacity: float = 0.5, minibatch: int = 0, swiglu_limit: float = 0.0,
              macrobatch: int = 0):
    """Functional form: x bf16 [T, H], router_w fp32 [T, k], top_experts int64
    [T, k]; routed weights [E, I, H], [E, I, H], [E, H, I]; shared weights
    [I_s, H], [I_s, H], [H, I_s] or None.  ``macrobatch``: rows of the token
    ring, forward and backward (0: one pass)."""
    return MoKFunction.apply(x, router_w, top_experts, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, mode, capacity,
                             minibatch, swiglu_limit, macrobatch)


class MoKLayer(torch.nn.Module):
    """Routed experts (E of them, intermediate size I) plus an optional shared
    expert (intermediate size I_s), in the weight layouts of the pages'
    ``GroupedExpertsMoK``.  The router stays outside (the caller passes the
    chosen experts and their weights), as on the pages."""

    def __init__(self, E: int, H: int, I: int, I_s: int = 0, mode: str = "bf16", capacity: float = 0.5,
                 minibatch: int = 0, swiglu_limit: float = 0.0, macrobatch: int = 0, device=None,
                 init_std: float = 0.02, generator=None):
        super().__init__()
        kw = dict(dtype=torch.bfloat16, device=device)

        def param(*shape):
            t = torch.empty(*shape, **kw)
            t.normal_(0.0, init_std, generator=generator)
            return torch.nn.Parameter(t)

        self.w_gate, self.w_up, self.w_down = param(E, I, H), param(E, I, H), param(E, H, I)
        if I_s:
            self.ws_gate, self.ws_up, self.ws_down = param(I_s, H), param(I_s, H), param(H, I_s)
        else:
            self.ws_gate = self.ws_up = self.ws_down = None
        self.mode, self.capacity, self.minibatch, self.swiglu_limit = mode, capacity, minibatch, swiglu_limit
        self.macrobatch = macrobatch

    def forward(self, x, router_w, top_experts):
        return mok_layer(x, router_w, top_experts, self.w_gate, self.w_up, self.w_down, self.ws_gate, self.ws_up,
                         self.ws_down, self.mode, self.capacity, self.minibatch, self.swiglu_limit, self.macrobatch)

"""Helpers shared by the GPU parity tests: run the layer through the C ABI and
compare with the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_mok_gb300 import inputs as gen

BF16_TOL = 5e-3     # relative L2, BF16 path and MXFP8 vs its same-quantisation oracle
MX_UNQ_TOL = 3e-2   # relative L2, MXFP8 forward vs the unquantised oracle


_built = False


def mok():
    global _built
    if not _built:
        import __graft_entry__ as g

        g.build()
        _built = True
    import mixture_experts_layer_mok_gb300 as m

    return m


def rel_l2(a, b) -> float:
    a = a.detach().double().cpu().numpy() if hasattr(a, "detach") else np.asarray(a, np.float64)
    b = b.detach().double().cpu().numpy() if hasattr(b, "detach") else np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def weights_of(g, mode="bf16"):
    m = mok()
    w = m.Weights(g.w_gate, g.w_up, g.w_down, g.ws_gate, g.ws_up, g.ws_down)
    if mode in ("mxfp8", "mxfp8_full"):
        w = m.quantize_weights(w, backward=(mode == "mxfp8_full"))
    return w


def run_layer(inp, mode="bf16", capacity=0.5, minibatch=0, device="cuda", swiglu_limit=0.0):
    """Forward + backward through the C ABI; returns (y, grads, sched, ctx)."""
    m = mok()
    g = inp.to(device)
    sched = m.schedule(g.top_experts, inp.meta["E"], capacity)
    w = weights_of(g, mode)
    y, ctx = m.forward(g.x, g.router_w, sched, w, mode=mode, minibatch=minibatch, swiglu_limit=swiglu_limit)
    grads = m.backward(g.dy, g.x, g.router_w, sched, ctx, w, minibatch=minibatch)
    torch.cuda.synchronize()
    return y, grads, sched, ctx


def oracle_args(inp):
    return (inp.x, inp.router_w, inp.top_experts, inp.w_gate, inp.w_up, inp.w_down,
            inp.ws_gate, inp.ws_up, inp.ws_down)


def oracle_fwd_bwd(inp, mode="bf16", swiglu_limit=0.0):
    a = oracle_args(inp)
    if mode == "mxfp8":
        y = oracle.layer_forward_mxfp8(*a, swiglu_limit=swiglu_limit)
        g = oracle.layer_backward_mxfp8(*a[:6], inp.dy, *a[6:], swiglu_limit=swiglu_limit)
    elif mode == "mxfp8_full":
        y = oracle.layer_forward_mxfp8(*a, swiglu_limit=swiglu_limit)
        g = oracle.layer_backward_mxfp8_full(*a[:6], inp.dy, *a[6:], swiglu_limit=swiglu_limit)
    else:
        y = oracle.layer_forward(*a, swiglu_limit=swiglu_limit)
        g = oracle.layer_backward(*a[:6], inp.dy, *a[6:], swiglu_limit=swiglu_limit)
    return y, g


GRAD_KEYS = ("dx", "d_router_w", "d_w_gate", "d_w_up", "d_w_down", "d_ws_gate", "d_ws_up", "d_ws_down")


def compare_all(y, grads, y_ref, g_ref, tol=BF16_TOL):
    errs = {"y": rel_l2(y, y_ref)}
    for key in GRAD_KEYS:
        if key in g_ref:
            errs[key] = rel_l2(grads[key], g_ref[key])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    return errs, bad


def subset_inputs(inp, tokens):
    """The same layer restricted to a subset of tokens (the layer is per-token
    in y, dx and d_router_w)."""
    idx = torch.as_tensor(tokens, dtype=torch.int64)
    return gen.LayerInputs(inp.x[idx], inp.router_w[idx], inp.top_experts[idx], inp.w_gate, inp.w_up,
                           inp.w_down, inp.ws_gate, inp.ws_up, inp.ws_down,
                           None if inp.dy is None else inp.dy[idx], dict(inp.meta))


def token_inputs(inp, t):
    """Token t alone, with its k experts remapped to a compact weight set (the
    layer is per-token, so the oracle on this gives y[t], dx[t], d_w[t])."""
    ex = inp.top_experts[t].cpu()
    k = ex.numel()
    sl = lambda a: None if a is None else a.cpu()  # noqa: E731
    return gen.LayerInputs(sl(inp.x[t:t + 1]), sl(inp.router_w[t:t + 1]),
                           torch.arange(k, dtype=torch.int64).reshape(1, k),
                           sl(inp.w_gate[ex.to(inp.w_gate.device)]), sl(inp.w_up[ex.to(inp.w_up.device)]),
                           sl(inp.w_down[ex.to(inp.w_down.device)]), sl(inp.ws_gate), sl(inp.ws_up), sl(inp.ws_down),
                           sl(inp.dy[t:t + 1]), dict(inp.meta))


def expert_slice_inputs(inp, e, i0, i1):
    """Only the rows routed to expert e (a k = 1 layer) and only intermediate
    columns [i0, i1): the oracle on this gives dW_gate[e][i0:i1],
    dW_up[e][i0:i1] and dW_down[e][:, i0:i1] exactly (those slices depend only
    on the same columns of h)."""
    te = inp.top_experts
    t_e, j_e = torch.nonzero(te == e, as_tuple=True)
    dev = inp.x.device
    return gen.LayerInputs(inp.x[t_e].cpu(), inp.router_w[t_e, j_e].reshape(-1, 1).cpu(),
                           torch.zeros((t_e.numel(), 1), dtype=torch.int64),
                           inp.w_gate[e:e + 1, i0:i1].cpu(), inp.w_up[e:e + 1, i0:i1].cpu(),
                           inp.w_down[e:e + 1, :, i0:i1].contiguous().cpu(), None, None, None,
                           inp.dy[t_e].cpu(), dict(inp.meta)), t_e.to(dev)


def gate_up_preactivations(inp, mode="bf16"):
    """Every gate and |up| pre-activation value the layer's forward forms
    (float64; those of the quantised forward in the MXFP8 modes), sorted."""
    x = inp.x.double().numpy()
    quant = mode in ("mxfp8", "mxfp8_full")
    q = oracle.mxfp8_roundtrip if quant else (lambda a: a)
    xq = q(x)
    te = inp.top_experts.numpy()
    vals = []
    for e in range(inp.w_gate.shape[0]):
        rows = np.nonzero((te == e).any(axis=1))[0]
        if rows.size == 0:
            continue
        vals.append((xq[rows] @ q(inp.w_gate[e].double().numpy()).T).ravel())
        vals.append(np.abs(xq[rows] @ q(inp.w_up[e].double().numpy()).T).ravel())
    if inp.ws_gate is not None:
        vals.append((xq @ q(inp.ws_gate.double().numpy()).T).ravel())
        vals.append(np.abs(xq @ q(inp.ws_up.double().numpy()).T).ravel())
    return np.sort(np.concatenate(vals))


def clamp_limit(inp, mode="bf16", lo_q=0.5, hi_q=0.8):
    """A swiglu_limit for parity tests: a midpoint between two consecutive
    bf16 values (so a value and its bf16 rounding fall on the same side of
    it), inside the given quantile range of the pre-activations, chosen as
    far as possible from every pre-activation value.  The kernels decide the
    clamp's derivative on bf16-rounded fp32 pre-activations and the oracle on
    float64 ones; at such a limit the two decisions agree unless a value lies
    within the fp32 accumulation error of the limit.  Returns (limit,
    distance to the nearest value)."""
    vals = gate_up_preactivations(inp, mode)
    lo, hi = np.quantile(vals, lo_q), np.quantile(vals, hi_q)
    assert lo > 0
    b0 = int(np.float32(lo).view(np.uint32)) >> 16
    b1 = int(np.float32(hi).view(np.uint32)) >> 16
    bf = (np.arange(b0, b1 + 2, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    mids = 0.5 * (bf[:-1] + bf[1:])              # exact in float32
    pos = np.searchsorted(vals, mids)
    left = np.abs(mids - vals[np.clip(pos - 1, 0, len(vals) - 1)])
    right = np.abs(vals[np.clip(pos, 0, len(vals) - 1)] - mids)
    gap = np.minimum(left, right)
    i = int(np.argmax(gap))
    return float(np.float32(mids[i])), float(gap[i])

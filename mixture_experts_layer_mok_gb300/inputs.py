"""Seeded synthetic inputs for the MoK layer.

This module holds none of the layer's arithmetic.  It draws the tensors that a
caller of the layer would supply (activations, routing decisions from a
softmax/top-k router that lives outside the library, weights, the upstream
gradient) and is the one piece both the CUDA path and the CPU oracle are fed
from.

Draw order (one ``torch.Generator``): x, router logits, routed W_gate, W_up,
W_down, shared W_gate, W_up, W_down, dy.  x, dy ~ N(0, 1) and weights
~ N(0, 0.02), all rounded to bf16; logits ~ N(0, 1) in fp32, plus an optional
per-expert bias log(p_e) with p_e proportional to rank^-s (Zipf) for skewed
routing.  The router keeps the k largest softmax probabilities (ties go to the
lower expert index; j runs in descending probability) and renormalises them to
sum to one in fp32.  Routed weight layouts follow the MoK-native layouts of
the NeMo AutoModel MoK expert backend (gate/up [E, I, H], down [E, H, I]).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Named workloads (sizes of the layer configurations this library is measured on)
WORKLOADS = {
    "tiny": dict(T=128, H=128, I=256, E=8, k=2, I_s=0, skew=None,
                 minibatch=0, capacity=0.5, mode="bf16"),
    "bf16_T4096": dict(T=4096, H=2048, I=1024, E=64, k=8, I_s=2048, skew=None,
                       minibatch=2048, capacity=0.5, mode="bf16"),
    "mxfp8_T4096": dict(T=4096, H=2048, I=1024, E=64, k=8, I_s=2048, skew=None,
                        minibatch=2048, capacity=0.5, mode="mxfp8"),
    "mxfp8full_T4096": dict(T=4096, H=2048, I=1024, E=64, k=8, I_s=2048, skew=None,
                            minibatch=2048, capacity=0.5, mode="mxfp8_full"),
    "skewed_T16384": dict(T=16384, H=4096, I=1536, E=128, k=8, I_s=0, skew=1.2,
                          minibatch=4096, capacity=0.5, mode="bf16"),
    "large_T65536": dict(T=65536, H=7168, I=2048, E=256, k=8, I_s=2048, skew=None,
                         minibatch=4096, capacity=0.5, mode="mxfp8"),
    "mxfp8full_T65536": dict(T=65536, H=7168, I=2048, E=256, k=8, I_s=2048, skew=None,
                             minibatch=4096, capacity=0.5, mode="mxfp8_full"),
}


@dataclass
class LayerInputs:
    x: torch.Tensor            # bf16 [T, H]
    router_w: torch.Tensor     # fp32 [T, k]
    top_experts: torch.Tensor  # int64 [T, k]
    w_gate: torch.Tensor       # bf16 [E, I, H]
    w_up: torch.Tensor         # bf16 [E, I, H]
    w_down: torch.Tensor       # bf16 [E, H, I]
    ws_gate: torch.Tensor | None = None  # bf16 [I_s, H]
    ws_up: torch.Tensor | None = None    # bf16 [I_s, H]
    ws_down: torch.Tensor | None = None  # bf16 [H, I_s]
    dy: torch.Tensor | None = None       # bf16 [T, H]
    meta: dict = field(default_factory=dict)

    def to(self, device):
        kw = {}
        for name in ("x", "router_w", "top_experts", "w_gate", "w_up", "w_down",
                     "ws_gate", "ws_up", "ws_down", "dy"):
            v = getattr(self, name)
            kw[name] = None if v is None else v.to(device)
        return LayerInputs(meta=dict(self.meta), **kw)


def _normal(shape, std, gen, device, chunk=1 << 26):
    """N(0, std) rounded to bf16, drawn in chunks to bound fp32 temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        v = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        flat[s:s + n].copy_(v)
    return out


def route(logits: torch.Tensor, k: int):
    """Softmax -> top-k (stable: ties to the lower index) -> renormalise."""
    probs = torch.softmax(logits.float(), dim=-1)
    order = torch.sort(-probs, dim=-1, stable=True).indices[:, :k]
    top_p = torch.gather(probs, 1, order)
    w = top_p / top_p.sum(dim=-1, keepdim=True)
    return w.contiguous(), order.to(torch.int64).contiguous()


def make_layer_inputs(T, H, I, E, k, I_s=0, skew=None, seed=0, device="cpu",
                      with_dy=True) -> LayerInputs:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = _normal((T, H), 1.0, gen, device)
    logits = torch.randn(T, E, generator=gen, device=device, dtype=torch.float32)
    if skew is not None:
        rank = torch.arange(1, E + 1, dtype=torch.float64, device=device)
        p = rank.pow(-float(skew))
        logits = logits + torch.log(p / p.sum()).float()
    router_w, top = route(logits, k)
    w_gate = _normal((E, I, H), 0.02, gen, device)
    w_up = _normal((E, I, H), 0.02, gen, device)
    w_down = _normal((E, H, I), 0.02, gen, device)
    ws_gate = ws_up = ws_down = None
    if I_s:
        ws_gate = _normal((I_s, H), 0.02, gen, device)
        ws_up = _normal((I_s, H), 0.02, gen, device)
        ws_down = _normal((H, I_s), 0.02, gen, device)
    dy = _normal((T, H), 1.0, gen, device) if with_dy else None
    meta = dict(T=T, H=H, I=I, E=E, k=k, I_s=I_s, skew=skew, seed=seed)
    return LayerInputs(x, router_w, top, w_gate, w_up, w_down, ws_gate, ws_up,
                       ws_down, dy, meta)


def make_workload(name: str, seed=0, device="cpu", with_dy=True) -> LayerInputs:
    c = WORKLOADS[name]
    inp = make_layer_inputs(c["T"], c["H"], c["I"], c["E"], c["k"], c["I_s"],
                            c["skew"], seed, device, with_dy)
    inp.meta.update(name=name, mode=c["mode"], minibatch=c["minibatch"],
                    capacity=c["capacity"])
    return inp


def make_routing(T, k, E, seed=0, skew=None) -> torch.Tensor:
    """Routing decisions only (int64 [T, k]) for schedule tests."""
    gen = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=gen)
    if skew is not None:
        rank = torch.arange(1, E + 1, dtype=torch.float64)
        p = rank.pow(-float(skew))
        logits = logits + torch.log(p / p.sum()).float()
    return route(logits, k)[1]


def make_matrix(R, K, std=1.0, seed=0) -> torch.Tensor:
    """A bf16 [R, K] matrix for quantiser tests."""
    gen = torch.Generator().manual_seed(seed)
    return _normal((R, K), std, gen, "cpu")

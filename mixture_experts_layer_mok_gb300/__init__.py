"""MoK layer on GB300: Python binding of libmok (argument marshalling only).

The calls mirror the C ABI in ``include/mok.h``:
``schedule`` (built once from the routing), ``mxfp8_quantize`` (weights,
ahead of time), ``forward`` -> (y, ctx), ``backward`` -> gradients.  PyTorch
provides device memory and the stream; every step of the layer runs in the
library's CUDA kernels.  The library is loaded on first use, never at import
time, so importing this package creates no CUDA context.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import MokError  # noqa: F401

__all__ = ["schedule", "schedule_noalloc", "mxfp8_quantize", "mxfp8_quantize_t", "mxfp8_quantize_dual", "forward",
           "backward", "Schedule", "Weights", "Context", "MokError", "quantize_weights", "macrobatch_plan", "MODES"]

# forward/backward precision: "bf16"; "mxfp8" (MXFP8 forward GEMMs, bf16
# backward); "mxfp8_full" (MXFP8 forward and backward GEMMs)
MODES = {"bf16": _lib.MOK_MODE_BF16, "mxfp8": _lib.MOK_MODE_MXFP8_FWD, "mxfp8_full": _lib.MOK_MODE_MXFP8}


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")
    return t


def _pointer_fields(struct_cls):
    return tuple(name for name, typ in struct_cls._fields_ if typ is _lib.P)


def _flatten_struct(c, buf):
    """The struct's scalar fields and its pointers: a pointer into buf as
    ("off", offset), NULL as None, and one that points elsewhere (the
    library's own fixed scratch array, which never moves) as ("abs", address).
    Everything needed to rebuild the struct over a copy of buf."""
    base, size = buf.data_ptr(), buf.numel() * buf.element_size()
    scalars, ptrs = {}, {}
    for name, _ in c._fields_:
        v = getattr(c, name)
        if name in _pointer_fields(type(c)):
            ptrs[name] = None if not v else (("off", v - base) if base <= v < base + size else ("abs", v))
        else:
            scalars[name] = v
    return scalars, ptrs


def _unflatten_struct(struct_cls, buf, scalars, ptrs):
    c = struct_cls(**scalars)
    base, size = buf.data_ptr(), buf.numel() * buf.element_size()
    for name, p in ptrs.items():
        if p is None:
            continue
        kind, v = p
        if kind == "off":
            if not 0 <= v < size:
                raise ValueError(f"{name}: offset {v} outside the {size}-byte buffer")
            v = base + v
        setattr(c, name, v)
    return c


@dataclass
class Schedule:
    """The dispatch/combine schedule; ``buf`` owns the device memory."""
    T: int
    k: int
    E: int
    buf: torch.Tensor
    c: _lib.MokSchedule

    def flatten(self):
        """(buf, meta): the one tensor that holds the schedule, and plain
        metadata.  Saving ``buf`` through ``save_for_backward`` lets saved-tensor
        hooks (offload, checkpointing) move it; ``unflatten`` rebuilds the
        schedule over wherever it lands (the arrays hold no pointers)."""
        return self.buf, (self.T, self.k, self.E) + _flatten_struct(self.c, self.buf)

    @classmethod
    def unflatten(cls, buf, meta):
        T, k, E, scalars, offsets = meta
        return cls(T, k, E, buf, _unflatten_struct(_lib.MokSchedule, buf, scalars, offsets))

    def status(self):
        st, nt, P = C.c_int32(), C.c_int32(), C.c_int32()
        _lib.check(_lib.load().mok_schedule_status(C.byref(self.c), C.byref(st), C.byref(nt), C.byref(P)),
                   "mok_schedule_status")
        return st.value, nt.value, P.value

    def arrays(self):
        """Device int32 views of the schedule arrays (for inspection/tests)."""
        base = self.buf.data_ptr()
        mt = self.c.max_tiles
        view = {}
        for name, n in (("cnt", self.E), ("row0", self.E + 1), ("row_src", mt * 128),
                        ("slot_row", self.T * self.k), ("tile_expert", mt), ("tile_row0", mt),
                        ("tile_rows", mt), ("header", 8), ("pair_tile", 2 * mt),
                        ("unit_group", 2 * mt)):
            off = getattr(self.c, name) - base
            view[name] = self.buf[off: off + 4 * n].view(torch.int32)
        return view


@dataclass
class Weights:
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    ws_gate: torch.Tensor | None = None
    ws_up: torch.Tensor | None = None
    ws_down: torch.Tensor | None = None
    mx: dict | None = None  # name -> (codes, scales) for the MXFP8 modes

    @property
    def dims(self):
        E, I, H = self.w_gate.shape
        I_s = 0 if self.ws_gate is None else self.ws_gate.shape[0]
        return E, H, I, I_s

    def struct(self):
        E, H, I, I_s = self.dims
        _need(self.w_gate, torch.bfloat16, (E, I, H), "w_gate")
        _need(self.w_up, torch.bfloat16, (E, I, H), "w_up")
        _need(self.w_down, torch.bfloat16, (E, H, I), "w_down")
        if I_s:
            _need(self.ws_gate, torch.bfloat16, (I_s, H), "ws_gate")
            _need(self.ws_up, torch.bfloat16, (I_s, H), "ws_up")
            _need(self.ws_down, torch.bfloat16, (H, I_s), "ws_down")
        w = _lib.MokWeights(E=E, H=H, I=I, I_s=I_s)
        w.w_gate, w.w_up, w.w_down = (t.data_ptr() for t in (self.w_gate, self.w_up, self.w_down))
        if I_s:
            w.ws_gate, w.ws_up, w.ws_down = (t.data_ptr() for t in (self.ws_gate, self.ws_up, self.ws_down))
        if self.mx:
            for name, (codes, scales) in self.mx.items():
                setattr(w, "mx" + name, codes.data_ptr())
                setattr(w, "mx" + name + "_sc", scales.data_ptr())
        return w


@dataclass
class Context:
    buf: torch.Tensor
    c: _lib.MokCtx
    mode: int

    def flatten(self):
        """(buf, meta), as ``Schedule.flatten``: the forward's saved
        activations live in ``buf`` and hold no pointers."""
        return self.buf, (self.mode,) + _flatten_struct(self.c, self.buf)

    @classmethod
    def unflatten(cls, buf, meta):
        mode, scalars, offsets = meta
        return cls(buf, _unflatten_struct(_lib.MokCtx, buf, scalars, offsets), mode)

    def status(self) -> int:
        st = C.c_int32()
        _lib.check(_lib.load().mok_ctx_status(C.byref(self.c), C.byref(st)), "mok_ctx_status")
        return st.value


def schedule(top_experts: torch.Tensor, E: int, capacity_multiplier: float = 0.5, stream=None) -> Schedule:
    lib = _lib.load()
    T, k = top_experts.shape
    _need(top_experts, torch.int64, (T, k), "top_experts")
    nbytes = lib.mok_schedule_bytes(T, k, E)
    if nbytes == 0:
        raise ValueError("invalid schedule shape")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=top_experts.device)
    c = _lib.MokSchedule()
    _lib.check(lib.mok_schedule(_ptr(top_experts), T, k, E, float(capacity_multiplier), _ptr(buf), nbytes,
                                C.byref(c), _stream(stream)), "mok_schedule")
    return Schedule(T, k, E, buf, c)


def schedule_noalloc(top_experts: torch.Tensor, E: int, capacity_multiplier: float = 0.5, out_buf=None,
                     stream=None) -> Schedule:
    """Same schedule as ``schedule``; the library takes the build's scratch from
    its own fixed device array (for callers that cannot allocate).  Pass
    ``out_buf`` (uint8, at least mok_schedule_bytes) to allocate nothing here."""
    lib = _lib.load()
    T, k = top_experts.shape
    _need(top_experts, torch.int64, (T, k), "top_experts")
    nbytes = lib.mok_schedule_bytes(T, k, E)
    if nbytes == 0:
        raise ValueError("invalid schedule shape")
    buf = out_buf if out_buf is not None else torch.empty(nbytes, dtype=torch.uint8, device=top_experts.device)
    c = _lib.MokSchedule()
    _lib.check(lib.mok_schedule_noalloc(_ptr(top_experts), T, k, E, float(capacity_multiplier), _ptr(buf),
                                        buf.numel(), C.byref(c), _stream(stream)), "mok_schedule_noalloc")
    return Schedule(T, k, E, buf, c)


def mxfp8_quantize(x: torch.Tensor, stream=None):
    """bf16 [..., K] -> (E4M3 codes uint8 [..., K], E8M0 scales uint8 [..., K/32])."""
    lib = _lib.load()
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be contiguous CUDA bf16")
    K = x.shape[-1]
    rows = x.numel() // K if K else 0
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty(tuple(x.shape[:-1]) + (K // 32,), dtype=torch.uint8, device=x.device)
    _lib.check(lib.mok_mxfp8_quantize(_ptr(x), rows, K, _ptr(codes), _ptr(scales), _stream(stream)),
               "mok_mxfp8_quantize")
    return codes, scales


def mxfp8_quantize_t(x: torch.Tensor, stream=None):
    """bf16 [batch, rows, cols] (or [rows, cols]) -> (E4M3 codes of the
    transpose uint8 [batch, cols, rows], E8M0 scales uint8 [batch, cols,
    rows/32]): one scale per 32 consecutive rows of each column."""
    lib = _lib.load()
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.dim() not in (2, 3):
        raise ValueError("x must be a contiguous CUDA bf16 matrix or batch of matrices")
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    B, R, Cc = x3.shape
    codes = torch.empty((B, Cc, R), dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, Cc, R // 32), dtype=torch.uint8, device=x.device)
    _lib.check(lib.mok_mxfp8_quantize_t(_ptr(x3), B, R, Cc, _ptr(codes), _ptr(scales), _stream(stream)),
               "mok_mxfp8_quantize_t")
    if x.dim() == 2:
        codes, scales = codes[0], scales[0]
    return codes, scales


def mxfp8_quantize_dual(x: torch.Tensor, stream=None):
    """Both orientations from one read: ((codes, scales) as ``mxfp8_quantize``,
    (codes_t, scales_t) as ``mxfp8_quantize_t``), for a [batch, rows, cols] or
    [rows, cols] bf16 tensor."""
    lib = _lib.load()
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.dim() not in (2, 3):
        raise ValueError("x must be a contiguous CUDA bf16 matrix or batch of matrices")
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    B, R, Cc = x3.shape
    codes = torch.empty((B, R, Cc), dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, R, Cc // 32), dtype=torch.uint8, device=x.device)
    codes_t = torch.empty((B, Cc, R), dtype=torch.uint8, device=x.device)
    scales_t = torch.empty((B, Cc, R // 32), dtype=torch.uint8, device=x.device)
    _lib.check(lib.mok_mxfp8_quantize_dual(_ptr(x3), B, R, Cc, _ptr(codes), _ptr(scales), _ptr(codes_t),
                                           _ptr(scales_t), _stream(stream)), "mok_mxfp8_quantize_dual")
    if x.dim() == 2:
        codes, scales, codes_t, scales_t = codes[0], scales[0], codes_t[0], scales_t[0]
    return (codes, scales), (codes_t, scales_t)


def quantize_weights(w: Weights, stream=None, backward: bool = False) -> Weights:
    """Prequantise every weight along its K axis for the MXFP8 modes; with
    ``backward`` also along its leading axis (the transposed copies the
    "mxfp8_full" backward's dgrad GEMMs read)."""
    names = [("_gate", "t_gate", w.w_gate), ("_up", "t_up", w.w_up), ("_down", "t_down", w.w_down)]
    if w.ws_gate is not None:
        names += [("s_gate", "ts_gate", w.ws_gate), ("s_up", "ts_up", w.ws_up), ("s_down", "ts_down", w.ws_down)]
    mx = {}
    for fwd_name, bwd_name, t in names:
        if backward:   # both copies from one read of the weight
            mx[fwd_name], mx[bwd_name] = mxfp8_quantize_dual(t, stream)
        else:
            mx[fwd_name] = mxfp8_quantize(t, stream)
    return Weights(w.w_gate, w.w_up, w.w_down, w.ws_gate, w.ws_up, w.ws_down, mx)


def macrobatch_plan(cnt, macrobatch: int):
    """The windows a macrobatch ring of ``macrobatch`` rows runs the routed
    experts in, for per-expert row counts ``cnt`` (a sequence of ints, e.g. the
    schedule's ``cnt`` read back): a list of (first expert, end expert).  Host
    only; raises MokError(MOK_ERR_CAPACITY) when one expert does not fit."""
    lib = _lib.load()
    E = len(cnt)
    arr = (C.c_int32 * E)(*[int(c) for c in cnt])
    first = (C.c_int32 * (E + 1))()
    nw = C.c_int()
    _lib.check(lib.mok_macrobatch_plan(arr, E, int(macrobatch), first, C.byref(nw)), "mok_macrobatch_plan")
    return [(first[i], first[i + 1]) for i in range(nw.value)]


def _config(mode, minibatch, debug, events=None, dispatch="auto", swiglu_limit=0.0, macrobatch=0):
    cfg = _lib.MokConfig(mode=mode, minibatch_size=minibatch, debug_flags=debug, dispatch=_lib.DISPATCH[dispatch],
                         num_events=0, events=None, swiglu_limit=float(swiglu_limit),
                         macrobatch_size=int(macrobatch))
    if events is not None:
        if len(events) != 2 * _lib.MOK_NUM_STAGES:
            raise ValueError("events must hold 2 * MOK_NUM_STAGES torch.cuda.Event objects (or None)")
        for e in events:                 # torch creates the CUDA event on first record
            if e is not None and not e.cuda_event:
                e.record()
        arr = (C.c_void_p * len(events))(*[None if e is None else e.cuda_event for e in events])
        cfg.num_events = len(events)
        cfg.events = C.cast(arr, C.POINTER(C.c_void_p))
        cfg._keep = arr
    return cfg


def forward(x, router_w, sched: Schedule, weights: Weights, mode: str = "bf16", minibatch: int = 0,
            debug: int = 0, out=None, ctx_buf=None, stream=None, events=None, dispatch="auto",
            swiglu_limit: float = 0.0, macrobatch: int = 0):
    """y = layer(x); returns (y, Context).  ``mode`` is "bf16", "mxfp8" or
    "mxfp8_full" (see ``MODES``; the backward follows the forward's mode);
    ``dispatch`` is "auto", "permute" or "fused" (same results, different kernels).
    ``swiglu_limit`` > 0 clamps the SwiGLU pre-activations (gate to <= L, up
    to [-L, L]); the backward follows the forward's value.
    ``macrobatch`` > 0: rows of the token ring (mok_config_t.macrobatch_size):
    the routed experts run in windows of whole experts over scratch of that
    many rows, with the same result bits (reads the expert counts back once).
    ``events``: optional list of 2 * MOK_NUM_STAGES torch.cuda.Event (timing); a
    None entry records nothing (each record costs a few microseconds on the
    device, so a timing run can watch one stage alone)."""
    lib = _lib.load()
    if mode not in MODES:
        raise ValueError(f"mode must be one of {sorted(MODES)}")
    m = MODES[mode]
    E, H, I, I_s = weights.dims
    T, k = sched.T, sched.k
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_w, torch.float32, (T, k), "router_w")
    ws = weights.struct()
    nbytes = lib.mok_ctx_bytes_ring(T, k, E, H, I, I_s, m, int(macrobatch))
    if nbytes == 0:
        raise ValueError("shape outside the kernels' contract")
    if ctx_buf is None or ctx_buf.numel() < nbytes:
        ctx_buf = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    c = _lib.MokCtx()
    cfg = _config(m, minibatch, debug, events, dispatch, swiglu_limit, macrobatch)
    _lib.check(lib.mok_forward(C.byref(cfg), _ptr(x), _ptr(router_w), C.byref(sched.c), C.byref(ws), _ptr(y),
                               _ptr(ctx_buf), ctx_buf.numel(), C.byref(c), _stream(stream)), "mok_forward")
    return y, Context(ctx_buf, c, m)


def backward(dy, x, router_w, sched: Schedule, ctx: Context, weights: Weights, minibatch: int = 0,
             grads: dict | None = None, ws_buf=None, stream=None, events=None, dispatch="auto", debug: int = 0,
             macrobatch: int = 0):
    """Returns dict dx, d_router_w, d_w_gate, d_w_up, d_w_down (+ d_ws_* with a shared expert).
    ``macrobatch``: the backward's own token ring (see ``forward``)."""
    lib = _lib.load()
    E, H, I, I_s = weights.dims
    T, k = sched.T, sched.k
    _need(dy, torch.bfloat16, (T, H), "dy")
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_w, torch.float32, (T, k), "router_w")
    dev = dy.device
    if grads is None:
        grads = {"dx": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                 "d_router_w": torch.empty((T, k), dtype=torch.float32, device=dev),
                 "d_w_gate": torch.empty_like(weights.w_gate), "d_w_up": torch.empty_like(weights.w_up),
                 "d_w_down": torch.empty_like(weights.w_down)}
        if I_s:
            grads.update(d_ws_gate=torch.empty_like(weights.ws_gate), d_ws_up=torch.empty_like(weights.ws_up),
                         d_ws_down=torch.empty_like(weights.ws_down))
    g = _lib.MokWeightGrads()
    for name in ("d_w_gate", "d_w_up", "d_w_down", "d_ws_gate", "d_ws_up", "d_ws_down"):
        if name in grads:
            setattr(g, name, grads[name].data_ptr())
    nbytes = lib.mok_bwd_workspace_bytes_ring(T, k, E, H, I, I_s, ctx.mode, int(macrobatch))
    if nbytes == 0:
        raise ValueError("shape outside the kernels' contract")
    if ws_buf is None or ws_buf.numel() < nbytes:
        ws_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    cfg = _config(ctx.mode, minibatch, debug, events, dispatch, macrobatch=macrobatch)
    wsd = weights.struct()
    _lib.check(lib.mok_backward(C.byref(cfg), _ptr(dy), _ptr(x), _ptr(router_w), C.byref(sched.c),
                                C.byref(ctx.c), C.byref(wsd), _ptr(grads["dx"]), _ptr(grads["d_router_w"]),
                                C.byref(g), _ptr(ws_buf), ws_buf.numel(), _stream(stream)), "mok_backward")
    return grads

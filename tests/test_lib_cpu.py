"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every symbol include/mok.h declares, sizes its buffers consistently
and rejects bad arguments before touching the device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    from mixture_experts_layer_mok_gb300 import _lib

    return _lib.load()


def _header_symbols():
    text = open(os.path.join(ROOT, "include", "mok.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mok_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = _header_symbols()
    assert len(syms) >= 11
    for s in syms:
        assert hasattr(lib, s), s
    from mixture_experts_layer_mok_gb300 import _lib

    assert sorted(_lib.SIGNATURES) == syms


def test_version_and_error(lib):
    assert lib.mok_version() >= 1
    assert isinstance(lib.mok_last_error(), bytes)


def test_buffer_sizes(lib):
    T, k, E = 4096, 8, 64
    mt = (T * k + 127 * E) // 128
    sb = lib.mok_schedule_bytes(T, k, E)
    assert sb >= 4 * (E + E + 1 + mt * 128 + T * k + 3 * mt + 8)
    H, I, Is = 2048, 1024, 2048
    cb = lib.mok_ctx_bytes(T, k, E, H, I, Is, 0)
    # gate|up + h per padded row, slots per routed row, shared gate|up/h/out
    assert cb >= 2 * (mt * 128 * 3 * I + T * k * H + T * 3 * Is + T * H)
    # MXFP8: bf16 gate|up (saved) and slots, E4M3 codes of x (token and
    # schedule order) and of h, plus their scales (1/32 of the codes)
    mb = lib.mok_ctx_bytes(T, k, E, H, I, Is, 1)
    codes = mt * 128 * (H + I) + T * (H + Is)
    assert mb >= 2 * (mt * 128 * 2 * I + T * k * H + T * 2 * Is + T * H) + codes + codes // 32
    wb = lib.mok_bwd_workspace_bytes(T, k, E, H, I, Is, 0)
    assert wb >= 2 * (mt * 128 * 3 * I + T * k * H)
    # after an MXFP8 forward the context holds x's schedule-order rows: no copy
    assert 0 <= wb - lib.mok_bwd_workspace_bytes(T, k, E, H, I, Is, 1) - 2 * mt * 128 * H < 256
    # MXFP8 backward: E4M3 codes of dy (rows and transposed), x (transposed),
    # dG|dU (rows and transposed) and w h (transposed) in place of the bf16
    # permuted copies and SwiGLU-backward rows (the dx rows in schedule order
    # go to the context's slots)
    wm = lib.mok_bwd_workspace_bytes(T, k, E, H, I, Is, 2)
    assert wm >= mt * 128 * (3 * H + 5 * I)
    assert wm < wb
    assert lib.mok_bwd_workspace_bytes(T, k, E, H, I, Is, 3) == 0
    # shapes outside the contract report 0
    assert lib.mok_ctx_bytes(T, k, E, 100, I, Is, 0) == 0
    assert lib.mok_ctx_bytes(T, k, E, H, 96, Is, 0) == 0
    assert lib.mok_schedule_bytes(0, k, E) == 0


def test_argument_errors_need_no_device(lib):
    from mixture_experts_layer_mok_gb300 import _lib

    s = _lib.MokSchedule()
    assert lib.mok_schedule(None, 4, 2, 8, 0.5, None, 0, C.byref(s), None) == _lib.MOK_ERR_INVALID_ARG
    buf = C.create_string_buffer(1 << 16)
    fake = C.c_void_p(16)  # never dereferenced: validation fails first
    assert lib.mok_schedule(fake, 4, 0, 8, 0.5, fake, 1 << 16, C.byref(s), None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_schedule(fake, 4, 2, 2000, 0.5, fake, 1 << 16, C.byref(s), None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_schedule(fake, 4, 2, 8, float("nan"), fake, 1 << 16, C.byref(s), None) == \
        _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_schedule(fake, 4, 2, 8, -1.0, fake, 1 << 16, C.byref(s), None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_schedule(fake, 4, 2, 8, 0.5, fake, 16, C.byref(s), None) == _lib.MOK_ERR_INVALID_ARG
    assert b"too small" in lib.mok_last_error()
    assert lib.mok_mxfp8_quantize(fake, 4, 33, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize_t(fake, 1, 48, 64, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG   # rows % 32
    assert lib.mok_mxfp8_quantize_t(fake, 1, 64, 96, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG   # cols % 64
    assert lib.mok_mxfp8_quantize_t(fake, -1, 64, 64, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize_t(None, 1, 64, 64, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize_t(fake, 0, 64, 64, fake, fake, None) == _lib.MOK_OK   # nothing to do
    assert lib.mok_mxfp8_quantize_dual(fake, 1, 48, 64, fake, fake, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize_dual(fake, 1, 64, 64, fake, fake, None, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize(C.c_void_p(17), 4, 64, fake, fake, None) == _lib.MOK_ERR_INVALID_ARG
    assert lib.mok_mxfp8_quantize(None, 0, 64, None, None, None) == _lib.MOK_OK   # empty input
    cfg = _lib.MokConfig(mode=7)
    assert lib.mok_forward(C.byref(cfg), fake, fake, C.byref(s), None, fake, fake, 0, None, None) == \
        _lib.MOK_ERR_INVALID_ARG
    w = _lib.MokWeights(E=8, H=128, I=128, I_s=0)
    ctx = _lib.MokCtx()
    for bad in (-0.5, float("nan"), float("inf")):   # swiglu_limit must be finite and >= 0
        cfg = _lib.MokConfig(mode=0, swiglu_limit=bad)
        assert lib.mok_forward(C.byref(cfg), fake, fake, C.byref(s), C.byref(w), fake, fake, 1 << 16,
                               C.byref(ctx), None) == _lib.MOK_ERR_INVALID_ARG
        assert b"swiglu_limit" in lib.mok_last_error()
    del buf


def test_layer_argument_checks_need_no_device(lib):
    """Mismatched or misaligned arguments to the layer calls are refused on
    the host, before any device work."""
    from mixture_experts_layer_mok_gb300 import _lib

    fake = C.c_void_p(16)           # never dereferenced: validation fails first
    odd = C.c_void_p(16 + 8)        # not 16-byte aligned
    cfg = _lib.MokConfig(mode=0)
    s = _lib.MokSchedule(T=8, k=2, E=4, max_tiles=6)
    w = _lib.MokWeights(E=4, H=128, I=128, I_s=128, w_gate=fake, w_up=fake, w_down=fake,
                        ws_gate=fake, ws_up=odd, ws_down=fake)
    ctx = _lib.MokCtx()
    assert lib.mok_forward(C.byref(cfg), fake, fake, C.byref(s), C.byref(w), fake, fake, 1 << 40,
                           C.byref(ctx), None) == _lib.MOK_ERR_INVALID_ARG
    assert b"misaligned shared weight" in lib.mok_last_error()

    w.ws_up = fake
    g = _lib.MokWeightGrads(d_w_gate=fake, d_w_up=fake, d_w_down=fake, d_ws_gate=fake, d_ws_up=odd, d_ws_down=fake)
    ctx = _lib.MokCtx(T=8, k=2, E=4, H=128, I=128, I_s=128, mode=0)

    def backward():
        return lib.mok_backward(C.byref(cfg), fake, fake, fake, C.byref(s), C.byref(ctx), C.byref(w), fake, fake,
                                C.byref(g), fake, 1 << 40, None)

    assert backward() == _lib.MOK_ERR_INVALID_ARG
    assert b"misaligned shared weight or grad" in lib.mok_last_error()
    g.d_ws_up = fake
    ctx.mode = 7                    # no forward records this mode
    assert backward() == _lib.MOK_ERR_INVALID_ARG
    assert b"context mode 7" in lib.mok_last_error()
    ctx.mode = 0
    w.E = 5                         # weights for another expert count than the schedule's
    assert backward() == _lib.MOK_ERR_INVALID_ARG
    assert b"weights have E=5" in lib.mok_last_error()
    w.E = 4
    ctx.I = 256                     # a context from another layer
    assert backward() == _lib.MOK_ERR_INVALID_ARG
    assert b"context does not match" in lib.mok_last_error()


def test_package_import_does_not_load_library():
    import subprocess
    import sys

    code = ("import sys; sys.path.insert(0, %r); import mixture_experts_layer_mok_gb300 as m; "
            "from mixture_experts_layer_mok_gb300 import _lib; print(_lib._lib is None)") % ROOT
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True)
    assert out.stdout.strip() == "True"


def test_autograd_layer_needs_cuda_tensors():
    """The autograd module is argument marshalling only: on CPU tensors it
    refuses (there is no CPU path) before touching the library."""
    import torch

    from mixture_experts_layer_mok_gb300.autograd import MoKLayer

    layer = MoKLayer(4, 128, 128, 0)
    assert tuple(layer.w_gate.shape) == (4, 128, 128) and tuple(layer.w_down.shape) == (4, 128, 128)
    assert layer.ws_gate is None
    x = torch.zeros(8, 128, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        layer(x, torch.full((8, 2), 0.5), torch.zeros(8, 2, dtype=torch.int64))


def test_schedule_and_context_flatten_over_a_moved_buffer():
    """flatten/unflatten carry the schedule and the context as (buffer,
    metadata): rebuilt over a copy of the buffer, every pointer keeps its
    offset, NULL stays NULL, and a pointer outside the buffer (the library's
    fixed scratch) keeps its address."""
    import torch

    import mixture_experts_layer_mok_gb300 as m
    from mixture_experts_layer_mok_gb300 import _lib

    buf = torch.zeros(4096, dtype=torch.uint8)
    base = buf.data_ptr()
    c = _lib.MokSchedule(T=8, k=2, E=4, max_tiles=3)
    c.cnt, c.row0, c.row_src, c.header = base + 0, base + 256, base + 512, base + 3840
    c.scratch = 0x7F0000001000                       # outside the buffer
    s = m.Schedule(8, 2, 4, buf, c)
    sbuf, meta = s.flatten()
    moved = sbuf.clone()
    s2 = m.Schedule.unflatten(moved, meta)
    nb = moved.data_ptr()
    assert (s2.T, s2.k, s2.E, s2.c.max_tiles) == (8, 2, 4, 3)
    assert (s2.c.cnt, s2.c.row0, s2.c.row_src, s2.c.header) == (nb, nb + 256, nb + 512, nb + 3840)
    assert s2.c.scratch == 0x7F0000001000 and not s2.c.slot_row
    cc = _lib.MokCtx(T=8, k=2, E=4, H=128, I=128, I_s=0, mode=2, max_tiles=3, dispatch=1, swiglu_limit=0.5)
    cc.gu, cc.status = base + 1024, base + 2048
    ctx = m.Context(buf, cc, 2)
    cbuf, cmeta = ctx.flatten()
    ctx2 = m.Context.unflatten(moved, cmeta)
    assert ctx2.mode == 2 and ctx2.c.mode == 2 and ctx2.c.dispatch == 1 and abs(ctx2.c.swiglu_limit - 0.5) < 1e-7
    assert (ctx2.c.gu, ctx2.c.status) == (nb + 1024, nb + 2048) and not ctx2.c.h
    with pytest.raises(ValueError):
        m.Schedule.unflatten(moved[:100], meta)      # offsets past a too-small buffer


def test_ctypes_structs_match_the_c_header(tmp_path):
    """The binding's ctypes structs against the C header itself: a C99 program
    built from include/mok.h prints each struct's size and every field's
    offset, and the ctypes view must agree field by field."""
    import shutil
    import subprocess

    from mixture_experts_layer_mok_gb300 import _lib

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pairs = [("mok_config_t", _lib.MokConfig), ("mok_schedule_t", _lib.MokSchedule),
             ("mok_weights_t", _lib.MokWeights), ("mok_ctx_t", _lib.MokCtx),
             ("mok_weight_grads_t", _lib.MokWeightGrads)]
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "mok.h"', "int main(void) {"]
    for cname, cls in pairs:
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {(a, b): int(c) for a, b, c in (ln.split() for ln in out if ln)}
    for cname, cls in pairs:
        assert got[(cname, "sizeof")] == C.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert got[(cname, field)] == getattr(cls, field).offset, (cname, field)


def test_schedule_calls_take_the_multiplier_as_double(tmp_path):
    """The two schedule builds take capacity_multiplier as a C double (so c*T
    is rounded up on exactly the caller's value), and the binding passes one:
    a C99 translation unit assigns each declaration to a pointer of the
    expected type, which -Werror turns into an error on any mismatch."""
    import shutil
    import subprocess

    from mixture_experts_layer_mok_gb300 import _lib

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "sig.c"
    src.write_text("\n".join([
        '#include "mok.h"',
        "typedef mok_status_t (*sched_fn)(const int64_t*, int, int, int, double, void*, size_t,",
        "                                 mok_schedule_t*, void*);",
        "sched_fn a = mok_schedule;",
        "sched_fn b = mok_schedule_noalloc;",
        "int main(void) { return a == b; }", ""]))
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                    str(tmp_path / "sig.o")], check=True, capture_output=True)
    for name in ("mok_schedule", "mok_schedule_noalloc"):
        assert _lib.SIGNATURES[name][1][4] is C.c_double, name


def _plan(lib, cnt, mb):
    import ctypes as C

    E = len(cnt)
    first = (C.c_int32 * (E + 1))()
    nw = C.c_int()
    rc = lib.mok_macrobatch_plan((C.c_int32 * E)(*cnt), E, mb, first, C.byref(nw))
    return rc, [first[i] for i in range(nw.value + 1)] if rc == 0 else None


def test_macrobatch_plan_is_the_greedy_split_of_whole_experts(lib):
    """The windows of a ring of mb rows: consecutive runs of whole experts
    covering 0..E in order, each run's 128-padded rows within the ring, and
    each run maximal (the next expert would not fit); an expert that alone
    exceeds the ring is MOK_ERR_CAPACITY.  Together these fix the split."""
    rng = np.random.default_rng(0)
    for trial in range(300):
        E = int(rng.integers(1, 40))
        cnt = rng.integers(0, 700, E) * (rng.random(E) < 0.8)
        mb = int(rng.integers(1, 3000))
        ring = -(-mb // 128) * 128
        padded = -(-cnt // 128) * 128
        rc, first = _plan(lib, [int(c) for c in cnt], mb)
        if padded.max() > ring:
            assert rc == 3, (cnt, mb)
            continue
        assert rc == 0
        assert first[0] == 0 and first[-1] == E and all(a < b for a, b in zip(first, first[1:]))
        for w in range(len(first) - 1):
            rows = padded[first[w]:first[w + 1]].sum()
            assert rows <= ring
            if first[w + 1] < E:
                assert rows + padded[first[w + 1]] > ring
    # no ring: one window; a ring that holds everything: one window
    assert _plan(lib, [5, 0, 300], 0)[1] == [0, 3]
    assert _plan(lib, [5, 0, 300], 10 ** 9)[1] == [0, 3]
    # one tile per window: every expert with rows starts a window, empty
    # experts ride along
    assert _plan(lib, [0, 3, 0, 128, 1, 0], 1)[1] == [0, 3, 4, 6]
    assert _plan(lib, [129], 128)[0] == 3
    assert _plan(lib, [-1], 128)[0] == 1
    assert _plan(lib, [1], -1)[0] == 1


def test_ring_buffer_sizes(lib):
    """The schedule-order scratch shrinks with the ring; 0, or a ring that holds
    every row, is the one-pass size; what stays full size (the saved gate|up
    rows, the slots, the router-weight partials) bounds it from below."""
    T, k, E, H, I, Is = 4096, 8, 64, 2048, 1024, 2048
    mt = (T * k + 127 * E) // 128
    for mode in (0, 1, 2):
        dims = (T, k, E, H, I, Is, mode)
        c0, w0 = lib.mok_ctx_bytes(*dims), lib.mok_bwd_workspace_bytes(*dims)
        assert lib.mok_ctx_bytes_ring(*dims, 0) == c0 and lib.mok_bwd_workspace_bytes_ring(*dims, 0) == w0
        assert lib.mok_ctx_bytes_ring(*dims, mt * 128) == c0
        assert lib.mok_bwd_workspace_bytes_ring(*dims, mt * 128 + 5) == w0
        prev = None
        for mb in (128, 1024, 4096, 16384):
            c, w = lib.mok_ctx_bytes_ring(*dims, mb), lib.mok_bwd_workspace_bytes_ring(*dims, mb)
            assert c < c0 and (w < w0 or mode == 1 and mb >= 16384)
            assert c >= 2 * mt * 128 * (2 * I + H)      # gate|up and the slots stay full size
            if prev:
                assert c >= prev[0] and w >= prev[1]
            prev = (c, w)
        assert lib.mok_ctx_bytes_ring(*dims, -1) == 0 and lib.mok_bwd_workspace_bytes_ring(*dims, -1) == 0

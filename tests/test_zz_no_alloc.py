"""The schedule entry point that allocates nothing (mok_schedule_noalloc).

Some callers cannot allocate device memory: code that runs inside another
framework's fixed memory pool, or a loop that must not call cudaMalloc
because it can synchronise the device.  For them the library takes the
schedule build's scratch from its own fixed device array.  This file checks,
through the C ABI, that the result matches mok_schedule() bit for bit on two
calls in a row, over scratch that earlier calls left behind, and that sizes
beyond the array's limit are refused.  It sits last in collection order
so a stop-at-first-failure run has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import mok

pytestmark = pytest.mark.gpu

ARRAYS = ("cnt", "row0", "row_src", "slot_row", "tile_expert", "tile_row0", "tile_rows", "header", "pair_tile",
          "unit_group")


def _views(sc, buf, T, k, E):
    base = buf.data_ptr()
    mt = sc.max_tiles
    sizes = {"cnt": E, "row0": E + 1, "row_src": mt * 128, "slot_row": T * k, "tile_expert": mt,
             "tile_row0": mt, "tile_rows": mt, "header": 8, "pair_tile": 2 * mt, "unit_group": 2 * mt}
    out = {}
    for name in ARRAYS:
        off = getattr(sc, name) - base
        out[name] = buf[off: off + 4 * sizes[name]].view(torch.int32).cpu().numpy().copy()
    return out


def _build(fn_name, te, E, c):
    m = mok()
    from mixture_experts_layer_mok_gb300 import _lib

    lib = _lib.load()
    T, k = te.shape
    nbytes = lib.mok_schedule_bytes(T, k, E)
    buf = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")   # poisoned output buffer
    sc = _lib.MokSchedule()
    st = getattr(lib, fn_name)(C.c_void_p(te.data_ptr()), T, k, E, float(c), C.c_void_p(buf.data_ptr()), nbytes,
                               C.byref(sc), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(st, fn_name)
    torch.cuda.synchronize()
    del m
    return _views(sc, buf, T, k, E)


def test_noalloc_schedule_matches_mok_schedule_on_two_calls_in_a_row():
    """Each case builds the schedule with mok_schedule(), then twice in a row
    with mok_schedule_noalloc(); both must match bit for bit.  The first case
    has the largest histogram footprint (128 chunks x 128 experts), so every
    later build runs over entries an earlier call left behind, and the last
    case repeats that footprint with other routing."""
    cases = [(16384, 8, 128, 1.2, 0.5, 2), (4096, 8, 64, None, 0.5, 1), (2560, 8, 16, 1.2, 0.05, 3),
             (16384, 8, 128, 1.2, 1.0, 4)]
    for T, k, E, skew, c, seed in cases:
        te = gen.make_routing(T, k, E, seed=seed, skew=skew).cuda()
        ref = _build("mok_schedule", te, E, c)
        for call in range(2):
            got = _build("mok_schedule_noalloc", te, E, c)
            for name in ARRAYS:
                assert np.array_equal(got[name], ref[name]), (T, E, call, name)
            assert got["header"][2] == 0


def test_noalloc_schedule_rejects_sizes_beyond_its_scratch():
    m = mok()
    from mixture_experts_layer_mok_gb300 import _lib

    lib = _lib.load()
    T, k, E = 300000, 8, 1024            # ceil(T*k/1024) * E = 2344 * 1024 > 1048576
    sc = _lib.MokSchedule()
    fake = C.c_void_p(256)               # never touched: the size check comes first
    st = lib.mok_schedule_noalloc(fake, T, k, E, 0.5, fake, 1 << 30, C.byref(sc), None)
    assert st == _lib.MOK_ERR_INVALID_ARG
    assert b"fixed scratch" in lib.mok_last_error()
    del m

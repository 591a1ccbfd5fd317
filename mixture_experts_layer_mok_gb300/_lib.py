"""ctypes view of libmok's C ABI (include/mok.h).  Loading fails loudly when the
library has not been built; nothing here computes any part of the layer."""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmok.so")

MOK_OK = 0
MOK_ERR_INVALID_ARG = 1
MOK_ERR_INDEX = 2
MOK_ERR_CAPACITY = 3
MOK_ERR_UNSUPPORTED = 4
MOK_ERR_TIMEOUT = 5
MOK_ERR_CUDA = 6
MOK_MODE_BF16 = 0
MOK_MODE_MXFP8_FWD = 1
MOK_MODE_MXFP8 = 2
MOK_DEBUG_DROP_ACC_SIGNAL = 1
MOK_DEBUG_TMA_GATHER4 = 2
MOK_DEBUG_STATIC_ORDER = 64
MOK_DEBUG_TICKET_ORDER = 128
MOK_DISPATCH_AUTO = 0
MOK_DISPATCH_PERMUTE = 1
MOK_DISPATCH_FUSED = 2
DISPATCH = {"auto": 0, "permute": 1, "fused": 2}

STATUS_NAMES = {0: "MOK_OK", 1: "MOK_ERR_INVALID_ARG", 2: "MOK_ERR_INDEX", 3: "MOK_ERR_CAPACITY",
                4: "MOK_ERR_UNSUPPORTED", 5: "MOK_ERR_TIMEOUT", 6: "MOK_ERR_CUDA"}

P = C.c_void_p
I32P = C.POINTER(C.c_int32)


MOK_NUM_STAGES = 17
STAGE_NAMES = ["fwd_prep", "fwd_shared_gateup", "fwd_shared_down", "fwd_gateup", "fwd_down", "fwd_combine",
               "bwd_down", "bwd_wgrad_down", "bwd_wgrad_gateup", "bwd_dgrad_gateup", "bwd_shared_down",
               "bwd_shared_wgrad_down", "bwd_shared_wgrad_gateup", "bwd_shared_dgrad", "bwd_reduce",
               "fwd_dispatch", "bwd_dispatch"]


class MokConfig(C.Structure):
    _fields_ = [("mode", C.c_int), ("minibatch_size", C.c_int), ("debug_flags", C.c_int),
                ("dispatch", C.c_int), ("num_events", C.c_int), ("events", C.POINTER(C.c_void_p)),
                ("swiglu_limit", C.c_float), ("macrobatch_size", C.c_int64)]


class MokSchedule(C.Structure):
    _fields_ = [("T", C.c_int), ("k", C.c_int), ("E", C.c_int), ("max_tiles", C.c_int),
                ("cnt", P), ("row0", P), ("row_src", P), ("slot_row", P), ("tile_expert", P),
                ("tile_row0", P), ("tile_rows", P), ("header", P), ("scratch", P), ("pair_tile", P),
                ("unit_group", P)]


class MokWeights(C.Structure):
    _fields_ = [("E", C.c_int), ("H", C.c_int), ("I", C.c_int), ("I_s", C.c_int),
                ("w_gate", P), ("w_up", P), ("w_down", P), ("ws_gate", P), ("ws_up", P), ("ws_down", P),
                ("mx_gate", P), ("mx_gate_sc", P), ("mx_up", P), ("mx_up_sc", P),
                ("mx_down", P), ("mx_down_sc", P), ("mxs_gate", P), ("mxs_gate_sc", P),
                ("mxs_up", P), ("mxs_up_sc", P), ("mxs_down", P), ("mxs_down_sc", P),
                ("mxt_gate", P), ("mxt_gate_sc", P), ("mxt_up", P), ("mxt_up_sc", P),
                ("mxt_down", P), ("mxt_down_sc", P), ("mxts_gate", P), ("mxts_gate_sc", P),
                ("mxts_up", P), ("mxts_up_sc", P), ("mxts_down", P), ("mxts_down_sc", P)]


class MokCtx(C.Structure):
    _fields_ = [("T", C.c_int), ("k", C.c_int), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int),
                ("I_s", C.c_int), ("mode", C.c_int), ("max_tiles", C.c_int),
                ("gu", P), ("h", P), ("hq", P), ("hq_sc", P), ("slots", P), ("gu_s", P), ("h_s", P),
                ("hq_s", P), ("hq_s_sc", P), ("shared_out", P), ("xq", P), ("xq_sc", P), ("status", P),
                ("x_perm", P), ("dispatch", C.c_int), ("xq_perm", P), ("xq_perm_sc", P),
                ("swiglu_limit", C.c_float), ("ring_rows", C.c_int64)]


class MokWeightGrads(C.Structure):
    _fields_ = [("d_w_gate", P), ("d_w_up", P), ("d_w_down", P), ("d_ws_gate", P), ("d_ws_up", P),
                ("d_ws_down", P)]


# name -> (restype, argtypes); every symbol include/mok.h declares
SIGNATURES = {
    "mok_version": (C.c_int, []),
    "mok_last_error": (C.c_char_p, []),
    "mok_schedule_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "mok_schedule": (C.c_int, [P, C.c_int, C.c_int, C.c_int, C.c_double, P, C.c_size_t,
                               C.POINTER(MokSchedule), P]),
    "mok_schedule_status": (C.c_int, [C.POINTER(MokSchedule), I32P, I32P, I32P]),
    "mok_schedule_noalloc": (C.c_int, [P, C.c_int, C.c_int, C.c_int, C.c_double, P, C.c_size_t,
                                       C.POINTER(MokSchedule), P]),
    "mok_mxfp8_quantize": (C.c_int, [P, C.c_int64, C.c_int, P, P, P]),
    "mok_mxfp8_quantize_t": (C.c_int, [P, C.c_int64, C.c_int, C.c_int, P, P, P]),
    "mok_mxfp8_quantize_dual": (C.c_int, [P, C.c_int64, C.c_int, C.c_int, P, P, P, P, P]),
    "mok_ctx_bytes": (C.c_size_t, [C.c_int] * 7),
    "mok_ctx_bytes_ring": (C.c_size_t, [C.c_int] * 7 + [C.c_int64]),
    "mok_forward": (C.c_int, [C.POINTER(MokConfig), P, P, C.POINTER(MokSchedule),
                              C.POINTER(MokWeights), P, P, C.c_size_t, C.POINTER(MokCtx), P]),
    "mok_ctx_status": (C.c_int, [C.POINTER(MokCtx), I32P]),
    "mok_bwd_workspace_bytes": (C.c_size_t, [C.c_int] * 7),
    "mok_bwd_workspace_bytes_ring": (C.c_size_t, [C.c_int] * 7 + [C.c_int64]),
    "mok_macrobatch_plan": (C.c_int, [I32P, C.c_int, C.c_int64, I32P, C.POINTER(C.c_int)]),
    "mok_backward": (C.c_int, [C.POINTER(MokConfig), P, P, P, C.POINTER(MokSchedule), C.POINTER(MokCtx),
                               C.POINTER(MokWeights), P, P, C.POINTER(MokWeightGrads), P, C.c_size_t, P]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libmok.so (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libmok.so not found at {path}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MokError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().mok_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != MOK_OK:
        raise MokError(code, where)

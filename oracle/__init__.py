"""Test infrastructure: the CPU oracle for the MoK layer.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never does.
"""
from .mok_oracle import (  # noqa: F401
    TILE_ROWS,
    max_tiles,
    capacity_tiles,
    STATUS_OK,
    STATUS_INDEX,
    mxfp8_roundtrip,
    mxfp8_roundtrip_cols,
    build_schedule,
    e4m3_decode,
    e4m3_encode,
    e8m0_scale_exponent,
    mxfp8_quantize,
    mxfp8_dequantize,
    silu,
    round_bf16,
    clamp_gate_up,
    layer_forward,
    layer_backward,
    layer_forward_mxfp8,
    layer_backward_mxfp8,
    layer_backward_mxfp8_full,
)

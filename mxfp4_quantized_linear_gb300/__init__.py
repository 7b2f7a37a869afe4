"""MX (MXFP8 / MXFP4) quantized linear for one GB300 (sm_103a).

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/mx.h``); this package only marshals arguments to it.
"""
from .binding import (  # noqa: F401
    MX_FMT_E2M1, MX_FMT_E4M3, MX_LAYOUT_GATE_UP, MX_LAYOUT_PLAIN, MX_LINEAR_CLUSTER_GEMV, MX_LINEAR_NO_FUSED_QUANT,
    MX_PACK_FOLD, MX_PACK_GATE_UP, MX_PACK_REQUIRE_BLOCK, MX_SCALE_BLOCK32X32, MX_SCALE_ROW1X32, MxError,
    PackedWeight, load_library, mx_check_device_errors, mx_dequant, mx_e4m3_from_dequant, mx_measure_mxf8_peak, mx_pack_size,
    mx_pack_weights, mx_quantize_act, mx_route_experts, mxfp4_moe_expert, mxfp4_moe_expert_workspace_size,
    mxfp4_moe_linear, mxfp4_moe_linear_w4a8, mxfp4_moe_workspace_size, mxfp8_linear, mxfp8_linear_noalloc, mxfp8_linear_q,
    mxfp8_linear_workspace_size)

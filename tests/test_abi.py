"""The C ABI library builds, loads, and exports every entry point include/mx.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from tests.helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(mx\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mx_quantize_act", "mx_dequant", "mxfp8_linear", "mxfp4_moe_linear", "mx_pack_weights"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ensure_built()
    from mxfp4_quantized_linear_gb300 import binding
    names = declared_functions()
    assert set(binding.EXPORTED) == set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_host_side_argument_checks_without_gpu():
    lib = ensure_built()
    from mxfp4_quantized_linear_gb300 import binding as b
    assert lib.mx_pack_size(b.MX_FMT_E4M3, 1, 7168, 2080) == 256 + 7168 * 2176 + 7168 * 68 + 56 * 17 * 512
    assert lib.mx_pack_size(b.MX_FMT_E4M3, 1, 64, 33) == 0
    assert lib.mx_pack_size(7, 1, 64, 64) == 0
    assert lib.mx_quantize_act(None, 4, 33, None, None, None) == b.MX_ERR_SHAPE
    assert b"multiple of 32" in lib.mx_last_error()
    assert lib.mx_quantize_act(None, 0, 64, None, None, None) == b.MX_OK     # M == 0: no-op
    assert lib.mx_quantize_act(None, 2, 64, None, None, None) == b.MX_ERR_ARG
    assert lib.mx_dequant(None, None, 9, 0, 32, 64, None, None) == b.MX_ERR_ARG
    assert lib.mx_dequant(None, None, 0, 0, 33, 64, None, None) == b.MX_ERR_SHAPE
    assert lib.mx_route_experts(None, 4, 2, 4096, None, None, None, None, None, None, None) == b.MX_ERR_UNSUPPORTED
    assert lib.mxfp8_linear(None, 1, None, None, None, 0, None, 0, None) == b.MX_ERR_ARG
    w = b.MxPackedWeightC(fmt=b.MX_FMT_E2M1, E=1, N=64, K=64, Kp=128)
    assert lib.mxfp8_linear(None, 1, ctypes.byref(w), None, None, 0, None, 0, None) == b.MX_ERR_ARG
    bad = ctypes.c_void_p(0x1001)  # misaligned (never dereferenced: rejected first)
    assert lib.mx_quantize_act(bad, 2, 64, bad, bad, None) == b.MX_ERR_ALIGN
    assert lib.mxfp4_moe_workspace_size(4, 2, 8, 128, 256) > 0


def test_product_path_fails_loudly_without_library(tmp_path):
    from mxfp4_quantized_linear_gb300 import binding
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library(str(tmp_path / "missing.so"))


def test_host_side_checks_of_the_newer_entry_points():
    """mxfp8_linear_q, mxfp4_moe_expert, mx_e4m3_from_dequant and the gate/up pack
    flag reject bad arguments before any device work."""
    lib = ensure_built()
    from mxfp4_quantized_linear_gb300 import binding as b
    e4 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=64, K=64, Kp=128)
    e2 = b.MxPackedWeightC(fmt=b.MX_FMT_E2M1, E=2, N=64, K=256, Kp=256, layout=b.MX_LAYOUT_GATE_UP)
    e2p = b.MxPackedWeightC(fmt=b.MX_FMT_E2M1, E=2, N=256, K=32, Kp=128, layout=b.MX_LAYOUT_PLAIN)
    # pre-quantized linear
    assert lib.mxfp8_linear_q(None, None, 1, ctypes.byref(e2p), None, None, 0, None, 0, None) == b.MX_ERR_ARG
    assert lib.mxfp8_linear_q(None, None, 1, ctypes.byref(e4), None, None, 8, None, 0, None) == b.MX_ERR_ARG
    assert lib.mxfp8_linear_q(None, None, 0, ctypes.byref(e4), None, None, 0, None, 0, None) == b.MX_OK
    assert lib.mxfp8_linear_q_workspace_size(32, ctypes.byref(e4)) == 0
    assert lib.mxfp8_linear_q_workspace_size(33, ctypes.byref(e4)) == 512
    # the GEMM's K split on a host without a device is sized for 152 SMs:
    # N=7168 K=8192 M=64 is 28 tiles of 128 x 256 -> 5 K ranges of f32 sums
    # [5, 64, 7168]; N=24576 K=1536 is 96 tiles -> no split
    w1 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=7168, K=8192, Kp=8192)
    base = 128 * 8192 + 128 * 256
    assert lib.mxfp8_linear_workspace_size(64, ctypes.byref(w1)) == base + 5 * 64 * 7168 * 4
    assert lib.mxfp8_linear_q_workspace_size(64, ctypes.byref(w1)) == 64 * 512 + 5 * 64 * 7168 * 4
    w2 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=24576, K=1536, Kp=1536)
    assert lib.mxfp8_linear_workspace_size(64, ctypes.byref(w2)) == 128 * 1536 + 128 * 48

    def split_room(M, w):
        """bytes past the required quantized activation and codes"""
        Mp = -(-M // 128) * 128
        need = -(-Mp * w.Kp // 256) * 256 + -(-Mp * (w.Kp // 32) // 256) * 256
        return lib.mxfp8_linear_workspace_size(M, ctypes.byref(w)) - need

    # 152 SMs: S = min(8, SMs / tiles, K steps / 4), ranges [S, M, N] f32
    assert split_room(33, w1) == 5 * 33 * 7168 * 4      # 28 tiles
    assert split_room(256, w1) == 2 * 256 * 7168 * 4    # 56 tiles
    assert split_room(384, w1) == 0                     # 84 tiles > 152 / 2
    w5 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=320, K=4160, Kp=4224)
    assert split_room(1000, w5) == 8 * 1000 * 320 * 4   # 16 tiles, 33 K steps
    w6 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=192, K=512, Kp=512)
    assert split_room(130, w6) == 0                     # 4 K steps: ranges would be shorter than 4
    w7 = b.MxPackedWeightC(fmt=b.MX_FMT_E4M3, E=1, N=7168, K=65536, Kp=65536)
    assert split_room(256, w7) == 2 * 256 * 7168 * 4    # 14.7 MB a range: under the 64 MB cap
    assert split_room(64 * 128, w7) == 0                # 1792 tiles
    # expert: w13 must carry the gate/up layout, w2 must fit it
    assert lib.mxfp4_moe_expert(None, None, None, 1, 1, ctypes.byref(e2p), ctypes.byref(e2p), None, None, 0, None,
                                None) == b.MX_ERR_ARG
    assert lib.mxfp4_moe_expert(None, None, None, 1, 1, ctypes.byref(e2), ctypes.byref(e2), None, None, 0, None,
                                None) == b.MX_ERR_ARG                  # w2 packed with the interleave
    assert lib.mxfp4_moe_expert(None, None, None, 1, 1, ctypes.byref(e2), ctypes.byref(e2p), None, None, 0, None,
                                None) == b.MX_ERR_ARG                  # shapes fit (I = 32 = w2 K): NULL x
    w2_bad = b.MxPackedWeightC(fmt=b.MX_FMT_E2M1, E=2, N=256, K=64, Kp=128, layout=b.MX_LAYOUT_PLAIN)
    assert lib.mxfp4_moe_expert(None, None, None, 1, 1, ctypes.byref(e2), ctypes.byref(w2_bad), None, None, 0, None,
                                None) == b.MX_ERR_SHAPE                # w2 K = 64 != I = 32
    assert b"does not fit" in lib.mx_last_error()
    assert lib.mxfp4_moe_expert_workspace_size(4, 2, 8, 128, 64, 128) > lib.mxfp4_moe_workspace_size(4, 2, 8, 128, 128)
    # from-dequant
    n = ctypes.c_int64(7)
    assert lib.mx_e4m3_from_dequant(None, None, 5, 32, 64, None, None, ctypes.byref(n), None) == b.MX_ERR_ARG
    assert n.value == 0
    assert lib.mx_e4m3_from_dequant(None, None, b.MX_SCALE_BLOCK32X32, 40, 64, None, None, None, None) == b.MX_ERR_SHAPE
    assert lib.mx_e4m3_from_dequant(None, None, b.MX_SCALE_ROW1X32, 0, 64, None, None, None, None) == b.MX_OK
    # gate/up flag only for E2M1 and 2 I a multiple of 16
    dst = b.MxPackedWeightC()
    buf = ctypes.c_void_p(0x100000)   # aligned, never dereferenced: rejected first
    assert lib.mx_pack_weights(buf, buf, b.MX_FMT_E4M3, 1, 64, 64, 64, b.MX_PACK_GATE_UP, buf, 1 << 20,
                               ctypes.byref(dst), None) == b.MX_ERR_ARG
    assert lib.mx_pack_weights(buf, buf, b.MX_FMT_E2M1, 1, 40, 64, 40, b.MX_PACK_GATE_UP, buf, 1 << 20,
                               ctypes.byref(dst), None) == b.MX_ERR_SHAPE

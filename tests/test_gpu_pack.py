"""K-PACK on the GPU against the oracle's layout maps, bit for bit."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import inputs
from oracle import layout as L
from tests.helpers import cuda_device, ensure_built, u8

pytestmark = pytest.mark.gpu


def gpu_pack(w, c, fmt, flags=mx.MX_PACK_FOLD):
    dev = cuda_device()
    ensure_built()
    return mx.mx_pack_weights(w.to(dev), c.to(dev), fmt, flags)


def check_e4m3(w, c, fold=True, require=False):
    flags = (mx.MX_PACK_FOLD if fold else 0) | (mx.MX_PACK_REQUIRE_BLOCK if require else 0)
    p = gpu_pack(w, c, "e4m3", flags)
    wn, cn = u8(w), u8(c)
    ref = L.pack_e4m3(wn[None] if wn.ndim == 2 else wn, cn[None] if cn.ndim == 2 else cn,
                      fold=fold, require_block=require)
    assert (p.scale_mode == mx.MX_SCALE_BLOCK32X32) == (ref["mode"] == "block")
    assert p.Kp == ref["Kp"]
    assert np.array_equal(u8(p.bytes_tensor()), ref["wq"])
    assert np.array_equal(u8(p.codes_tensor()), ref["codes"])
    assert np.array_equal(u8(p.sf_tensor()), ref["sf"])
    return p


def test_e4m3_block_codes_ragged_k():
    g = inputs.generator(1)
    check_e4m3(inputs.e4m3_bytes((96, 2080), g), inputs.e8m0_codes((3, 65), 118, 132, g))


def test_e4m3_row_codes_fold_and_keep():
    g = inputs.generator(2)
    w = inputs.e4m3_bytes((128, 256), g)
    block = inputs.e8m0_codes((4, 8), 118, 132, g)
    row = block.repeat_interleave(32, dim=0)
    assert check_e4m3(w, row).scale_mode == mx.MX_SCALE_BLOCK32X32
    assert check_e4m3(w, row, fold=False).scale_mode == mx.MX_SCALE_ROW1X32
    bad = row.clone()
    bad[70, 3] ^= 1
    assert check_e4m3(w, bad).scale_mode == mx.MX_SCALE_ROW1X32
    with pytest.raises(mx.MxError) as ei:
        gpu_pack(w, bad, "e4m3", mx.MX_PACK_REQUIRE_BLOCK)
    assert ei.value.code == L.MX_ERR_NOT_BLOCK32
    nan = row.clone()
    nan[5, 5] = 255
    with pytest.raises(mx.MxError) as ei:
        gpu_pack(w, nan, "e4m3")
    assert ei.value.code == L.MX_ERR_SCALE


def test_e4m3_row_codes_n_not_multiple_of_32():
    g = inputs.generator(3)
    check_e4m3(inputs.e4m3_bytes((40, 96), g), inputs.e8m0_codes((40, 3), 120, 130, g))


def test_e4m3_decode_linear_full_size():
    c = inputs.decode_linear(K=2048, Ms=())
    check_e4m3(c["w"], c["codes"])


def check_e2m1(w, c, experts=None):
    p = gpu_pack(w, c, "e2m1")
    wn, cn = u8(w), u8(c)
    sel = slice(None) if experts is None else experts
    ref = L.pack_e2m1(wn[sel], cn[sel])
    assert p.Kp == ref["Kp"] and p.scale_mode == mx.MX_SCALE_ROW1X32
    assert np.array_equal(u8(p.bytes_tensor())[sel], ref["wq"])
    assert np.array_equal(u8(p.codes_tensor())[sel], ref["codes"])
    assert np.array_equal(u8(p.sf_tensor())[sel], ref["sf"])
    if experts is None:
        assert p.neg_zero_count == ref["neg_zero_count"]
    else:
        assert p.neg_zero_count == L.count_negative_zero(wn)
    return p


def test_e2m1_ragged_and_negative_zero():
    g = inputs.generator(4)
    check_e2m1(inputs.fp4x2_bytes((3, 48, 1040), g), inputs.e8m0_codes((3, 48, 65), 122, 130, g))


def test_e2m1_block_codes_expand():
    g = inputs.generator(5)
    w = inputs.fp4x2_bytes((2, 64, 64), g)
    cb = inputs.e8m0_codes((2, 2, 4), 122, 130, g)
    p = gpu_pack(w, cb, "e2m1")
    ref = L.pack_e2m1(u8(w), u8(cb))
    assert np.array_equal(u8(p.codes_tensor()), ref["codes"])


def test_e2m1_moe_full_size_sampled_experts():
    m = inputs.moe_gate_up(T=1)
    check_e2m1(m["w"], m["codes"], experts=[0, 17, 63])


def test_e2m1_gate_up_interleave():
    g = inputs.generator(6)
    w = inputs.fp4x2_bytes((3, 96, 1040), g)          # 2 I = 96, ragged K = 2080
    c = inputs.e8m0_codes((3, 96, 65), 122, 130, g)
    p = gpu_pack(w, c, "e2m1", mx.MX_PACK_GATE_UP)
    ref = L.pack_e2m1(u8(w), u8(c), gate_up=True)
    assert p.desc.layout == mx.MX_LAYOUT_GATE_UP
    assert np.array_equal(u8(p.bytes_tensor()), ref["wq"])
    assert np.array_equal(u8(p.codes_tensor()), ref["codes"])
    assert np.array_equal(u8(p.sf_tensor()), ref["sf"])
    assert p.neg_zero_count == ref["neg_zero_count"]
    plain = gpu_pack(w, c, "e2m1", 0)
    assert plain.desc.layout == mx.MX_LAYOUT_PLAIN


def test_gate_up_flag_refusals():
    g = inputs.generator(7)
    w = inputs.fp4x2_bytes((1, 40, 64), g)
    c = inputs.e8m0_codes((1, 40, 4), 122, 130, g)
    with pytest.raises(mx.MxError):
        gpu_pack(w, c, "e2m1", mx.MX_PACK_GATE_UP)           # 2 I = 40 is not a multiple of 16
    with pytest.raises(mx.MxError):
        gpu_pack(inputs.e4m3_bytes((64, 128), g), inputs.e8m0_codes((2, 4), 120, 130, g), "e4m3",
                 mx.MX_PACK_GATE_UP)                          # E4M3 weights have no gate / up form

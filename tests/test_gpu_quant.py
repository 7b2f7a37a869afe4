"""K-QUANT and K-DEQ on the GPU against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import inputs
from oracle import formats as F
from oracle.linear import dequant_bf16
from oracle.quant import quantize_act
from tests.helpers import bf16_np, cuda_device, ensure_built, u8
from tests.test_oracle_quant import load_golden

pytestmark = pytest.mark.gpu


def gpu_quant(x):
    dev = cuda_device()
    ensure_built()
    q, c = mx.mx_quantize_act(x.to(dev))
    torch.cuda.synchronize()
    return u8(q), u8(c)


def check_quant(x):
    q, c = gpu_quant(x)
    rq, rc = quantize_act(bf16_np(x))
    assert np.array_equal(c, rc), np.argwhere(c != rc)[:5]
    assert np.array_equal(q, rq), np.argwhere(q != rq)[:5]


def test_golden_blocks():
    cases = load_golden()
    x = torch.tensor(np.stack([c[1] for c in cases]), dtype=torch.float32).to(torch.bfloat16)
    q, c = gpu_quant(x)
    for i, (name, _, code, b) in enumerate(cases):
        assert c[i, 0] == code, name
        assert np.array_equal(q[i], b), (name, [hex(v) for v in q[i]])


@pytest.mark.parametrize("M,K", [(1, 32), (5, 96), (37, 2080), (128, 7168)])
def test_random_normal(M, K):
    check_quant(inputs.bf16_normal((M, K), inputs.generator(M + K)))


def test_wide_dynamic_range_and_ties():
    rng = np.random.default_rng(11)
    n = 4096
    scale = np.exp2(rng.integers(-140, 120, size=(n, 1)).astype(np.float64))
    x = rng.standard_normal((n, 32)) * scale
    k = rng.integers(-120, 100, size=n)
    x[np.arange(n), rng.integers(0, 32, size=n)] = np.ldexp(448.0, k) * rng.choice([-1, 1], size=n)
    x[::7] = 0.0
    x[3::11, 5] = -0.0
    xb = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).reshape(-1, 128)
    check_quant(xb)


def test_nan_and_inf_blocks():
    x = inputs.bf16_normal((4, 128), inputs.generator(3))
    x[0, 5] = float("nan")
    x[1, 40] = float("inf")
    x[2, 127] = -float("inf")
    check_quant(x)


def test_full_size_prefill_rows_sampled():
    x = inputs.bf16_normal((4096, 7168), inputs.generator(0))
    q, c = gpu_quant(x)
    rows = np.random.default_rng(0).choice(4096, size=96, replace=False)
    rq, rc = quantize_act(bf16_np(x[rows]))
    assert np.array_equal(c[rows], rc) and np.array_equal(q[rows], rq)
    # invariants on every row: |q| <= 448, tight scale
    v = F.e4m3_decode(q.reshape(4096, -1, 32))
    assert np.nanmax(np.abs(v)) <= 448
    assert np.all(np.max(np.abs(v), axis=2)[c > 0] >= 224)


def gpu_dequant(b, c, fmt, mode):
    dev = cuda_device()
    ensure_built()
    out = mx.mx_dequant(b.to(dev), c.to(dev), fmt, mode)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def compare_bf16_bits(got, ref):
    nan_g = np.isnan(F.bf16_value(got))
    nan_r = np.isnan(F.bf16_value(ref))
    assert np.array_equal(nan_g, nan_r)
    assert np.array_equal(got[~nan_g], ref[~nan_r])


def test_dequant_e4m3_every_byte_and_code():
    codes_list = [0, 1, 2, 3, 100, 118, 120, 127, 132, 200, 246, 250, 253, 254, 255]
    b = np.tile(np.arange(256, dtype=np.uint8), (len(codes_list), 1))   # [15, 256]
    c = np.repeat(np.array(codes_list, dtype=np.uint8)[:, None], 8, axis=1)
    got = gpu_dequant(torch.tensor(b), torch.tensor(c), "e4m3", mx.MX_SCALE_ROW1X32)
    compare_bf16_bits(got, dequant_bf16(b, c, "e4m3", len(codes_list), 256))


def test_dequant_e4m3_block_codes():
    g = inputs.generator(5)
    b = inputs.e4m3_bytes((64, 2080), g)
    c = inputs.e8m0_codes((2, 65), 118, 132, g)
    got = gpu_dequant(b, c, "e4m3", mx.MX_SCALE_BLOCK32X32)
    compare_bf16_bits(got, dequant_bf16(u8(b), u8(c), "e4m3", 64, 2080))


def test_dequant_e2m1_every_nibble_and_code():
    codes_list = [0, 1, 120, 127, 130, 200, 252, 254, 255]
    b = np.tile(np.arange(256, dtype=np.uint8), (len(codes_list), 1))   # [9, 256] bytes = K 512
    c = np.repeat(np.array(codes_list, dtype=np.uint8)[:, None], 16, axis=1)
    got = gpu_dequant(torch.tensor(b), torch.tensor(c), "e2m1", mx.MX_SCALE_ROW1X32)
    compare_bf16_bits(got, dequant_bf16(b, c, "e2m1", len(codes_list), 512))


# ------------------------------------------------ e4m3 bytes from a bf16 dequant

def _bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.tensor(bits.astype(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("codes_lohi", [(118, 132), (3, 40), (200, 246)])
def test_from_dequant_recovers_the_bytes(codes_lohi):
    """weights942 ocp_from_dequant on the GPU: the bf16 dequant of random bytes
    (the oracle's bits) gives every byte back, block and row codes alike."""
    from oracle.linear import e4m3_from_dequant
    dev = cuda_device()
    ensure_built()
    g = inputs.generator(codes_lohi[0])
    b = inputs.e4m3_bytes((96, 2080), g)
    cb = inputs.e8m0_codes((3, 65), *codes_lohi, g)
    w = _bf16_tensor(dequant_bf16(u8(b), u8(cb), "e4m3", 96, 2080)).to(dev)
    q = mx.mx_e4m3_from_dequant(w, cb.to(dev), mx.MX_SCALE_BLOCK32X32)
    torch.cuda.synchronize()
    assert np.array_equal(u8(q), u8(b))
    cr = inputs.e8m0_codes((96, 65), *codes_lohi, g)
    w = _bf16_tensor(dequant_bf16(u8(b), u8(cr), "e4m3", 96, 2080))
    q = mx.mx_e4m3_from_dequant(w.to(dev), cr.to(dev), mx.MX_SCALE_ROW1X32)
    assert np.array_equal(u8(q), u8(b))
    assert e4m3_from_dequant(bf16_np(w), u8(cr))[1] == 0


def test_from_dequant_refusals_count_like_the_oracle():
    from oracle.linear import e4m3_from_dequant
    dev = cuda_device()
    ensure_built()
    g = inputs.generator(12)
    b = inputs.e4m3_bytes((64, 256), g)
    cb = inputs.e8m0_codes((2, 8), 118, 132, g)
    bits = dequant_bf16(u8(b), u8(cb), "e4m3", 64, 256).copy()
    rng = np.random.default_rng(0)
    idx = rng.choice(bits.size, size=37, replace=False)
    flat = bits.reshape(-1)
    flat[idx[:30]] ^= 0x0001                 # one bf16 ulp away (off the e4m3 grid, or +-0 -> subnormal)
    flat[idx[30:33]] = 0x7FC0                # NaN
    flat[idx[33:35]] = 0x7F80                # inf
    flat[idx[35:]] = 0x7F00                  # 2^127: far beyond 448 x the block scale
    w = _bf16_tensor(bits)
    with pytest.raises(mx.MxError) as ei:
        mx.mx_e4m3_from_dequant(w.to(dev), cb.to(dev))
    assert ei.value.code == mx.binding.MX_ERR_INEXACT
    _, bad = mx.mx_e4m3_from_dequant(w.to(dev), cb.to(dev), strict=False)
    assert bad == e4m3_from_dequant(bf16_np(w), u8(cb))[1]


def test_large_activation_every_element():
    """A large activation (4.3 M elements, an odd row count, several rounds
    of the grid-stride loop): every byte and code against the oracle, with
    NaN / inf / all-zero blocks."""
    x = inputs.bf16_normal((1031, 4128), inputs.generator(5))
    x[3, 40] = float("nan")
    x[500, 4127] = float("inf")
    x[1030, :64] = 0.0
    check_quant(x)

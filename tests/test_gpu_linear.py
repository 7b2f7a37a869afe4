"""mxfp8_linear (quantize + split-K GEMV / large-M path) on the GPU against the
oracle: normalised max error <= 1e-2 (see tests/helpers.TOL), plus bitwise
batch invariance and fused / unfused agreement."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import inputs
from oracle.linear import mxfp8_linear as ref_linear, normalized_error
from tests.helpers import TOL, bf16_np, cuda_device, elementwise_excess, ensure_built, u8

pytestmark = pytest.mark.gpu


def pack(w, c, flags=mx.MX_PACK_FOLD):
    dev = cuda_device()
    ensure_built()
    return mx.mx_pack_weights(w.to(dev), c.to(dev), "e4m3", flags)


def gpu_linear(p, x, bias=None, flags=0):
    dev = cuda_device()
    y = mx.mxfp8_linear(x.to(dev), p, None if bias is None else bias.to(dev), flags=flags)
    torch.cuda.synchronize()
    return y


def row_codes(codes: np.ndarray, N: int) -> np.ndarray:
    return np.repeat(codes, 32, axis=0)[:N] if codes.shape[0] != N else codes


def check(p, w, c, x, bias=None, rows=None, flags=0, tol=TOL):
    y = gpu_linear(p, x, bias, flags).float().cpu().numpy()
    wn, cn = u8(w), row_codes(u8(c), w.shape[0])
    if rows is not None:
        wn, cn, y = wn[rows], cn[rows], y[:, rows]
    ref = ref_linear(bf16_np(x), wn, cn, None if bias is None else bf16_np(bias)[rows if rows is not None else slice(None)])
    err = normalized_error(y, ref["y"], ref["A"], ref["B"])
    assert err <= tol, err
    excess = elementwise_excess(y, ref)
    assert excess <= 0.0, excess
    return err


def test_gemv_small_m1_row_codes():
    c = inputs.gemv_small()
    p = pack(c["w"], c["codes"])
    assert p.scale_mode == mx.MX_SCALE_ROW1X32
    for M in (1, 2, 4):
        check(p, c["w"], c["codes"], inputs.bf16_normal((M, c["K"]), inputs.generator(M)))


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 32])
def test_ragged_rows_and_k(M):
    g = inputs.generator(100 + M)
    w = inputs.e4m3_bytes((96, 2080), g)
    c = inputs.e8m0_codes((3, 65), 118, 132, g)
    check(pack(w, c), w, c, inputs.bf16_normal((M, 2080), g))


def test_row_mode_small_n_short_k_with_bias():
    g = inputs.generator(7)
    w = inputs.e4m3_bytes((40, 96), g)
    c = inputs.e8m0_codes((40, 3), 120, 130, g)
    b = inputs.bf16_normal((40,), g)
    p = pack(w, c)
    for M in (1, 5, 12):
        check(p, w, c, inputs.bf16_normal((M, 96), g), bias=b)


@pytest.mark.parametrize("K", [2048, 2080])
def test_decode_linear_full_size(K):
    c = inputs.decode_linear(K=K)
    p = pack(c["w"], c["codes"])
    assert p.scale_mode == mx.MX_SCALE_BLOCK32X32
    for M, x in c["xs"].items():
        check(p, c["w"], c["codes"], x)


def test_large_m_path():
    g = inputs.generator(9)
    w = inputs.e4m3_bytes((192, 512), g)
    c = inputs.e8m0_codes((6, 16), 118, 132, g)
    p = pack(w, c)
    for M in (33, 64, 130):
        check(p, w, c, inputs.bf16_normal((M, 512), g))


@pytest.mark.parametrize("M", [33, 150, 300])
def test_large_m_row_codes_ragged_k_with_bias(M):
    """1x32 per-row weight codes that do not fold into 32x32 blocks, K not a
    multiple of 128 (padded to Kp), on the block-scaled GEMM (M > 32)."""
    g = inputs.generator(400 + M)
    N, K = 200, 1056
    w = inputs.e4m3_bytes((N, K), g)
    c = inputs.e8m0_codes((N, K // 32), 116, 134, g)
    b = inputs.bf16_normal((N,), g)
    p = pack(w, c)
    assert p.scale_mode == mx.MX_SCALE_ROW1X32
    check(p, w, c, inputs.bf16_normal((M, K), g), bias=b)


def test_batch_invariance_and_fused_equals_unfused():
    c = inputs.decode_linear(K=2080, Ms=(32,), seed=3)
    p = pack(c["w"], c["codes"])
    x = c["xs"][32]
    y32 = gpu_linear(p, x).cpu()
    for m in (0, 7, 31):
        y1 = gpu_linear(p, x[m:m + 1]).cpu()
        assert torch.equal(y1[0].view(torch.int16), y32[m].view(torch.int16)), m
    y4 = gpu_linear(p, x[:4]).cpu()
    y4u = gpu_linear(p, x[:4], flags=mx.MX_LINEAR_NO_FUSED_QUANT).cpu()
    assert torch.equal(y4.view(torch.int16), y4u.view(torch.int16))
    assert torch.equal(y4.view(torch.int16), y32[:4].view(torch.int16))


@pytest.mark.parametrize("N,K", [(24576, 1536), (24576, 896), (4096, 7168), (7168, 8192)])
def test_batch_invariance_where_the_ring_depth_follows_m(N, K):
    """Shapes whose weight ring depth differs between M <= 16 and M > 16 (a
    third stage, or a fourth on long slices), or whose slices are 3 and 4
    steps long (K=896: 7 steps over 2 slices): each token's output is the same
    bits at M = 1, 16, 17 and 32."""
    g = inputs.generator(N + K + 1)
    w = inputs.e4m3_bytes((N, K), g)
    c = inputs.e8m0_codes((N // 32, K // 32), 118, 132, g)
    p = pack(w, c)
    x = inputs.bf16_normal((32, K), g)
    y32 = gpu_linear(p, x).cpu()
    for M in (1, 16, 17):
        yM = gpu_linear(p, x[:M]).cpu()
        assert torch.equal(yM.view(torch.int16), y32[:M].view(torch.int16)), M


@pytest.mark.parametrize("N,K", [(24576, 1536), (7168, 8192)])
def test_layer_sweep_linears_sampled_rows(N, K):
    g = inputs.generator(N + K)
    w = inputs.e4m3_bytes((N, K), g)
    c = inputs.e8m0_codes((N // 32, K // 32), 118, 132, g)
    p = pack(w, c)
    rows = np.sort(np.random.default_rng(1).choice(N, size=256, replace=False))
    for M in (1, 8, 32, 64, 128, 256):
        check(p, w, c, inputs.bf16_normal((M, K), g), rows=rows)


def test_prefill_full_size_sampled():
    c = inputs.prefill_gemm()
    p = pack(c["w"], c["codes"])
    y = gpu_linear(p, c["x"]).float().cpu().numpy()
    rng = np.random.default_rng(2)
    ms = np.sort(rng.choice(4096, size=24, replace=False))
    ns = np.sort(rng.choice(7168, size=48, replace=False))
    wn = u8(c["w"])[ns]
    cn = row_codes(u8(c["codes"]), 7168)[ns]
    ref = ref_linear(bf16_np(c["x"][ms]), wn, cn)
    err = normalized_error(y[np.ix_(ms, ns)], ref["y"], ref["A"], ref["B"])
    assert err <= TOL, err
    assert elementwise_excess(y[np.ix_(ms, ns)], ref) <= 0.0


@pytest.mark.parametrize("M,K", [(1, 2048), (5, 2080), (17, 2080), (32, 2048)])
def test_tensor_core_gemv_separate_quantizer_is_bit_identical(M, K):
    """MX_LINEAR_NO_FUSED_QUANT on the tensor-core GEMV: x quantized by its own
    launch into the workspace gives the fused path's bits (and the oracle's)."""
    c = inputs.decode_linear(K=K, Ms=(M,), N=704, seed=M)
    p = pack(c["w"], c["codes"])
    x = c["xs"][M]
    y = gpu_linear(p, x)
    yu = gpu_linear(p, x, flags=mx.MX_LINEAR_NO_FUSED_QUANT)
    assert torch.equal(y.view(torch.int16), yu.view(torch.int16))
    check(p, c["w"], c["codes"], x, flags=mx.MX_LINEAR_NO_FUSED_QUANT)


@pytest.mark.parametrize("M", [1, 5, 9, 32])
def test_cluster_gemv_path(M):
    """The mma.sync GEMV with cluster split-K (MX_LINEAR_CLUSTER_GEMV)."""
    g = inputs.generator(300 + M)
    w = inputs.e4m3_bytes((96, 2080), g)
    c = inputs.e8m0_codes((3, 65), 118, 132, g)
    p = pack(w, c)
    x = inputs.bf16_normal((M, 2080), g)
    check(p, w, c, x, flags=mx.MX_LINEAR_CLUSTER_GEMV)
    check(p, w, c, x, flags=mx.MX_LINEAR_CLUSTER_GEMV | mx.MX_LINEAR_NO_FUSED_QUANT)
    cr = inputs.e8m0_codes((96, 65), 118, 132, g)
    check(pack(w, cr), w, cr, x, flags=mx.MX_LINEAR_CLUSTER_GEMV)


def test_decode_linear_cluster_gemv_full_size():
    c = inputs.decode_linear(K=2048, Ms=(1, 32), seed=4)
    p = pack(c["w"], c["codes"])
    for M, x in c["xs"].items():
        check(p, c["w"], c["codes"], x, flags=mx.MX_LINEAR_CLUSTER_GEMV)


def test_workspace_too_small_is_an_error():
    g = inputs.generator(4)
    w = inputs.e4m3_bytes((64, 256), g)
    c = inputs.e8m0_codes((2, 8), 120, 130, g)
    p = pack(w, c)
    dev = cuda_device()
    x = inputs.bf16_normal((40, 256), g).to(dev)   # M > 32: the GEMM needs the workspace
    with pytest.raises(mx.MxError) as ei:
        mx.mxfp8_linear(x, p, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert ei.value.code == mx.binding.MX_ERR_WORKSPACE
    x = inputs.bf16_normal((20, 256), g).to(dev)   # so does the cluster GEMV past the fused range
    with pytest.raises(mx.MxError) as ei:
        mx.mxfp8_linear(x, p, flags=mx.MX_LINEAR_CLUSTER_GEMV,
                        workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert ei.value.code == mx.binding.MX_ERR_WORKSPACE


# ------------------------------------------------ pre-quantized activation input

@pytest.mark.parametrize("M,K", [(1, 2048), (5, 2080), (32, 2080), (40, 2080), (200, 1024)])
def test_prequantized_equals_fused_quant_bitwise(M, K):
    """mxfp8_linear_q on mx_quantize_act(x) is bit-identical to mxfp8_linear(x)
    (decode GEMV for M <= 32, GEMM reading xq in place for larger M)."""
    dev = cuda_device()
    c = inputs.decode_linear(K=K, Ms=(M,), N=704)
    p = pack(c["w"], c["codes"])
    x = c["xs"][M].to(dev)
    bias = inputs.bf16_normal((704,), inputs.generator(3)).to(dev)
    xq, xc = mx.mx_quantize_act(x)
    y1 = mx.mxfp8_linear(x, p, bias)
    y2 = mx.mxfp8_linear_q(xq, xc, p, bias)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M", [3, 77])
def test_prequantized_arbitrary_bytes_vs_oracle(M):
    """Activation bytes and codes that no quantizer produced (every non-NaN e4m3
    byte, codes 110..140) against the oracle's pre-quantized linear."""
    from oracle.linear import mxfp8_linear_q as ref_q
    dev = cuda_device()
    g = inputs.generator(M)
    N, K = 320, 1056
    w = inputs.e4m3_bytes((N, K), g)
    wc = inputs.e8m0_codes((N // 32, K // 32), 118, 132, g)
    xq = inputs.e4m3_bytes((M, K), g)
    xc = inputs.e8m0_codes((M, K // 32), 110, 140, g)
    p = pack(w, wc)
    y = mx.mxfp8_linear_q(xq.to(dev), xc.to(dev), p).float().cpu().numpy()
    ref = ref_q(u8(xq), u8(xc), u8(w), row_codes(u8(wc), N))
    assert normalized_error(y, ref["y"], ref["A"], ref["B"]) <= TOL
    assert elementwise_excess(y, ref) <= 0.0


def test_zero_tokens_linear():
    """M = 0: the linear returns at once with an empty output."""
    dev = cuda_device()
    ensure_built()
    c = inputs.gemv_small()
    p = mx.mx_pack_weights(c["w"].to(dev), c["codes"].to(dev), "e4m3")
    y = mx.mxfp8_linear(c["x"][:0].to(dev), p)
    torch.cuda.synchronize()
    assert y.shape == (0, p.desc.N)


def test_large_m_padded_rows_and_k():
    """The block-scaled GEMM with a large activation, padded rows (M = 1000 ->
    1024) and padded K (4160 -> 4224, pad code 127), per-row weight codes and
    a bias; every output against the oracle."""
    g = inputs.generator(77)
    N, K, M = 320, 4160, 1000
    w = inputs.e4m3_bytes((N, K), g)
    c = inputs.e8m0_codes((N, K // 32), 118, 132, g)
    b = inputs.bf16_normal((N,), g)
    check(pack(w, c), w, c, inputs.bf16_normal((M, K), g), bias=b)


@pytest.mark.parametrize("M,N", [(45, 203), (130, 1000)])
def test_gemm_k_split_ragged_n_with_bias(M, N):
    """Few output tiles on a long K: the GEMM splits K into ranges (f32 partial
    sums, then the ranges added in order, the bias, one rounding).  N = 203
    takes the element-wise partial and finishing stores, N = 1000 the vector
    ones; every output against the oracle."""
    K = 4128
    g = inputs.generator(M + N)
    w = inputs.e4m3_bytes((N, K), g)
    c = inputs.e8m0_codes((N, K // 32), 118, 132, g)
    b = inputs.bf16_normal((N,), g)
    p = pack(w, c)
    Mp, Kp = (M + 127) // 128 * 128, p.desc.Kp
    no_split = -(-Mp * Kp // 256) * 256 + -(-Mp * Kp // 32 // 256) * 256
    full = mx.mxfp8_linear_workspace_size(M, p)
    assert full >= no_split + 2 * M * N * 4   # room for two or more K ranges
    x = inputs.bf16_normal((M, K), g)
    check(p, w, c, x, bias=b)
    dev = cuda_device()
    # the required bytes only (no split), then room for two ranges: both
    # against the oracle too
    for nbytes in (no_split, no_split + 2 * M * N * 4):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        y2 = mx.mxfp8_linear(x.to(dev), p, b.to(dev), workspace=ws)
        torch.cuda.synchronize()
        wn, cn = u8(w), row_codes(u8(c), N)
        ref = ref_linear(bf16_np(x), wn, cn, bf16_np(b))
        y2n = y2.float().cpu().numpy()
        assert normalized_error(y2n, ref["y"], ref["A"], ref["B"]) <= TOL
        assert elementwise_excess(y2n, ref) <= 0.0

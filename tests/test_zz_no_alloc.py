"""mxfp8_linear_noalloc: the decode linear for callers that cannot allocate
device memory (engines with pre-planned memory, plugins handed only their
input and output buffers).  It keeps its scratch in a fixed library-owned
device array; on two calls in a row that share that array it must match the
oracle within the tests' tolerance (the 1e-2 gate and the per-element bound)
and give the workspace entry point's bits.

This file is named so pytest collects it last, and it depends on no other test:
it passes alone in a fresh process and after the rest of the suite."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import inputs
from oracle.linear import mxfp8_linear as ref_linear, normalized_error
from tests.helpers import TOL, bf16_np, cuda_device, elementwise_excess, ensure_built, u8

pytestmark = pytest.mark.gpu


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    dev = cuda_device()
    ensure_built()
    c = inputs.decode_linear(K=2080, Ms=(16, 32), seed=21)
    p = mx.mx_pack_weights(c["w"].to(dev), c["codes"].to(dev), "e4m3")
    row_codes = np.repeat(u8(c["codes"]), 32, axis=0)
    for M in (32, 16):  # the second call reuses the array the first one filled
        x = c["xs"][M].to(dev)
        want = mx.mxfp8_linear(x, p, flags=mx.MX_LINEAR_CLUSTER_GEMV | mx.MX_LINEAR_NO_FUSED_QUANT)
        got = mx.mxfp8_linear_noalloc(x, p)
        torch.cuda.synchronize()
        ref = ref_linear(bf16_np(c["xs"][M]), u8(c["w"]), row_codes)
        y = got.float().cpu().numpy()
        err = normalized_error(y, ref["y"], ref["A"], ref["B"])
        assert err <= TOL, (M, err)
        assert elementwise_excess(y, ref) <= 0.0, M
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), M


def test_noalloc_rejects_sizes_beyond_its_array():
    dev = cuda_device()
    ensure_built()
    g = inputs.generator(22)
    p = mx.mx_pack_weights(inputs.e4m3_bytes((64, 32768), g).to(dev),
                           inputs.e8m0_codes((2, 1024), 120, 130, g).to(dev), "e4m3")
    with pytest.raises(mx.MxError) as ei:
        mx.mxfp8_linear_noalloc(inputs.bf16_normal((32, 32768), g).to(dev), p)
    assert ei.value.code == mx.binding.MX_ERR_UNSUPPORTED and "scratch" in str(ei.value)
    with pytest.raises(mx.MxError) as ei:
        mx.mxfp8_linear_noalloc(inputs.bf16_normal((33, 32768), g).to(dev), p)
    assert ei.value.code == mx.binding.MX_ERR_UNSUPPORTED

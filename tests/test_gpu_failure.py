"""Failure detection without a GPU fault: a bounded wait that nothing completes
runs out after its limit, the kernel returns normally, and the host reads
MX_ERR_TIMEOUT from mx_check_device_errors; the context stays usable."""
import ctypes

import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import binding
from tests.helpers import cuda_device, ensure_built

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_is_reported():
    dev = cuda_device()
    lib = ensure_built()
    mx.mx_check_device_errors()                       # start clean
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.mx_selftest_bounded_wait(2000, ctypes.c_void_p(flag.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == binding.MX_OK
    torch.cuda.synchronize()
    assert int(flag.item()) == 1                      # the wait gave up
    with pytest.raises(mx.MxError) as ei:
        mx.mx_check_device_errors()
    assert ei.value.code == binding.MX_ERR_TIMEOUT
    mx.mx_check_device_errors()                       # flag cleared by the read
    # the context still runs kernels
    q, c = mx.mx_quantize_act(torch.ones((1, 64), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    # all ones: code 127 + ceil(log2(1 / 448)) = 119, each value 1 x 2^8 = e4m3 0x78
    assert int(c[0, 0]) == 119 and int(q[0, 0]) == 0x78

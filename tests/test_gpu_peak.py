"""mx_measure_mxf8_peak: the dense MXFP8 tensor throughput measured by an
MMA-only tcgen05 loop (the roofline denominator of the block-scaled GEMM).
The loop checks its own accumulators; here the figure must also be physical:
above the best the library's GEMM kernel reaches on a GB300 (2.8 PFLOP/s) and below
twice the nominal dense fp8 rate (4.5 PFLOP/s)."""
import pytest

import mxfp4_quantized_linear_gb300 as mx
from tests.helpers import cuda_device, ensure_built

pytestmark = pytest.mark.gpu


def test_measured_mxf8_peak_is_physical():
    cuda_device()
    ensure_built()
    tf = mx.mx_measure_mxf8_peak(iters=1000, reps=3)
    assert 2800.0 < tf < 9000.0, tf


def test_peak_rejects_bad_arguments():
    cuda_device()
    ensure_built()
    with pytest.raises(mx.MxError) as ei:
        mx.mx_measure_mxf8_peak(iters=0, reps=1)
    assert ei.value.code == mx.binding.MX_ERR_ARG

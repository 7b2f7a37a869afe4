"""Shared test helpers: device selection, tolerance, oracle comparisons."""
import numpy as np
import pytest
import torch

TOL = 1e-2  # max-abs error normalised by ||w_n||_2 ||x_m||_2 of the operands


def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def ensure_built():
    from mxfp4_quantized_linear_gb300 import binding, build
    import os
    if not os.path.exists(binding.lib_path()):
        build.build()
    return binding.load_library()


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> fp64 numpy of its exact values."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()

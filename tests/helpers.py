"""Shared test helpers: device selection, tolerance, oracle comparisons."""
import numpy as np
import pytest
import torch

TOL = 1e-2  # max-abs error normalised by ||w_n||_2 ||x_m||_2 of the operands


def elementwise_excess(y, ref) -> float:
    """Largest excess of |y - y_ref| over 2^-8 |y_ref| + 1e-5 ||A_m|| ||B_n||,
    normalised by ||A_m|| ||B_n|| (<= 0 passes); ``ref`` holds the oracle's
    y, A (activation rows as multiplied) and B (weight rows).  Exact products
    with f32 sums and one bf16 rounding stay far inside this bound; one 32-wide
    K block dropped or scaled by a wrong code moves an output by about
    sqrt(32) / K of ||A_m|| ||B_n|| (7e-4 at K = 8192), which the 1e-2 gate
    alone does not see."""
    y = np.asarray(y, dtype=np.float64)
    den = np.linalg.norm(ref["A"], axis=1)[:, None] * np.linalg.norm(ref["B"], axis=1)[None, :]
    den = np.where(den > 0, den, 1.0)
    excess = np.abs(y - ref["y"]) - (2.0 ** -8 * np.abs(ref["y"]) + 1e-5 * den)
    return float(np.max(excess / den)) if excess.size else 0.0


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

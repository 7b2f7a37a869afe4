"""MXFP8 dequant and the MX x MX linear, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* Dequant: w = e4m3(byte) x 2^(code - 127) (weights942, ``ocp_from_dequant``;
  rocm_native names it ``dequant_mxfp8_to_bf16``), rounded once to bf16
  (round-to-nearest-even).  e2m1 bytes dequantize the same way with the e2m1
  value (a16w4, ``dequant``: fp4x2 with its E8M0 scale to BF16).
* Linear: out = x @ w.T (rocm_native, ``_launch``) where the bf16 activation
  is MXFP8-quantized per token inside the call (rocm_native,
  ``apply_weights``: the op quantizes the activation itself), each 32-wide K
  block scaled by the weight code times the activation code:

      y[m, n] = sum_b 2^(cw[n,b]-127) 2^(cx[m,b]-127) sum_{k in b} W[n,k] xq[m,k]

  plus an optional bias added after the product (``apply_weights``).  The sum
  is taken by a float64 matrix product of the exactly dequantized operands.

``mxfp8_linear_q`` is the same product on an activation given already
quantized (rocm_native, apply_weights: QuantizedActivation, row-major
[M, K/32] E8M0 scales); ``mxfp8_linear`` quantizes first, then calls it.

Pinned by tests/test_oracle_linear.py: exact rational (Fraction) brute force on
tiny shapes (from bf16 activations and from arbitrary e4m3 bytes and codes),
the one-hot / all-ones special cases, and invariance under permuting 32-wide K
chunks together with their code columns.
"""
import numpy as np

from .formats import bf16_rne_bits, bf16_value, e2m1_decode, e2m1_unpack, e4m3_decode, e4m3_rne, e8m0_decode
from .quant import quantize_act


def expand_codes(codes, N: int, K: int) -> np.ndarray:
    """Codes [N/32, K/32] (32x32 blocks) or [N, K/32] (1x32 rows) -> per-element
    scale factors [N, K] in fp64."""
    codes = np.asarray(codes, dtype=np.uint8)
    f = e8m0_decode(codes)
    if codes.shape[0] != N:
        f = np.repeat(f, 32, axis=0)[:N]
    return np.repeat(f, 32, axis=1)[:, :K]


def dequant_values(w_bytes, codes, fmt: str, N: int, K: int) -> np.ndarray:
    """Exact fp64 values value(byte) x 2^(code - 127), [N, K]."""
    if fmt == "e4m3":
        v = e4m3_decode(np.asarray(w_bytes).reshape(N, K))
    elif fmt == "e2m1":
        v = e2m1_decode(e2m1_unpack(np.asarray(w_bytes).reshape(N, K // 2)))
    else:
        raise ValueError(fmt)
    return v * expand_codes(codes, N, K)


def e4m3_from_dequant(w_bf16_values, codes) -> tuple:
    """weights942, ocp_from_dequant: the OCP e4m3 bytes [N, K] behind a bf16
    weight w = e4m3 value x 2^(code - 127) (codes [N/32, K/32] blocks or
    [N, K/32] rows).  Each value is scaled by 2^(127 - code) and rounded to
    e4m3 (nearest-even); it is given back exactly when that byte's dequant,
    rounded to bf16, equals w (-0 and +0 compare equal, NaN never does).

    Returns (bytes uint8 [N, K], number of values not given back)."""
    w = np.asarray(w_bf16_values, dtype=np.float64)
    N, K = w.shape
    scale = expand_codes(codes, N, K)               # 2^(code - 127), fp64 (exact)
    v = w / scale                                    # exact power-of-two scaling
    finite = np.isfinite(v) & (np.abs(v) <= 448.0)
    q = np.full((N, K), 0x7F, dtype=np.uint8)        # values outside e4m3 -> NaN byte
    q[finite] = e4m3_rne(v[finite])
    back = bf16_value(bf16_rne_bits(e4m3_decode(q) * scale))
    with np.errstate(invalid="ignore"):
        bad = ~(back == w)
    return q, int(np.count_nonzero(bad))


def dequant_bf16(w_bytes, codes, fmt: str, N: int, K: int) -> np.ndarray:
    """bf16 bit patterns [N, K] of the dequantized weight."""
    return bf16_rne_bits(dequant_values(w_bytes, codes, fmt, N, K))


def mxfp8_linear_q(xq, xcodes, w_bytes, w_codes, bias=None) -> dict:
    """The linear on an activation that arrives already MXFP8-quantized
    (rocm_native, apply_weights: a QuantizedActivation with row-major
    [M, K/32] E8M0 scales, input_quant_key): xq [M, K] e4m3 bytes, xcodes
    [M, K/32]; weight and bias as in mxfp8_linear.

    Returns dict(y=[M, N] fp64, A=[M, K] dequantized activation, B)."""
    xq = np.asarray(xq, dtype=np.uint8)
    M, K = xq.shape
    w_bytes = np.asarray(w_bytes, dtype=np.uint8)
    N = w_bytes.shape[0]
    A = e4m3_decode(xq) * expand_codes(xcodes, M, K)
    B = dequant_values(w_bytes, w_codes, "e4m3", N, K)
    y = A @ B.T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    return {"y": y, "A": A, "B": B}


def mxfp8_linear(x, w_bytes, w_codes, bias=None) -> dict:
    """x: fp64 [M, K] (bf16 values); w_bytes [N, K] e4m3; w_codes block
    [N/32, K/32] or row [N, K/32]; bias fp64 [N] or None.  The activation is
    quantized per token first, then multiplied as in mxfp8_linear_q.

    Returns dict(y=[M, N] fp64, xq, xcodes, A=[M, K] dequantized activation,
    B=[N, K] dequantized weight)."""
    x = np.asarray(x, dtype=np.float64)
    xq, xcodes = quantize_act(x)
    r = mxfp8_linear_q(xq, xcodes, w_bytes, w_codes, bias)
    r.update(xq=xq, xcodes=xcodes)
    return r


def normalized_error(y, y_ref, A, B) -> float:
    """max_{m,n} |y - y_ref| / (||A_m||_2 ||B_n||_2): the output tolerance
    measure (max-abs error normalised by the L2 norms of the operands' rows).
    Rows with a zero norm count only where y differs from y_ref."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    na = np.linalg.norm(np.asarray(A, dtype=np.float64), axis=1)
    nb = np.linalg.norm(np.asarray(B, dtype=np.float64), axis=1)
    denom = na[:, None] * nb[None, :]
    diff = np.abs(y - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(denom > 0, diff / np.where(denom > 0, denom, 1.0),
                     np.where(diff > 0, np.inf, 0.0))
    return float(np.max(e)) if e.size else 0.0

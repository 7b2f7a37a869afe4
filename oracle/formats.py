"""Number formats used by the MX linear: OCP e4m3, e2m1, E8M0 and bf16.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Decoding follows the closed forms of the formats; encoding is round-to-nearest,
ties-to-even, computed exactly in fp64 with power-of-two scalings only.

Sources:
* e4m3 is the OCP ``float8_e4m3fn`` type that the weights942 page names in
  ``linear_copy`` / ``ocp_from_dequant`` and that the rocm_native page casts to
  in ``_quant_mxfp8_tile``.
* e2m1 is "fp4x2, low nibble first" (a16w4, ``dequant``); its -0 nibble is 0x8
  (weights942, ``fp4_drop_negative_zero_``).  The value set itself is not
  printed on the pages: the reading taken is the OCP MX v1.0 e2m1 format
  (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, subnormals, no
  inf/NaN).
* E8M0 code c stands for 2^(c - 127) (weights942, ``ocp_from_dequant``:
  w = e4m3 value x 2^(code - 127)); code 255 is NaN (OCP).  The a16w4 page's
  ``scale_f32`` builds the factor as ``code << 23`` reinterpreted as f32, which
  gives 0.0 instead of 2^-127 for code 0; the reading taken here is the OCP
  value 2^-127.

Pinned by tests/test_oracle_formats.py: the e4m3 table against torch's CPU
``float8_e4m3fn`` decode (all 256 codes), the rounding against torch's CPU cast
and a brute-force nearest-value search, e2m1 through the same generic
minifloat decoder as e4m3 plus its printed -0 code, bf16 rounding against
torch's CPU fp32->bf16 cast.
"""
import math

import numpy as np


def minifloat_value(code: int, ebits: int, mbits: int, bias: int) -> float:
    """Value of a sign / exponent / mantissa code with subnormals (no inf/NaN)."""
    sign = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        mag = math.ldexp(m, 1 - bias - mbits)
    else:
        mag = math.ldexp((1 << mbits) + m, e - bias - mbits)
    return -mag if sign else mag


def _e4m3_value(code: int) -> float:
    # float8_e4m3fn: exponent 15 with mantissa 7 is NaN (both signs); no inf.
    if code & 0x7F == 0x7F:
        return math.nan
    return minifloat_value(code, 4, 3, 7)


E4M3_VALUES = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0
E2M1_VALUES = np.array([minifloat_value(c, 2, 1, 1) for c in range(16)], dtype=np.float64)
# the 127 non-negative, non-NaN e4m3 codes 0x00..0x7E, in increasing value
_E4M3_POS = E4M3_VALUES[:0x7F]
BF16_MAX = math.ldexp(255, 127 - 7)  # (2 - 2^-7) * 2^127


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> fp64 values (NaN for 0x7F / 0xFF, -0.0 for 0x80)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e2m1_decode(nibbles) -> np.ndarray:
    """4-bit codes (0..15) -> fp64 values; 0x8 is -0.0."""
    return E2M1_VALUES[np.asarray(nibbles, dtype=np.uint8) & 0xF]


def e2m1_unpack(packed) -> np.ndarray:
    """fp4x2 bytes [..., K/2] -> nibbles [..., K]; element 2i is the low nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def e8m0_decode(codes) -> np.ndarray:
    """uint8 E8M0 codes -> fp64 2^(c - 127); code 255 -> NaN."""
    c = np.asarray(codes, dtype=np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


def _rne_to_grid(a: np.ndarray, min_exp: int, mbits: int) -> np.ndarray:
    """Round non-negative a to the nearest number with ``mbits`` fraction bits
    whose exponent is at least ``min_exp`` (subnormal spacing below it), ties to
    even.  All steps are exact in fp64: the quantum is a power of two and rint
    rounds half to even."""
    _, ex = np.frexp(a)  # a in [2^(ex-1), 2^ex) for a > 0
    e = np.maximum(ex - 1, min_exp)
    quantum = np.ldexp(1.0, e - mbits)
    return np.rint(a / quantum) * quantum


def e4m3_rne(v) -> np.ndarray:
    """fp64 values with |v| <= 448 -> e4m3 codes, round-to-nearest-even.

    The sign is kept, so a negative value that rounds to zero gives 0x80.
    NaN gives 0x7F.  |v| > 448 is outside this function's domain (the
    quantizer's scale choice guarantees |v| <= 448) and raises.
    """
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    a = np.abs(np.where(nan, 0.0, v))
    if np.any(a > E4M3_MAX):
        raise ValueError("e4m3_rne: |v| > 448 is outside the quantizer's range")
    mag = _rne_to_grid(a, -6, 3)
    code = np.searchsorted(_E4M3_POS, mag).astype(np.uint8)
    assert np.array_equal(_E4M3_POS[code], mag), "rounded value is not an e4m3 value"
    code = code | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def bf16_rne_bits(v) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), round-to-nearest-even,
    overflow to +-inf, subnormals kept, NaN -> 0x7FC0."""
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    a = np.abs(np.where(nan, 0.0, v))
    finite = np.isfinite(a)
    mag = _rne_to_grid(np.where(finite, a, 0.0), -126, 7)
    mag = np.where(finite & (mag <= BF16_MAX), mag, np.inf)
    # mag is exactly representable in bf16, hence in fp32: take its top 16 bits
    bits = (mag.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = bits | np.where(np.signbit(v), 0x8000, 0).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), bits).astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)

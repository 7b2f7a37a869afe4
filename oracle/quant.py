"""Per-token MXFP8 activation quantizer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows rocm_native (vllm.model_executor.kernels.linear.mxfp8.rocm_native),
section ``_quant_mxfp8_tile``: for each row and each block of 32 consecutive
K elements,

    amax = max(max_k |x_k|, TINY)
    sb   = clamp(ceil(log2(amax / FP8_MAX)) + 127, 0, 254)
    q_k  = e4m3(x_k * 2^(127 - sb))

returning the e4m3 codes and the E8M0 codes ``sb``, with the codes row-major
[M, K/32] (rocm_native, ``input_quant_key``).  The page multiplies by the
reciprocal power of two rather than dividing (``_quant_mxfp8_tile``).

Readings where the page is silent:
* FP8_MAX is named (``_FP8_MAX``) but not printed: 448, the e4m3 maximum.
* TINY is named (``_TINY``) but not printed: 2^-126, the float32 ``tiny``.
  Only the code of a block whose |x| are all below 2^-126 depends on it (it is
  then 0).  This value is parity unpinned against the pages.
* ceil(log2(.)) is taken in exact arithmetic: sb - 127 is the smallest
  integer e with amax <= 448 * 2^e.
* The cast to e4m3 rounds to nearest, ties to even, keeps the sign (so -tiny
  gives 0x80) and keeps subnormals.  It never saturates: |x * 2^(127 - sb)|
  <= 448 by the choice of sb.
* NaN or +-inf anywhere in a block (undefined on the page): the block's code is
  255 (the E8M0 NaN) and all its bytes are 0x7F (the e4m3 NaN).

Pinned by tests/test_oracle_quant.py: hand-derived golden blocks
(tests/golden/quant_blocks.txt), a brute-force search over all 255 codes,
the invariants max|q| <= 448 and tightness (some |q| >= 224 when sb > 0), and
the exact dequant -> requant round trip.
"""
import numpy as np

from .formats import e4m3_rne

FP8_MAX = 448.0
TINY = 2.0 ** -126
MX_BLOCK = 32


def block_code(amax) -> np.ndarray:
    """E8M0 code sb = clamp(ceil(log2(amax / 448)) + 127, 0, 254), exactly.

    Write amax = f * 2^ex with f in [0.5, 1).  Then amax / 2^(ex - 9) = 512 f
    lies in [256, 512), so the smallest e with amax <= 448 * 2^e is ex - 9
    when 512 f <= 448 and ex - 8 otherwise.
    """
    amax = np.asarray(amax, dtype=np.float64)
    f, ex = np.frexp(amax)
    e = ex.astype(np.int64) - 9 + (512.0 * f > FP8_MAX)
    return np.clip(e + 127, 0, 254).astype(np.int64)


def quantize_act(x) -> tuple:
    """x: fp64 [M, K] (bf16 values), K % 32 == 0 ->
    (q uint8 [M, K] e4m3 codes, codes uint8 [M, K/32] E8M0)."""
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    assert K % MX_BLOCK == 0, "K must be a multiple of 32"
    xb = x.reshape(M, K // MX_BLOCK, MX_BLOCK)
    bad = ~np.all(np.isfinite(xb), axis=2)
    xb_clean = np.where(bad[..., None], 0.0, xb)
    amax = np.maximum(np.max(np.abs(xb_clean), axis=2), TINY)
    sb = block_code(amax)
    rescale = np.ldexp(1.0, 127 - sb)
    q = e4m3_rne(xb_clean * rescale[..., None])
    q = np.where(bad[..., None], np.uint8(0x7F), q).astype(np.uint8)
    sb = np.where(bad, 255, sb).astype(np.uint8)
    return q.reshape(M, K), sb

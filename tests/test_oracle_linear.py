"""Pins for oracle/linear.py: exact rational brute force, special cases, and
K-chunk permutation invariance."""
import math
from fractions import Fraction

import numpy as np
import torch

from oracle import formats as F
from oracle.linear import dequant_bf16, dequant_values, mxfp8_linear, normalized_error
from oracle.quant import quantize_act


def torch_e4m3(b):
    return torch.tensor(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def bf16_vals(rng, shape):
    return F.bf16_value(F.bf16_rne_bits(rng.standard_normal(shape)))


def rand_e4m3(rng, shape):
    r = rng.integers(0, 254, size=shape)
    return (r + (r >= 0x7F)).astype(np.uint8)


def brute_linear(x, w, codes, block: bool):
    """Exact rational y[m][n] from raw bytes and codes, element by element."""
    M, K = x.shape
    N = w.shape[0]
    xq, xc = quantize_act(x)
    xv, wv = torch_e4m3(xq), torch_e4m3(w)
    y = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                cw = codes[n // 32, k // 32] if block else codes[n, k // 32]
                sa = Fraction(2) ** (int(xc[m, k // 32]) - 127)
                sw = Fraction(2) ** (int(cw) - 127)
                acc += Fraction(xv[m, k]) * sa * Fraction(wv[n, k]) * sw
            y[m][n] = acc
    return y


def test_linear_matches_rational_brute_force_row_and_block():
    rng = np.random.default_rng(0)
    for block, N in ((False, 5), (True, 32)):
        M, K = 3, 96
        x = bf16_vals(rng, (M, K))
        w = rand_e4m3(rng, (N, K))
        codes = rng.integers(118, 133, size=((N // 32) if block else N, K // 32)).astype(np.uint8)
        y = mxfp8_linear(x, w, codes)["y"]
        ref = brute_linear(x, w, codes, block)
        for m in range(M):
            for n in range(N):
                assert math.isclose(y[m, n], float(ref[m][n]), rel_tol=1e-13, abs_tol=1e-300)


def test_all_ones_weight_gives_row_sums():
    rng = np.random.default_rng(1)
    M, N, K = 4, 32, 128
    x = bf16_vals(rng, (M, K))
    w = np.full((N, K), 0x38, dtype=np.uint8)            # e4m3 1.0
    codes = np.full((1, K // 32), 127, dtype=np.uint8)   # 2^0
    out = mxfp8_linear(x, w, codes)
    rows = out["A"].sum(axis=1)
    assert np.allclose(out["y"], rows[:, None], rtol=1e-14, atol=0)


def test_one_hot_weight_selects_activation_and_code_shift_scales():
    rng = np.random.default_rng(2)
    M, N, K = 3, 32, 128
    x = bf16_vals(rng, (M, K))
    w = np.zeros((N, K), dtype=np.uint8)
    for n in range(N):
        w[n, (5 * n + 3) % K] = 0x38
    codes = np.full((1, 4), 127, dtype=np.uint8)
    out = mxfp8_linear(x, w, codes)
    for n in range(N):
        assert np.array_equal(out["y"][:, n], out["A"][:, (5 * n + 3) % K])
    # code + 3 multiplies every product by 8, exactly
    y8 = mxfp8_linear(x, w, codes + 3)["y"]
    assert np.array_equal(y8, 8 * out["y"])


def test_k_chunk_permutation_invariance():
    rng = np.random.default_rng(3)
    M, N, K = 5, 64, 256
    x = bf16_vals(rng, (M, K))
    w = rand_e4m3(rng, (N, K))
    codes = rng.integers(118, 133, size=(N, K // 32)).astype(np.uint8)
    perm = rng.permutation(K // 32)
    cols = (perm[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    y = mxfp8_linear(x, w, codes)["y"]
    yp = mxfp8_linear(x[:, cols], w[:, cols], codes[:, perm])["y"]
    assert np.allclose(y, yp, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_bias_is_added_after_the_product():
    rng = np.random.default_rng(4)
    x = bf16_vals(rng, (2, 64))
    w = rand_e4m3(rng, (32, 64))
    codes = np.full((1, 2), 127, dtype=np.uint8)
    b = bf16_vals(rng, (32,))
    assert np.array_equal(mxfp8_linear(x, w, codes, b)["y"], mxfp8_linear(x, w, codes)["y"] + b)


def test_dequant_exhaustive_bytes_and_codes_vs_torch():
    """bf16(e4m3(b) * 2^(c-127)) for every byte and codes 118..132, against torch's
    fp8 decode times the power of two (exact in fp32) cast to bf16."""
    b = np.arange(256, dtype=np.uint8)
    for c in range(118, 133):
        w = np.tile(b, (32, 1))[:, :256]
        codes = np.full((1, 8), c, dtype=np.uint8)
        got = dequant_bf16(w, codes, "e4m3", 32, 256)
        ref = (torch.tensor(w).view(torch.float8_e4m3fn).float() * 2.0 ** (c - 127)).to(torch.bfloat16)
        ref = ref.view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(F.bf16_value(got))
        assert np.array_equal(nan, np.isnan(F.bf16_value(ref)))
        assert np.array_equal(got[~nan], ref[~nan])


def test_dequant_requant_round_trip():
    """weights942 ocp_from_dequant: the bytes behind a dequantized weight come back
    exactly, for every non-NaN byte (-0 stays -0)."""
    rng = np.random.default_rng(5)
    b = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    for c in rng.integers(3, 247, size=40):
        w = b[None, :].repeat(32, 0)[:, :224]
        codes = np.full((1, 7), c, dtype=np.uint8)
        deq = F.bf16_value(dequant_bf16(w, codes, "e4m3", 32, 224))
        back = F.e4m3_rne(deq * math.ldexp(1.0, 127 - int(c)))
        assert np.array_equal(back, w), c


def test_dequant_e2m1_values():
    w = np.tile(np.array([[0x21, 0x8F]], dtype=np.uint8), (1, 8))
    codes = np.full((1, 1), 128, dtype=np.uint8)
    v = dequant_values(w, codes, "e2m1", 1, 32)
    assert list(v[0, :4]) == [1.0, 2.0, -12.0, -0.0]


def test_normalized_error_measure():
    A = np.array([[3.0, 4.0]])
    B = np.array([[1.0, 0.0], [0.0, 2.0]])
    y_ref = A @ B.T
    y = y_ref + np.array([[0.5, 1.0]])
    assert normalized_error(y, y_ref, A, B) == max(0.5 / 5.0, 1.0 / 10.0)


def test_prequantized_linear_matches_rational_brute_force():
    """Arbitrary e4m3 activation bytes (NaN codes excluded) and codes across the
    E8M0 range, with row codes on the weight: exact rational sums."""
    from oracle.linear import mxfp8_linear_q
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 96
    xq = rand_e4m3(rng, (M, K))
    xc = rng.integers(100, 150, size=(M, K // 32)).astype(np.uint8)
    w = rand_e4m3(rng, (N, K))
    wc = rng.integers(110, 140, size=(N, K // 32)).astype(np.uint8)
    y = mxfp8_linear_q(xq, xc, w, wc)["y"]
    xv, wv = torch_e4m3(xq), torch_e4m3(w)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += (Fraction(xv[m, k]) * Fraction(2) ** (int(xc[m, k // 32]) - 127)
                        * Fraction(wv[n, k]) * Fraction(2) ** (int(wc[n, k // 32]) - 127))
            assert abs(float(acc) - y[m, n]) <= 1e-12 * max(1.0, abs(float(acc)))


def test_e4m3_from_dequant_round_trip_and_refusals():
    """weights942 ocp_from_dequant: every non-NaN e4m3 byte comes back from its
    bf16 dequant at the codes where that dequant is exact (3..246); a value
    moved by one bf16 ulp, or one between two e4m3 values, is refused."""
    from oracle.linear import e4m3_from_dequant
    b = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    for code in (3, 64, 118, 127, 132, 200, 246):
        N = 32
        w = np.tile(b[None, :224], (N, 1))                      # [32, 224]
        codes = np.full((1, 7), code, dtype=np.uint8)           # 32x32 blocks
        wv = F.bf16_value(dequant_bf16(w, codes, "e4m3", N, 224))
        q, bad = e4m3_from_dequant(wv, codes)
        assert bad == 0
        assert np.array_equal(q, w)
    rest = np.tile(b[None, 224:], (32, 1))                     # the last 30 bytes, row codes
    rc = np.full((32, 1), 120, dtype=np.uint8)
    wv = F.bf16_value(dequant_bf16(np.pad(rest, ((0, 0), (0, 2))), rc, "e4m3", 32, 32))
    q, bad = e4m3_from_dequant(wv, rc)
    assert bad == 0 and np.array_equal(q[:, :30], rest)
    # refusals
    codes = np.full((1, 1), 127, dtype=np.uint8)
    w = np.ones((32, 32))
    q, bad = e4m3_from_dequant(w, codes)
    assert bad == 0 and np.all(q == 0x38)                      # 1.0 = 0x38
    w[3, 4] = 1.0625                                           # between 1.0 and 1.125
    w[7, 9] = F.bf16_value(np.array([0x3F81], dtype=np.uint16))[0]   # 1.0 + one bf16 ulp
    w[8, 1] = 449.0                                            # beyond e4m3
    w[9, 2] = np.nan
    assert e4m3_from_dequant(w, codes)[1] == 4
    w2 = np.ones((32, 32))
    w2[0, 0] = -0.0                                            # -0 is e4m3 0x80
    q, bad = e4m3_from_dequant(w2, codes)
    assert bad == 0 and q[0, 0] == 0x80


def test_elementwise_bound_sees_a_lost_k_block_the_gate_misses():
    """The GPU tests' per-element bound (tests/helpers.elementwise_excess)
    against planted mistakes, on the CPU: at K = 8192 a y that drops one
    32-wide K block, or applies that block's weight code one binade off,
    passes the 1e-2 normalised gate but fails the bound; the exact y and y
    rounded once to bf16 pass both."""
    from tests.helpers import elementwise_excess
    rng = np.random.default_rng(11)
    M, N, K = 2, 64, 8192
    x = bf16_vals(rng, (M, K))
    w = rand_e4m3(rng, (N, K))
    codes = rng.integers(118, 133, size=(N // 32, K // 32)).astype(np.uint8)
    ref = mxfp8_linear(x, w, codes)
    A, B = ref["A"], ref["B"]
    b = 100
    blk = slice(32 * b, 32 * b + 32)
    dropped = ref["y"] - A[:, blk] @ B[:, blk].T
    doubled = ref["y"] + A[:, blk] @ B[:, blk].T
    rounded = F.bf16_value(F.bf16_rne_bits(ref["y"]))
    for bad in (dropped, doubled):
        assert normalized_error(bad, ref["y"], A, B) <= 1e-2
        assert elementwise_excess(bad, ref) > 0.0
    assert elementwise_excess(rounded, ref) <= 0.0
    assert elementwise_excess(ref["y"], ref) <= 0.0

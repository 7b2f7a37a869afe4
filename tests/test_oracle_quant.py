"""Pins for oracle/quant.py: hand-derived golden blocks, brute force over all
codes, invariants and the dequant -> requant round trip."""
import math
import os

import numpy as np
import torch

from oracle import formats as F
from oracle.quant import block_code, quantize_act

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.txt")


def load_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, fill, ov, code, fb, bov = [s.strip() for s in line.split("|")]
            x = np.full(32, float(fill))
            if ov != "-":
                for kv in ov.split(","):
                    i, v = kv.split("=")
                    x[int(i)] = float(v)
            b = np.full(32, int(fb, 16), dtype=np.uint8)
            if bov != "-":
                for kv in bov.split(","):
                    i, v = kv.split("=")
                    b[int(i)] = int(v, 16)
            cases.append((name, x, int(code), b))
    return cases


def test_golden_blocks():
    cases = load_golden()
    assert len(cases) >= 14
    for name, x, code, b in cases:
        # every golden input is exactly a bf16 value
        fin = np.isfinite(x)
        assert np.array_equal(F.bf16_value(F.bf16_rne_bits(x[fin])), x[fin]), name
        q, c = quantize_act(x[None, :])
        assert c[0, 0] == code, (name, c[0, 0], code)
        assert np.array_equal(q[0], b), (name, [hex(v) for v in q[0]])


def brute_force_code(block):
    """Smallest code c in 0..254 with max(|x|, 2^-126) * 2^(127 - c) <= 448,
    i.e. ceil(log2(amax / 448)) + 127 clamped to [0, 254], by search."""
    amax = max(float(np.max(np.abs(block))), 2.0 ** -126)
    for c in range(255):
        if amax * math.ldexp(1.0, 127 - c) <= 448.0:
            return c
    return 254


def _bf16_blocks(rng, n):
    """Random bf16 blocks over a wide exponent range, incl. exact 448*2^k amaxes."""
    scale = np.exp2(rng.integers(-140, 120, size=(n, 1)).astype(np.float64))
    x = rng.standard_normal((n, 32)) * scale
    x = F.bf16_value(F.bf16_rne_bits(x))
    # force some blocks to have amax exactly 448 * 2^k or one bf16 ulp either side
    k = rng.integers(-120, 100, size=n // 4)
    idx = rng.integers(0, 32, size=n // 4)
    tie = np.ldexp(448.0, k)
    bump = rng.integers(-1, 2, size=n // 4)
    tie_bits = F.bf16_rne_bits(tie).astype(np.int64) + bump
    rows = np.arange(n // 4)
    x[rows] = np.clip(x[rows], -np.abs(F.bf16_value(tie_bits.astype(np.uint16)))[:, None] / 2,
                      np.abs(F.bf16_value(tie_bits.astype(np.uint16)))[:, None] / 2)
    x[rows, idx] = F.bf16_value(tie_bits.astype(np.uint16))
    return x


def test_code_matches_brute_force_search():
    rng = np.random.default_rng(5)
    x = _bf16_blocks(rng, 4000)
    _, codes = quantize_act(x.reshape(-1, 32))
    for i in range(x.shape[0]):
        assert codes[i, 0] == brute_force_code(x[i]), (i, x[i])


def test_block_code_tie_points():
    for k in range(-130, 121):
        a = math.ldexp(448.0, k)
        assert block_code(np.array([max(a, 2.0 ** -126)]))[0] == min(max(k + 127, 0), 254)


def test_invariants_and_round_trip():
    rng = np.random.default_rng(6)
    x = _bf16_blocks(rng, 20000).reshape(-1, 64)  # 2 blocks per row
    q, c = quantize_act(x)
    v = F.e4m3_decode(q).reshape(-1, 2, 32)
    assert np.all(np.abs(v) <= 448)
    ci = c.astype(np.int64)
    # tight scale: with sb > 0, the block max lands in (224, 448]
    amax = np.max(np.abs(x.reshape(-1, 2, 32)), axis=2)
    scaled = amax * np.ldexp(1.0, 127 - ci)
    pos = ci > 0
    assert np.all(scaled[pos] > 224) and np.all(scaled <= 448)
    assert np.all(np.max(np.abs(v), axis=2)[pos] >= 224)
    # requantizing the dequantized values with the same code gives the same bytes
    deq = v * np.ldexp(1.0, ci - 127)[..., None]
    back = F.e4m3_rne(deq * np.ldexp(1.0, 127 - ci)[..., None])
    assert np.array_equal(back.reshape(q.shape), q)


def test_matches_pages_formula_in_fp32_on_normal_range():
    """An fp32 evaluation of the page's formula (torch.log2 / ceil / exp2 and
    the e4m3 cast) agrees on normal-range bf16 inputs."""
    rng = np.random.default_rng(7)
    x = F.bf16_value(F.bf16_rne_bits(rng.standard_normal((2048, 128))))
    q, c = quantize_act(x)
    t = torch.tensor(x, dtype=torch.float32).reshape(2048, 4, 32)
    amax = t.abs().amax(dim=2).clamp_min(torch.finfo(torch.float32).tiny)
    sb = (torch.ceil(torch.log2(amax / 448.0)) + 127).clamp(0, 254)
    tq = (t * torch.exp2(127 - sb)[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(sb.to(torch.uint8).numpy(), c)
    assert np.array_equal(tq.reshape(2048, 128).numpy(), q)

"""Pins for oracle/formats.py against libraries, specifications and brute force."""
import math

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def test_e4m3_table_matches_torch_decode_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_VALUES
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))  # 0x80 is -0


def test_e4m3_special_codes():
    assert F.E4M3_VALUES[0x7E] == 448.0 == torch.finfo(torch.float8_e4m3fn).max
    assert math.isnan(F.E4M3_VALUES[0x7F]) and math.isnan(F.E4M3_VALUES[0xFF])
    assert F.E4M3_VALUES[0x80] == 0.0 and math.copysign(1, F.E4M3_VALUES[0x80]) < 0
    assert F.E4M3_VALUES[0x01] == 2.0 ** -9            # smallest subnormal
    assert F.E4M3_VALUES[0x08] == 2.0 ** -6            # smallest normal
    assert F.E4M3_VALUES[0x38] == 1.0


def _e4m3_grid_and_midpoints():
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    quarter = pos[:-1] + (pos[1:] - pos[:-1]) / 4
    v = np.concatenate([pos, mids, quarter, pos[1:] - (pos[1:] - pos[:-1]) / 4])
    return np.concatenate([v, -v])


def _torch_e4m3(v):
    t = torch.tensor(np.asarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rne_matches_torch_cast_on_grid_ties_and_random():
    rng = np.random.default_rng(1)
    rand = rng.uniform(-448, 448, 200000)
    small = rng.uniform(-2.0 ** -5, 2.0 ** -5, 100000)
    logu = np.sign(rng.uniform(-1, 1, 100000)) * np.exp2(rng.uniform(-12, 8.8, 100000))
    v = np.concatenate([_e4m3_grid_and_midpoints(), rand, small, logu]).astype(np.float32)
    v = v[np.abs(v) <= 448].astype(np.float64)
    assert np.array_equal(F.e4m3_rne(v), _torch_e4m3(v))


def test_e4m3_rne_brute_force_nearest_even():
    """Nearest finite e4m3 value by exhaustive search, ties to the even code."""
    finite = [c for c in range(256) if not math.isnan(F.E4M3_VALUES[c])]
    vals = np.array([F.E4M3_VALUES[c] for c in finite])
    rng = np.random.default_rng(2)
    samples = np.concatenate([_e4m3_grid_and_midpoints()[::7], rng.uniform(-448, 448, 3000)])
    for x in samples:
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        cands = [finite[i] for i in best]
        # equal magnitude candidates: +-0 ties resolve by the sign of x
        if len(cands) > 1 and all(F.E4M3_VALUES[c] == 0 for c in cands):
            want = 0x80 if math.copysign(1, x) < 0 else 0x00
        else:
            even = [c for c in cands if c % 2 == 0]
            want = even[0] if len(cands) > 1 else cands[0]
        assert F.e4m3_rne(np.array([x]))[0] == want, (x, cands)


def test_e4m3_rne_sign_of_zero_and_nan():
    out = F.e4m3_rne(np.array([0.0, -0.0, -1e-30, 1e-30, np.nan]))
    assert list(out) == [0x00, 0x80, 0x80, 0x00, 0x7F]
    with pytest.raises(ValueError):
        F.e4m3_rne(np.array([449.0]))


def test_e2m1_generic_decoder_matches_ocp_table():
    table = {}
    with open(f"{GOLDEN}/e2m1_ocp.txt") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                table[int(c)] = float(v)
    for c in range(16):
        got = F.E2M1_VALUES[c]
        assert got == table[c] and math.copysign(1, got) == math.copysign(1, table[c]), c
    # the same generic decoder, parametrised for e4m3, is pinned by torch above
    for c in range(256):
        if c & 0x7F != 0x7F:
            assert F.minifloat_value(c, 4, 3, 7) == F.E4M3_VALUES[c]


def test_e2m1_unpack_low_nibble_first():
    assert list(F.e2m1_unpack(np.array([0x21], dtype=np.uint8))) == [0x1, 0x2]
    assert list(F.e2m1_decode(F.e2m1_unpack(np.array([0x8F], dtype=np.uint8)))) == [-6.0, -0.0]


def test_e8m0_all_codes():
    c = np.arange(256)
    v = F.e8m0_decode(c)
    assert math.isnan(v[255])
    for code in range(255):
        assert v[code] == math.ldexp(1.0, code - 127)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(ref[:255], v[:255]) and math.isnan(ref[255])


def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 400000, dtype=np.uint64).astype(np.uint32)
    f32 = bits.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    # ties: bf16 values plus half an ulp, subnormals, near-overflow
    bf = (rng.integers(0, 2 ** 16, 50000, dtype=np.uint64).astype(np.uint32) << 16)
    ties = (bf | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    v = np.concatenate([f32, ties, np.float32([3.3961e38, -3.3961e38, 1e-40, -1e-45, 0.0, -0.0])])
    ref = torch.tensor(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.bf16_rne_bits(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_value_roundtrip():
    bits = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    vals = F.bf16_value(bits)
    finite = np.isfinite(vals)
    assert np.array_equal(F.bf16_rne_bits(vals[finite]), bits[finite])

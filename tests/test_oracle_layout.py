"""Pins for oracle/layout.py: inverses, padding values, fold decisions, -0 count."""
import numpy as np
import pytest

from oracle import layout as L


def rand_bytes(rng, shape):
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def test_e4m3_block_codes_roundtrip_and_padding():
    rng = np.random.default_rng(0)
    E, N, K = 2, 64, 2080
    w = rand_bytes(rng, (E, N, K))
    codes = rng.integers(118, 133, size=(E, N // 32, K // 32), dtype=np.uint8)
    p = L.pack_e4m3(w, codes)
    assert p["mode"] == "block" and p["Kp"] == 2176
    assert p["wq"].shape == (E, N, 2176) and np.all(p["wq"][:, :, K:] == 0)
    assert p["codes"].shape == (E, 2, 68) and np.all(p["codes"][:, :, 65:] == 128)
    w2, row = L.unpack_e4m3(p)
    assert np.array_equal(w2, w)
    assert np.array_equal(row, np.repeat(codes, 32, axis=1))
    # SF atoms hold the per-row codes; padded K blocks 128, padded rows 127
    back = L.sf_atoms_inverse(p["sf"], N, 68)
    assert np.array_equal(back[:, :, :65], row) and np.all(back[:, :, 65:] == 128)
    assert p["sf"].shape == (E, 1, 17, 512)
    assert np.all(p["sf"][:, 0, :, (100 % 32) * 16 + (100 // 32) * 4] == 127)  # row 100 >= N


def test_sf_atom_byte_position_by_hand():
    # row n = 37 (m = 37: m % 32 = 5, m // 32 = 1), K block j = 6 (kt 1, kb 2)
    codes = np.full((1, 128, 8), 120, dtype=np.uint8)
    codes[0, 37, 6] = 7
    atoms = L.sf_atoms(codes, 256)
    assert atoms.shape == (1, 1, 2, 512)
    assert atoms[0, 0, 1, 5 * 16 + 1 * 4 + 2] == 7
    assert np.count_nonzero(atoms != 120) == 1


def test_fold_decisions():
    rng = np.random.default_rng(1)
    E, N, K = 1, 96, 256
    w = rand_bytes(rng, (E, N, K))
    block = rng.integers(118, 133, size=(E, N // 32, K // 32), dtype=np.uint8)
    row = np.repeat(block, 32, axis=1)
    p = L.pack_e4m3(w, row)                           # rows agree: folds
    assert p["mode"] == "block" and np.array_equal(p["codes"][:, :, :8], block)
    assert L.pack_e4m3(w, row, fold=False)["mode"] == "row"
    bad = row.copy()
    bad[0, 40, 3] ^= 1                                # one row disagrees
    assert L.pack_e4m3(w, bad)["mode"] == "row"
    with pytest.raises(L.PackError) as ei:
        L.pack_e4m3(w, bad, require_block=True)
    assert ei.value.code == L.MX_ERR_NOT_BLOCK32
    # N not a multiple of 32 cannot fold
    p = L.pack_e4m3(w[:, :40], bad[:, :40])
    assert p["mode"] == "row"
    with pytest.raises(L.PackError) as ei:
        L.pack_e4m3(w, np.full_like(row, 255))
    assert ei.value.code == L.MX_ERR_SCALE


def test_e2m1_plain_order_and_atoms_by_positions():
    rng = np.random.default_rng(9)
    E, N, K = 2, 136, 160                    # two row tiles, ragged K (Kp = 256)
    w = (rng.integers(0, 256, size=(E, N, K // 2)) & 0x77).astype(np.uint8)   # no -0 nibbles
    codes = rng.integers(118, 133, size=(E, N, K // 32), dtype=np.uint8)
    p = L.pack_e2m1(w, codes)
    assert p["wq"].shape == (E, 2, 2, 128, 64) and p["sf"].shape == (E, 2, 2, 512)
    for e, n, k in [(0, 0, 0), (1, 5, 77), (0, 135, 159), (1, 129, 33)]:
        byte = int(p["wq"][e, n // 128, k // 128, n % 128, (k % 128) // 2])
        assert (byte >> (4 * (k % 2))) & 0xF == (int(w[e, n, k // 2]) >> (4 * (k % 2))) & 0xF
        m, rt = n % 128, n // 128
        j = k // 32
        assert p["sf"][e, rt, j // 4, (m % 32) * 16 + (m // 32) * 4 + j % 4] == codes[e, n, j]
    assert np.all(L.e2m1_rows(p)[:, :, K // 2:] == 0)
    assert np.all(p["wq"][:, 1, :, N - 128:] == 0)       # rows 136..255 of tile 1
    # K blocks 5..7 of the second step are padding (128); rows 136..255 of tile 1 are 127
    assert p["sf"][0, 0, 1, 1 * 4 + 1] == 128            # row 32, block 5
    assert p["sf"][1, 1, 0, (8 % 32) * 16] == 127         # row 136 >= N


def test_e2m1_roundtrip_padding_and_negative_zero_count():
    rng = np.random.default_rng(2)
    E, N, K = 3, 48, 2080
    w = rand_bytes(rng, (E, N, K // 2))
    codes = rng.integers(122, 131, size=(E, N, K // 32), dtype=np.uint8)
    p = L.pack_e2m1(w, codes)
    count = 0
    for byte in w.reshape(-1).tolist():
        count += (byte & 0xF) == 8
        count += (byte >> 4) == 8
    assert p["neg_zero_count"] == count
    back, c2 = L.unpack_e2m1(p)
    assert np.array_equal(back, L.drop_negative_zero(w))
    assert np.array_equal(c2, codes)
    assert np.all(p["codes"][:, :, K // 32:] == 128)
    assert not np.any((p["wq"] & 0x0F) == 0x08) and not np.any((p["wq"] & 0xF0) == 0x80)
    # the padded tail past K/2 bytes is zero
    assert np.all(L.e2m1_rows(p)[:, :, K // 2:] == 0)


def test_gate_up_interleave_rows_and_inverse():
    from oracle import layout as L
    src = L.gate_up_source_rows(48)          # I = 24
    assert src[:8].tolist() == list(range(8))            # gate rows 0..7
    assert src[8:16].tolist() == list(range(24, 32))     # up rows 0..7
    assert src[16:24].tolist() == list(range(8, 16))     # gate rows 8..15
    assert sorted(src.tolist()) == list(range(48))
    rng = np.random.default_rng(9)
    w = rng.integers(0, 256, size=(2, 48, 80), dtype=np.uint8)
    c = rng.integers(118, 133, size=(2, 48, 5), dtype=np.uint8)
    p = L.pack_e2m1(w, c, gate_up=True)
    plain = L.pack_e2m1(w[:, src], c[:, src])
    assert np.array_equal(p["wq"], plain["wq"]) and np.array_equal(p["codes"], plain["codes"])
    assert np.array_equal(p["sf"], plain["sf"])
    back, cb = L.unpack_e2m1(p)
    assert np.array_equal(back, L.drop_negative_zero(w)) and np.array_equal(cb, c)
    with pytest.raises(L.PackError):
        L.pack_e2m1(w[:, :40], c[:, :40], gate_up=True)

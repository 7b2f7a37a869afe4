"""The library's packed weight layout, written as plain index maps.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The layout is this library's own design (the pages' gfx942/gfx950 shuffles are
prior art), so every map here is "parity unpinned" against the pages; the
pages fix only the semantics the maps must keep:

* K is zero-padded to a multiple of 128 and a padded block gets code 128
  (weights942, ``dense_copy``).
* Row codes [N, K/32] fold to 32x32 block codes [N/32, K/32] exactly when every
  32 consecutive rows agree (rocm_native ``_as_block32_scale``); when they do
  not, weights942 ``linear_copy`` refuses, and rocm_native keeps row codes.
* -0 nibbles (0x8) are rewritten to +0 and counted (weights942,
  ``fp4_drop_negative_zero_``).
* Each K block keeps its code when bytes move within a row (weights942,
  ``fp4_lane_major``).

Packed E4M3 weight (dense MXFP8), E experts of [N, K]:
  wq     [E, N, Kp]           row-major bytes, zero past K
  codes  [E, N/32, Kp/32]     block mode, or [E, N, Kp/32] row mode; 128 past K
  sf     [E, ceil(N/128), Kp/128, 512]   per-row codes in 512-byte atoms: row
         n = 128 rt + m and K block j = 4 kt + kb sit at byte
         (m % 32) * 16 + (m // 32) * 4 + kb of atom (rt, kt); rows past N
         hold 127, blocks past K hold 128.

Packed E2M1 weight (MXFP4 experts), E experts of [N, K]:
  wq     [E, ceil(N/128), Kp/128, 128, 64]   128-row x 128-value tiles: tile
         (rt, kt) row m holds values 128 kt .. 128 kt + 127 of row 128 rt + m
         as 64 fp4x2 bytes in the input order (element 2i in the low nibble of
         byte i); zero past K and past N; -0 nibbles are +0
  codes  [E, N, Kp/32]  per-row codes (32x32 block codes are expanded), 128
         past K
  sf     [E, ceil(N/128), Kp/128, 512]   the per-row codes in atoms, as for E4M3
  gate / up experts (w13 [E, 2 I, K/2], gate rows then up rows, weights942
  ``moe_copies``) can be packed with their halves interleaved in 8-row groups:
  packed row 16 q + i holds gate row 8 q + i for i < 8 and up row
  8 q + i - 8 for i >= 8 (codes and atoms alike), so a 32-row slice of the
  accumulator holds the gate and up rows of the same 16 intermediate indices
  (lane l and lane l + 8).  (The page's gfx942 copy interleaves single rows,
  2 i and 2 i + 1, for its own MFMA fragment.)

Pinned by tests/test_oracle_layout.py: unpack(pack(w)) == w, the padding
values, the fold / refuse decisions on agreeing and disagreeing rows, and the
-0 count against a per-nibble Python count.
"""
import numpy as np

KSTEP = 128          # K is padded to a multiple of this
PAD_CODE = 128       # code of a padded K block
PAD_ROW_CODE = 127   # code of a row past N inside an SF atom
ATOM_ROWS = 128
ATOM_BLOCKS = 4
ATOM_BYTES = 512

MX_ERR_SHAPE = 1
MX_ERR_SCALE = 5
MX_ERR_NOT_BLOCK32 = 4


class PackError(ValueError):
    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


def padded_k(K: int) -> int:
    return -(-K // KSTEP) * KSTEP


def fold_block_codes(row_codes: np.ndarray):
    """[E, N, K/32] row codes -> [E, N/32, K/32] block codes, or None when N is
    not a multiple of 32 or some 32-row group disagrees (rocm_native,
    ``_as_block32_scale``)."""
    E, N, KB = row_codes.shape
    if N % 32 != 0:
        return None
    groups = row_codes.reshape(E, N // 32, 32, KB)
    if not np.array_equal(groups, np.broadcast_to(groups[:, :, :1], groups.shape)):
        return None
    return groups[:, :, 0].copy()


def expand_block_codes(block_codes: np.ndarray, N: int) -> np.ndarray:
    """[E, N/32, KB] -> [E, N, KB]: each block code repeated over its 32 rows."""
    return np.repeat(block_codes, 32, axis=1)[:, :N]


def sf_atoms(row_codes: np.ndarray, Kp: int) -> np.ndarray:
    """Per-row codes [E, R, KB] (KB <= Kp/32) -> atoms [E, ceil(R/128), Kp/128, 512]."""
    E, R, KB = row_codes.shape
    RT = -(-R // ATOM_ROWS)
    KT = Kp // KSTEP
    out = np.empty((E, RT, KT, ATOM_BYTES), dtype=np.uint8)
    for rt in range(RT):
        for m in range(ATOM_ROWS):
            n = rt * ATOM_ROWS + m
            for kt in range(KT):
                for kb in range(ATOM_BLOCKS):
                    j = kt * ATOM_BLOCKS + kb
                    if n >= R:
                        c = PAD_ROW_CODE
                    elif j >= KB:
                        c = PAD_CODE
                    else:
                        c = row_codes[:, n, j]
                    out[:, rt, kt, (m % 32) * 16 + (m // 32) * 4 + kb] = c
    return out


def sf_atoms_inverse(atoms: np.ndarray, R: int, KB: int) -> np.ndarray:
    """Atoms -> per-row codes [E, R, KB] (drops padding)."""
    E = atoms.shape[0]
    out = np.empty((E, R, KB), dtype=np.uint8)
    for n in range(R):
        rt, m = divmod(n, ATOM_ROWS)
        for j in range(KB):
            kt, kb = divmod(j, ATOM_BLOCKS)
            out[:, n, j] = atoms[:, rt, kt, (m % 32) * 16 + (m // 32) * 4 + kb]
    return out


def _pad_codes(codes: np.ndarray, KBp: int) -> np.ndarray:
    E, R, KB = codes.shape
    out = np.full((E, R, KBp), PAD_CODE, dtype=np.uint8)
    out[:, :, :KB] = codes
    return out


def pack_e4m3(w, codes, fold: bool = True, require_block: bool = False) -> dict:
    """Dense MXFP8 weight: bytes [E, N, K], codes [E, N/32, K/32] (block) or
    [E, N, K/32] (row) -> packed dict (see module text)."""
    w = np.asarray(w, dtype=np.uint8)
    codes = np.asarray(codes, dtype=np.uint8)
    E, N, K = w.shape
    if K % 32 != 0 or N < 1 or K < 32:
        raise PackError(MX_ERR_SHAPE, "K must be a positive multiple of 32")
    if np.any(codes == 255):
        raise PackError(MX_ERR_SCALE, "E8M0 code 255 (NaN) in the weight scales")
    KB = K // 32
    Kp = padded_k(K)
    if N % 32 == 0 and codes.shape == (E, N // 32, KB) and N // 32 != N:
        block = codes
    elif codes.shape == (E, N, KB):
        block = fold_block_codes(codes) if (fold or require_block) else None
        if block is None and require_block:
            raise PackError(MX_ERR_NOT_BLOCK32, "row scales are not 32 x 32 blocks")
    else:
        raise PackError(MX_ERR_SHAPE, f"codes shape {codes.shape} does not fit w {w.shape}")
    wq = np.zeros((E, N, Kp), dtype=np.uint8)
    wq[:, :, :K] = w
    if block is not None:
        mode = "block"
        codes_c = _pad_codes(block, Kp // 32)
        row = expand_block_codes(block, N)
    else:
        mode = "row"
        codes_c = _pad_codes(codes, Kp // 32)
        row = codes
    return {"fmt": "e4m3", "mode": mode, "E": E, "N": N, "K": K, "Kp": Kp,
            "wq": wq, "codes": codes_c, "sf": sf_atoms(row, Kp)}


def unpack_e4m3(p: dict) -> tuple:
    """Inverse of pack_e4m3: (bytes [E, N, K], row codes [E, N, K/32])."""
    N, K = p["N"], p["K"]
    w = p["wq"][:, :, :K].copy()
    c = p["codes"][:, :, : K // 32]
    row = expand_block_codes(c, N) if p["mode"] == "block" else c.copy()
    return w, row


def count_negative_zero(w) -> int:
    w = np.asarray(w, dtype=np.uint8)
    return int(np.count_nonzero((w & 0x0F) == 0x08) + np.count_nonzero((w & 0xF0) == 0x80))


def drop_negative_zero(w) -> np.ndarray:
    """Rewrite every 0x8 nibble to 0x0 (weights942, ``fp4_drop_negative_zero_``)."""
    w = np.asarray(w, dtype=np.uint8).copy()
    lo = (w & 0x0F) == 0x08
    w = np.where(lo, w & 0xF0, w)
    hi = (w & 0xF0) == 0x80
    return np.where(hi, w & 0x0F, w).astype(np.uint8)


def gate_up_source_rows(N: int) -> np.ndarray:
    """Packed row r -> source row of a gate-then-up [2 I = N] expert tensor
    under the 8-row-group interleave (see module text)."""
    if N % 16 != 0:
        raise PackError(MX_ERR_SHAPE, "gate/up interleave needs 2 I a multiple of 16")
    r = np.arange(N)
    q, i = r // 16, r % 16
    return np.where(i < 8, 8 * q + i, N // 2 + 8 * q + i - 8)


def pack_e2m1(w, codes, gate_up: bool = False) -> dict:
    """MXFP4 experts: bytes [E, N, K/2] (fp4x2, low nibble first), codes
    [E, N, K/32] or [E, N/32, K/32] -> packed dict (see module text).
    ``gate_up``: interleave the gate and up halves (see module text)."""
    w = np.asarray(w, dtype=np.uint8)
    codes = np.asarray(codes, dtype=np.uint8)
    E, N, KH = w.shape
    K = 2 * KH
    if K % 32 != 0 or K < 32 or N < 1:
        raise PackError(MX_ERR_SHAPE, "K must be a positive multiple of 32")
    if np.any(codes == 255):
        raise PackError(MX_ERR_SCALE, "E8M0 code 255 (NaN) in the weight scales")
    KB = K // 32
    if codes.shape == (E, N, KB):
        row = codes
    elif N % 32 == 0 and codes.shape == (E, N // 32, KB):
        row = expand_block_codes(codes, N)
    else:
        raise PackError(MX_ERR_SHAPE, f"codes shape {codes.shape} does not fit w {w.shape}")
    if gate_up:
        src = gate_up_source_rows(N)
        w, row = w[:, src], row[:, src]
    Kp = padded_k(K)
    negz = count_negative_zero(w)
    clean = drop_negative_zero(w)
    RT, KT = -(-N // ATOM_ROWS), Kp // KSTEP
    padded = np.zeros((E, RT * ATOM_ROWS, Kp // 2), dtype=np.uint8)
    padded[:, :N, :KH] = clean
    tiles = padded.reshape(E, RT, ATOM_ROWS, KT, KSTEP // 2).transpose(0, 1, 3, 2, 4).copy()
    return {"fmt": "e2m1", "mode": "row", "E": E, "N": N, "K": K, "Kp": Kp,
            "wq": tiles, "codes": _pad_codes(row, Kp // 32), "sf": sf_atoms(row, Kp),
            "neg_zero_count": negz, "gate_up": bool(gate_up)}


def e2m1_rows(p: dict) -> np.ndarray:
    """Packed E2M1 tiles -> rows [E, N, Kp/2] (packed row order)."""
    E, RT, KT = p["wq"].shape[:3]
    rows = p["wq"].transpose(0, 1, 3, 2, 4).reshape(E, RT * ATOM_ROWS, KT * KSTEP // 2)
    return rows[:, : p["N"]]


def unpack_e2m1(p: dict) -> tuple:
    """Inverse of pack_e2m1 (up to -0 -> +0): (bytes [E, N, K/2], codes [E, N, K/32])."""
    K = p["K"]
    back = e2m1_rows(p)[:, :, : K // 2]
    codes = p["codes"][:, :, : K // 32]
    if p.get("gate_up"):
        src = gate_up_source_rows(p["N"])
        w, c = np.empty_like(back), np.empty_like(codes)
        w[:, src], c[:, src] = back, codes
        return w, c
    return back.copy(), codes.copy()

"""Pins for oracle/moe.py: routing vs Python's stable sort, E=1/top-1 vs an exact
rational A16W4 brute force, permutation invariance and -0 / +0 equivalence."""
import collections
import os
from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle.moe import MX_ERR_EXPERT_ID, moe_linear, route

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_ocp.txt")


def e2m1_table():
    t = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            c, v = line.split()
            t[int(c)] = Fraction(float(v))
    return t


def test_route_matches_stable_sort():
    rng = np.random.default_rng(0)
    T, topk, E = 37, 5, 11
    ids = rng.integers(-1, E, size=(T, topk))
    r = route(ids, E)
    flat = ids.reshape(-1).tolist()
    order = sorted((p for p in range(T * topk) if flat[p] >= 0), key=lambda p: flat[p])
    assert r["pairs"].tolist() == order
    cnt = collections.Counter(v for v in flat if v >= 0)
    assert r["counts"].tolist() == [cnt.get(e, 0) for e in range(E)]
    assert r["offsets"][-1] == len(order)
    assert r["active"].tolist() == sorted(cnt)
    assert r["status"] == 0
    ids[3, 2] = E        # out of range: error status, pair skipped
    ids[4, 0] = -7
    r2 = route(ids, E)
    assert r2["status"] == MX_ERR_EXPERT_ID
    assert 3 * topk + 2 not in r2["pairs"].tolist() and 4 * topk not in r2["pairs"].tolist()


def test_single_expert_top1_is_a16w4_linear_exact():
    rng = np.random.default_rng(1)
    T, N, K = 3, 4, 64
    x = F.bf16_value(F.bf16_rne_bits(rng.standard_normal((T, K))))
    w = rng.integers(0, 256, size=(1, N, K // 2), dtype=np.uint8)
    codes = rng.integers(122, 131, size=(1, N, K // 32), dtype=np.uint8)
    y = moe_linear(x, np.zeros((T, 1), dtype=np.int32), w, codes)
    tab = e2m1_table()
    for t in range(T):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                byte = int(w[0, n, k // 2])
                nib = byte & 0xF if k % 2 == 0 else byte >> 4
                acc += tab[nib] * Fraction(2) ** (int(codes[0, n, k // 32]) - 127) * Fraction(x[t, k])
            assert abs(float(acc) - y[t, 0, n]) <= 1e-13 * max(1.0, abs(float(acc)))


def test_token_permutation_and_negative_zero():
    rng = np.random.default_rng(2)
    T, E, N, K, topk = 9, 6, 32, 128, 3
    x = F.bf16_value(F.bf16_rne_bits(rng.standard_normal((T, K))))
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    ids[2, 1] = -1
    w = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    codes = rng.integers(122, 131, size=(E, N, K // 32), dtype=np.uint8)
    y = moe_linear(x, ids, w, codes)
    assert np.all(y[2, 1] == 0)
    perm = rng.permutation(T)
    yp = moe_linear(x[perm], ids[perm], w, codes)
    assert np.array_equal(yp, y[perm])
    # +0 nibbles rewritten to -0 give the same products
    wneg = w.copy()
    lo0 = (wneg & 0x0F) == 0
    wneg[lo0] |= 0x08
    hi0 = (wneg & 0xF0) == 0
    wneg[hi0] |= 0x80
    assert np.array_equal(moe_linear(x, ids, wneg, codes), y)


# ---------------------------------------------------------------- full expert

def test_silu_matches_torch_cpu():
    import torch
    v = np.concatenate([np.linspace(-40, 40, 2001), [-700.0, -50.0, 0.0, 50.0, 700.0]])
    from oracle.moe import silu
    ref = torch.nn.functional.silu(torch.tensor(v, dtype=torch.float64)).numpy()
    assert np.allclose(silu(v), ref, rtol=1e-15, atol=1e-300)
    assert silu(np.array([0.0]))[0] == 0.0


def _table_dequant(w, codes):
    """[N, K/2] fp4x2 bytes + [N, K/32] codes -> fp64 [N, K] from the OCP table fixture."""
    tab = e2m1_table()
    N, KH = w.shape
    out = np.empty((N, 2 * KH))
    for n in range(N):
        for k in range(2 * KH):
            byte = int(w[n, k // 2])
            nib = byte & 0xF if k % 2 == 0 else byte >> 4
            out[n, k] = float(tab[nib]) * 2.0 ** (int(codes[n, k // 32]) - 127)
    return out


def _expert_case(seed, T=3, topk=2, E=3, I=32, K=64, H=48):
    rng = np.random.default_rng(seed)
    x = F.bf16_value(F.bf16_rne_bits(rng.standard_normal((T, K))))
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, topk))
    w13 = rng.integers(0, 256, size=(E, 2 * I, K // 2), dtype=np.uint8)
    c13 = rng.integers(122, 131, size=(E, 2 * I, K // 32), dtype=np.uint8)
    w2 = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    c2 = rng.integers(122, 131, size=(E, H, I // 32), dtype=np.uint8)
    return x, ids, wts, w13, c13, w2, c2


def test_expert_single_expert_matches_torch_chain():
    import torch
    from oracle.moe import moe_expert
    x, _, _, w13, c13, w2, c2 = _expert_case(2, E=1)
    T, I = x.shape[0], w13.shape[1] // 2
    ids = np.zeros((T, 1), dtype=np.int32)
    wts = np.full((T, 1), 0.75)
    r = moe_expert(x, ids, wts, w13, c13, w2, c2)
    W13 = torch.tensor(_table_dequant(w13[0], c13[0]))
    W2 = torch.tensor(_table_dequant(w2[0], c2[0]))
    xt = torch.tensor(x)
    g, u = xt @ W13[:I].T, xt @ W13[I:].T
    act = torch.nn.functional.silu(g) * u
    # bf16 rounding of act: compare within one bf16 ulp, then feed the oracle's
    # rounded act to the down projection
    # bf16 spacing at |act|, never below the subnormal spacing 2^-133
    ulp = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(act.numpy()), 1e-300))) - 7), 2.0 ** -133)
    assert np.all(np.abs(r["act"][:, 0] - act.numpy()) <= ulp)
    out = 0.75 * (torch.tensor(r["act"][:, 0]) @ W2.T)
    assert np.allclose(r["out"], out.numpy(), rtol=1e-12, atol=1e-12 * np.abs(out.numpy()).max())


def test_expert_gate_and_up_roles():
    from oracle.moe import moe_expert, silu
    x, ids, wts, w13, c13, w2, c2 = _expert_case(3)
    I = w13.shape[1] // 2
    up0 = w13.copy()
    up0[:, I:] = 0                          # up = 0 -> act = 0 -> out = 0
    assert np.all(moe_expert(x, ids, wts, up0, c13, w2, c2)["out"] == 0.0)
    gate0 = w13.copy()
    gate0[:, :I] = 0                        # silu(0) = 0 -> act = 0
    assert np.all(moe_expert(x, ids, wts, gate0, c13, w2, c2)["out"] == 0.0)
    r = moe_expert(x, ids, wts, w13, c13, w2, c2)
    g, u = r["y13"][:, :, :I], r["y13"][:, :, I:]
    assert np.array_equal(r["act"], F.bf16_value(F.bf16_rne_bits(silu(g) * u)))


def test_expert_slot_permutation_weights_and_invalid_ids():
    from oracle.moe import moe_expert
    x, ids, wts, w13, c13, w2, c2 = _expert_case(4, topk=3, E=4)
    base = moe_expert(x, ids, wts, w13, c13, w2, c2)["out"]
    perm = [2, 0, 1]
    p = moe_expert(x, ids[:, perm], wts[:, perm], w13, c13, w2, c2)["out"]
    assert np.allclose(p, base, rtol=1e-13, atol=1e-13 * np.abs(base).max())
    d = moe_expert(x, ids, 2.0 * wts, w13, c13, w2, c2)["out"]
    assert np.array_equal(d, 2.0 * base)    # power-of-two scaling is exact
    ids_bad = ids.copy()
    ids_bad[:, 1] = -1
    wts0 = wts.copy()
    wts0[:, 1] = 0.0
    assert np.array_equal(moe_expert(x, ids_bad, wts, w13, c13, w2, c2)["out"],
                          moe_expert(x, ids, wts0, w13, c13, w2, c2)["out"])


def test_w4a8_single_expert_top1_exact():
    """W4A8 at E = 1, top-1: the exact rational sum of e2m1(w) 2^(cw-127) times
    the quantized activation, its e4m3 bytes decoded by torch (not by the
    oracle's decoder)."""
    import torch
    from oracle.moe import moe_linear_w4a8
    rng = np.random.default_rng(11)
    T, N, K = 3, 4, 64
    x = F.bf16_value(F.bf16_rne_bits(rng.standard_normal((T, K)) * 3.0))
    w = rng.integers(0, 256, size=(1, N, K // 2), dtype=np.uint8)
    codes = rng.integers(122, 131, size=(1, N, K // 32), dtype=np.uint8)
    r = moe_linear_w4a8(x, np.zeros((T, 1), dtype=np.int32), w, codes)
    qv = torch.tensor(r["xq"].astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = e2m1_table()
    for t in range(T):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                byte = int(w[0, n, k // 2])
                nib = byte & 0xF if k % 2 == 0 else byte >> 4
                a = Fraction(float(qv[t, k])) * Fraction(2) ** (int(r["xcodes"][t, k // 32]) - 127)
                acc += tab[nib] * Fraction(2) ** (int(codes[0, n, k // 32]) - 127) * a
            assert abs(float(acc) - r["y"][t, 0, n]) <= 1e-13 * max(1.0, abs(float(acc)))


def test_w4a8_equals_a16w4_on_exactly_representable_activations():
    """An activation that MXFP8 represents exactly (every block: e4m3 values
    under one scale whose largest magnitude is 256..448, so the quantizer
    keeps that scale) gives the same W4A8 and A16W4 outputs."""
    from oracle.moe import moe_linear_w4a8
    rng = np.random.default_rng(12)
    T, E, N, K, topk = 5, 3, 6, 96, 2
    vals = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    ok = np.isfinite(vals) & (np.abs(vals) <= 448)
    pool = vals[ok]
    x = rng.choice(pool, size=(T, K))
    blocks = x.reshape(T, K // 32, 32)
    blocks[:, :, 0] = 448.0 * np.where(rng.random((T, K // 32)) < 0.5, -1, 1)   # block max 448
    scale = np.ldexp(1.0, rng.integers(-3, 4, size=(T, K // 32)))
    x = (blocks * scale[..., None]).reshape(T, K)
    w = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    codes = rng.integers(120, 133, size=(E, N, K // 32), dtype=np.uint8)
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    r = moe_linear_w4a8(x, ids, w, codes)
    assert np.array_equal(r["A"], x)                      # the quantization is exact here
    y16 = moe_linear(x, ids, w, codes)
    assert np.allclose(r["y"], y16, rtol=1e-12, atol=0.0)

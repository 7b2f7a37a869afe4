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

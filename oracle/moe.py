"""Token -> expert routing and the routed A16W4 expert linear, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The expert weights are MXFP4: fp4x2 bytes [E, N, K/2], low nibble first, with
per-row E8M0 codes [E, N, K/32] (weights942, ``moe_copies``; a16w4 module
text).  The A16W4 product dequantizes each e2m1 value with its scale to bf16
and multiplies by the bf16 token activation (a16w4, ``dequant`` /
``step_mfma``):

    y[t, j, n] = sum_k bf16(e2m1(W_e[n, k]) 2^(c_e[n, k/32] - 127)) x[t, k],
    e = topk_ids[t, j]

Routing is the plainest reading of "routed experts" (the pages show no router):
pairs p = t * topk + j are grouped by expert id, in increasing (t, j) order
within an expert; ids of -1 are skipped and their outputs are zero; any other
id outside [0, E) is an error and is skipped the same way.  Routing weights
are not applied (the gate/up GEMM output is per (token, slot)).

Pinned by tests/test_oracle_moe.py: E = 1 / top-1 reduces to a dense A16W4
linear checked by exact rational brute force, invariance under permuting the
tokens, -0 and +0 nibbles giving identical outputs (weights942,
``fp4_drop_negative_zero_``), and routing against Python's stable sort.
"""
import numpy as np

from .formats import bf16_rne_bits, bf16_value
from .linear import dequant_values

MX_ERR_EXPERT_ID = 7


def route(topk_ids, E: int) -> dict:
    """topk_ids int [T, topk] -> counts [E], offsets [E+1], pairs (sorted
    p = t*topk + j), active (experts with count > 0, ascending), status."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    flat = ids.reshape(-1)
    bad = (flat != -1) & ((flat < 0) | (flat >= E))
    valid = (flat >= 0) & (flat < E)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat[valid]:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    pairs = np.zeros(int(offsets[-1]), dtype=np.int64)
    fill = offsets[:-1].copy()
    for p in range(T * topk):          # increasing (t, j): stable within an expert
        if valid[p]:
            e = flat[p]
            pairs[fill[e]] = p
            fill[e] += 1
    active = np.nonzero(counts)[0]
    status = MX_ERR_EXPERT_ID if np.any(bad) else 0
    return {"counts": counts, "offsets": offsets, "pairs": pairs,
            "active": active, "status": status}


def dequant_experts_bf16(w_bytes, codes) -> np.ndarray:
    """[E, N, K/2] bytes, [E, N, K/32] codes -> bf16-rounded fp64 weights [E, N, K]."""
    w_bytes = np.asarray(w_bytes, dtype=np.uint8)
    E, N, KH = w_bytes.shape
    K = 2 * KH
    out = np.empty((E, N, K), dtype=np.float64)
    for e in range(E):
        out[e] = bf16_value(bf16_rne_bits(dequant_values(w_bytes[e], codes[e], "e2m1", N, K)))
    return out


def moe_linear(x, topk_ids, w_bytes, codes, wdeq=None) -> np.ndarray:
    """x fp64 [T, K] (bf16 values) -> y fp64 [T, topk, N].  ``wdeq`` may pass a
    precomputed ``dequant_experts_bf16`` result."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    E, N = np.asarray(w_bytes).shape[:2]
    W = dequant_experts_bf16(w_bytes, codes) if wdeq is None else wdeq
    y = np.zeros((T, topk, N), dtype=np.float64)
    for t in range(T):
        for j in range(topk):
            e = ids[t, j]
            if 0 <= e < E:
                y[t, j] = W[e] @ x[t]
    return y

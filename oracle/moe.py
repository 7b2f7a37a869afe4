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

The full routed expert (``moe_expert``) follows the tensors weights942
``moe_copies`` describes: w13 [E, 2 I, K/2] with the I gate rows first, then
the I up rows, and w2 [E, H, I/2].  Readings where the pages are silent:

* the gated activation is SiLU-and-mul: act = silu(gate) * up, silu(v) =
  v / (1 + e^-v);
* act is rounded to bf16 before the down projection (the down GEMM is A16W4
  too: bf16 activations times MXFP4 weights);
* the routing weights scale each slot's down-projection row and the top-k
  slots are summed: out[t] = sum_j weight[t, j] y2[t, j]; slots whose id is
  not a valid expert contribute nothing.

``moe_linear_w4a8`` is the same routed GEMM with the activation quantized per
token to MXFP8 first (MXFP4 x MXFP8).

Pinned by tests/test_oracle_moe.py: E = 1 / top-1 reduces to a dense A16W4
linear checked by exact rational brute force, invariance under permuting the
tokens, -0 and +0 nibbles giving identical outputs (weights942,
``fp4_drop_negative_zero_``), routing against Python's stable sort; silu
against torch's CPU ``silu``; the full expert at E = 1 / top-1 against the
same chain in torch CPU ops on a table-decoded weight; gate / up roles,
slot permutation, linearity in the routing weights and skipped invalid slots;
W4A8 at E = 1 / top-1 against an exact rational sum over torch's e4m3
decode, and equal to A16W4 on activations that MXFP8 represents exactly.
"""
import numpy as np

from .formats import bf16_rne_bits, bf16_value, e4m3_decode
from .linear import dequant_values, expand_codes
from .quant import quantize_act

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


def moe_linear_w4a8(x, topk_ids, w_bytes, codes) -> dict:
    """The routed expert GEMM with MXFP8 activations (the prefill form of the
    layer: MXFP4 weights times per-token MXFP8-quantized activations, as the
    dense MXFP8 linear quantizes its input -- rocm_native, _quant_mxfp8_tile).
    x fp64 [T, K] (bf16 values) is quantized per token with the block
    quantizer of quant.quantize_act; then, in fp64,

        y[t, j, n] = sum_k e2m1(W_e[n, k]) 2^(c_e[n, k/32] - 127)
                           e4m3(q[t, k]) 2^(cx[t, k/32] - 127).

    Returns dict(y=[T, topk, N], A=[T, K] dequantized activation,
    xq, xcodes)."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    w_bytes = np.asarray(w_bytes, dtype=np.uint8)
    E, N, KH = w_bytes.shape
    K = 2 * KH
    xq, xcodes = quantize_act(x)
    A = e4m3_decode(xq) * expand_codes(xcodes, T, K)
    y = np.zeros((T, topk, N), dtype=np.float64)
    W = {}
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            if 0 <= e < E:
                if e not in W:
                    W[e] = dequant_values(w_bytes[e], codes[e], "e2m1", N, K)
                y[t, j] = W[e] @ A[t]
    return {"y": y, "A": A, "xq": xq, "xcodes": xcodes}


def silu(v) -> np.ndarray:
    """SiLU in fp64: v / (1 + e^-v) (-> 0 for v -> -inf, -> v for v -> +inf)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def moe_expert(x, topk_ids, topk_weights, w13_bytes, w13_codes, w2_bytes, w2_codes) -> dict:
    """The routed expert MLP, fp64.

    x [T, K] (bf16 values), topk_ids [T, topk], topk_weights [T, topk];
    w13 bytes [E, 2 I, K/2] (gate rows 0..I-1, up rows I..2I-1) with per-row
    codes [E, 2 I, K/32]; w2 bytes [E, H, I/2] with codes [E, H, I/32].

    Returns dict(out [T, H], act [T, topk, I] (bf16 values), y13 [T, topk, 2I],
    y2 [T, topk, H])."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    wts = np.asarray(topk_weights, dtype=np.float64)
    T, topk = ids.shape
    E, I2 = np.asarray(w13_bytes).shape[:2]
    I = I2 // 2
    H = np.asarray(w2_bytes).shape[1]
    y13 = moe_linear(x, ids, w13_bytes, w13_codes)                 # [T, topk, 2I]
    act = bf16_value(bf16_rne_bits(silu(y13[:, :, :I]) * y13[:, :, I:]))
    W2 = dequant_experts_bf16(w2_bytes, w2_codes)                  # [E, H, I]
    y2 = np.zeros((T, topk, H), dtype=np.float64)
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(topk):
            e = ids[t, j]
            if 0 <= e < E:
                y2[t, j] = W2[e] @ act[t, j]
                out[t] += wts[t, j] * y2[t, j]
    return {"out": out, "act": act, "y13": y13, "y2": y2}

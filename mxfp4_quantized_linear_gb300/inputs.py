"""Seeded synthetic workloads shaped like the decode, MoE and prefill layers.

This module only draws random numbers (CPU ``torch.Generator``, fixed seed,
fixed draw order) and returns plain CPU tensors; it holds none of the MX
method's arithmetic.  Tests feed the same tensors to the CUDA library and to
the CPU oracle; ``bench.py`` uses them for timing.

Recipes (seed 0 unless stated, draws in the order listed):

* e4m3 weight bytes: uniform over the 254 non-NaN codes (0x7F, 0xFF excluded)
* E8M0 codes: uniform integers in an inclusive range (e.g. 118..132)
* bf16 activations: N(0, 1) drawn in fp32, cast to bf16
* fp4x2 expert bytes: uniform bytes (so uniform nibbles, -0 included; the
  packer rewrites -0 to +0)
* top-k expert ids: per token the first ``topk`` entries of a random
  permutation of the E experts (distinct experts)

A generator made for a CUDA device draws there (same recipes, another
stream of numbers): the benchmark uses that for the multi-GB expert sweep,
whose inputs never go to the oracle.
"""
import torch


def generator(seed: int = 0, device=None) -> torch.Generator:
    g = torch.Generator() if device is None else torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def e4m3_bytes(shape, g: torch.Generator) -> torch.Tensor:
    r = torch.randint(0, 254, tuple(shape), generator=g, dtype=torch.int32, device=g.device)
    r = r + (r >= 0x7F).to(torch.int32)          # skip 0x7F; 0xFF is never reached
    return r.to(torch.uint8)


def e8m0_codes(shape, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32, device=g.device).to(torch.uint8)


def bf16_normal(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=g.device).to(torch.bfloat16)


def fp4x2_bytes(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randint(0, 256, tuple(shape), generator=g, dtype=torch.int32, device=g.device).to(torch.uint8)


def topk_ids(T: int, E: int, topk: int, g: torch.Generator) -> torch.Tensor:
    out = torch.empty((T, topk), dtype=torch.int32, device=g.device)
    for t in range(T):
        out[t] = torch.randperm(E, generator=g, device=g.device)[:topk].to(torch.int32)
    return out


# ---------------------------------------------------------------- workloads

def gemv_small(seed: int = 0) -> dict:
    """MXFP8 GEMV M=1, N=512, K=1024, 1x32 row codes 120..130."""
    g = generator(seed)
    N, K, M = 512, 1024, 1
    w = e4m3_bytes((N, K), g)
    codes = e8m0_codes((N, K // 32), 120, 130, g)
    x = bf16_normal((M, K), g)
    return {"w": w, "codes": codes, "x": x, "N": N, "K": K}


def decode_linear(K: int = 2048, Ms=(1, 4, 16, 32), N: int = 7168, seed: int = 0) -> dict:
    """MXFP8 decode linear N=7168, K=2048 (or 2080), 32x32 block codes
    118..132, activations at each M in ``Ms``."""
    g = generator(seed)
    w = e4m3_bytes((N, K), g)
    codes = e8m0_codes((N // 32, K // 32), 118, 132, g)
    xs = {M: bf16_normal((M, K), g) for M in Ms}
    return {"w": w, "codes": codes, "xs": xs, "N": N, "K": K}


def moe_gate_up(E: int = 64, N: int = 4096, K: int = 4096, T: int = 64, topk: int = 8,
                code_lo: int = 122, code_hi: int = 130, seed: int = 0, device=None) -> dict:
    """MXFP4 A16W4 MoE gate/up: w13 [E, N, K/2], per-row codes, T tokens top-k."""
    g = generator(seed, device)
    w = fp4x2_bytes((E, N, K // 2), g)
    codes = e8m0_codes((E, N, K // 32), code_lo, code_hi, g)
    x = bf16_normal((T, K), g)
    ids = topk_ids(T, E, topk, g)
    return {"w": w, "codes": codes, "x": x, "ids": ids, "E": E, "N": N, "K": K,
            "T": T, "topk": topk}


def moe_expert(E: int = 64, I: int = 2048, H: int = 4096, T: int = 64, topk: int = 8,
               code_lo: int = 122, code_hi: int = 130, seed: int = 0, device=None) -> dict:
    """MXFP4 routed expert MLP: w13 [E, 2 I, H/2] (gate rows, then up rows) and
    w2 [E, H, I/2] with per-row codes, x [T, H], top-k ids and routing weights
    (uniform draws, each token's row divided by its sum)."""
    g = generator(seed, device)
    w13 = fp4x2_bytes((E, 2 * I, H // 2), g)
    c13 = e8m0_codes((E, 2 * I, H // 32), code_lo, code_hi, g)
    w2 = fp4x2_bytes((E, H, I // 2), g)
    c2 = e8m0_codes((E, H, I // 32), code_lo, code_hi, g)
    x = bf16_normal((T, H), g)
    ids = topk_ids(T, E, topk, g)
    u = torch.rand((T, topk), generator=g, dtype=torch.float32, device=g.device)
    wts = u / u.sum(dim=1, keepdim=True)
    return {"w13": w13, "c13": c13, "w2": w2, "c2": c2, "x": x, "ids": ids, "weights": wts,
            "E": E, "I": I, "H": H, "T": T, "topk": topk}


def prefill_gemm(M: int = 4096, N: int = 7168, K: int = 7168, seed: int = 0) -> dict:
    """MXFP8 prefill GEMM: bf16 x [M, K], e4m3 W [N, K], 32x32 codes 118..132."""
    g = generator(seed)
    x = bf16_normal((M, K), g)
    w = e4m3_bytes((N, K), g)
    codes = e8m0_codes((N // 32, K // 32), 118, 132, g)
    return {"x": x, "w": w, "codes": codes, "M": M, "N": N, "K": K}

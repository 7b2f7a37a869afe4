"""K-ROUTE (bit-exact) and the routed A16W4 expert GEMM (normalised error) on the
GPU against the oracle."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_linear_gb300 as mx
from mxfp4_quantized_linear_gb300 import inputs
from oracle.linear import normalized_error
from oracle.moe import MX_ERR_EXPERT_ID, dequant_experts_bf16, moe_linear, route
from oracle.formats import bf16_rne_bits, bf16_value
from oracle.linear import dequant_values
from tests.helpers import TOL, bf16_np, cuda_device, ensure_built, u8

pytestmark = pytest.mark.gpu


def gpu_route(ids, E):
    dev = cuda_device()
    ensure_built()
    r = mx.mx_route_experts(ids.to(dev), E)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


@pytest.mark.parametrize("T,topk,E", [(37, 5, 11), (64, 8, 64), (256, 8, 256), (1, 8, 256), (300, 4, 512)])
def test_route_bit_exact(T, topk, E):
    rng = np.random.default_rng(T * E)
    ids = rng.integers(-1, E, size=(T, topk)).astype(np.int32)
    if T > 2:
        ids[1, 0] = E + 3
        ids[2, 1] = -9
    r = gpu_route(torch.tensor(ids), E)
    ref = route(ids, E)
    assert np.array_equal(r["counts"], ref["counts"])
    assert np.array_equal(r["offsets"], ref["offsets"])
    n = int(ref["offsets"][-1])
    assert np.array_equal(r["pairs"][:n], ref["pairs"])
    na = int(r["n_active"][0])
    assert na == len(ref["active"]) and np.array_equal(r["active"][:na], ref["active"])
    assert int(r["status"][0]) == ref["status"]


def test_route_empty():
    r = gpu_route(torch.zeros((0, 4), dtype=torch.int32), 8)
    assert int(r["n_active"][0]) == 0 and np.all(r["offsets"] == 0) and np.all(r["counts"] == 0)


def gpu_moe(m, ids=None, status=None):
    dev = cuda_device()
    ensure_built()
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    ids = m["ids"] if ids is None else ids
    y = mx.mxfp4_moe_linear(m["x"].to(dev), ids.to(dev), p, dev_status=status)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


def check_moe(m, ids=None):
    ids = m["ids"] if ids is None else ids
    dev = cuda_device()
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    y = gpu_moe(m, ids, status)
    xv = bf16_np(m["x"])
    W = dequant_experts_bf16(u8(m["w"]), u8(m["codes"]))
    ref = moe_linear(xv, u8(ids), u8(m["w"]), u8(m["codes"]), wdeq=W)
    idn = u8(ids)
    E = m["E"]
    for t in range(idn.shape[0]):
        for j in range(idn.shape[1]):
            e = int(idn[t, j])
            if 0 <= e < E:
                err = normalized_error(y[t, j][None], ref[t, j][None], xv[t][None], W[e])
                assert err <= TOL, (t, j, err)
            else:
                assert np.all(y[t, j] == 0)
    return int(status.item())


def test_moe_small_with_invalid_ids():
    m = inputs.moe_gate_up(E=8, N=256, K=512, T=13, topk=3, seed=1)
    ids = m["ids"].clone()
    ids[4, 1] = -1
    assert check_moe(m, ids) == 0
    ids[6, 2] = 99
    assert check_moe(m, ids) == MX_ERR_EXPERT_ID


def test_moe_ragged_rows_and_k():
    m = inputs.moe_gate_up(E=5, N=136, K=2080, T=9, topk=2, seed=2)
    assert check_moe(m) == 0


def test_moe_many_tokens_one_expert():
    m = inputs.moe_gate_up(E=3, N=128, K=256, T=40, topk=1, seed=3)
    ids = torch.zeros((40, 1), dtype=torch.int32)
    ids[::5] = 2
    assert check_moe(m, ids) == 0


def test_moe_several_passes_of_pairs():
    """70 pairs on one expert: three 32-pair passes over the same weight tiles
    (the last one ragged), ragged rows (N = 200) and three K steps."""
    m = inputs.moe_gate_up(E=4, N=200, K=384, T=70, topk=2, seed=7)
    ids = torch.full((70, 2), 3, dtype=torch.int32)
    ids[:, 1] = torch.arange(70, dtype=torch.int32) % 3
    assert check_moe(m, ids) == 0


def test_moe_a16_close_to_exact():
    """The bf16 activation enters the tensor core as two MXFP8 pieces hi + lo;
    their sum is x except below the e4m3 range of a block's residual scale, so
    each output is the exact A16W4 value up to its bf16 rounding (2^-9 |y|)
    plus a term far below the 1e-2 tolerance: |y - ref| <= 2^-8 |ref| +
    5e-5 ||w|| ||x||.  Dropping the lo piece alone would leave ~2^-5 / sqrt(K)
    of ||w|| ||x|| and fail this."""
    m = inputs.moe_gate_up(E=6, N=256, K=4096, T=24, topk=2, seed=8)
    y = gpu_moe(m)
    xv = bf16_np(m["x"])
    W = dequant_experts_bf16(u8(m["w"]), u8(m["codes"]))
    ids = u8(m["ids"])
    ref = moe_linear(xv, ids, u8(m["w"]), u8(m["codes"]), wdeq=W)
    worst = 0.0
    for t in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            den = np.linalg.norm(W[e].astype(np.float64), axis=1) * np.linalg.norm(xv[t].astype(np.float64))
            bound = 2.0 ** -8 * np.abs(ref[t, j]) + 5e-5 * den
            excess = np.abs(y[t, j] - ref[t, j]) - bound
            worst = max(worst, float(np.max(excess / den)))
    assert worst <= 0.0, worst


def test_moe_gate_up_full_size_sampled():
    m = inputs.moe_gate_up()
    y = gpu_moe(m)
    rng = np.random.default_rng(4)
    wb, cb, ids = u8(m["w"]), u8(m["codes"]), u8(m["ids"])
    xv = bf16_np(m["x"])
    for _ in range(48):
        t, j = int(rng.integers(0, 64)), int(rng.integers(0, 8))
        ns = np.sort(rng.choice(4096, size=64, replace=False))
        e = int(ids[t, j])
        Wd = bf16_value(bf16_rne_bits(dequant_values(wb[e, ns], cb[e, ns], "e2m1", len(ns), 4096)))
        ref = Wd @ xv[t]
        err = normalized_error(y[t, j, ns][None], ref[None], xv[t][None], Wd)
        assert err <= TOL, (t, j, err)


# ---------------------------------------------------------------- full expert

def test_moe_linear_on_gate_up_packing_is_identical():
    """The interleaved packing only moves rows: every output of mxfp4_moe_linear
    is bit-identical to the plain packing's."""
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_gate_up(E=6, N=192, K=1056, T=11, topk=3, seed=5)
    x, ids = m["x"].to(dev), m["ids"].to(dev)
    pp = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1", 0)
    pg = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1", mx.MX_PACK_GATE_UP)
    yp, yg = mx.mxfp4_moe_linear(x, ids, pp), mx.mxfp4_moe_linear(x, ids, pg)
    torch.cuda.synchronize()
    assert torch.equal(yp.view(torch.int16), yg.view(torch.int16))


def expert_error(out, ref, t, h, x_unused=None):
    """|out - out_ref| / sum_j |w_tj| ||W2[e_j, h]|| ||act_tj||: the normalised
    error of the combine (Cauchy-Schwarz bound of each slot's term)."""
    return abs(out - ref["out"][t, h]) / ref["den"][t, h] if ref["den"][t, h] > 0 else abs(out - ref["out"][t, h])


def oracle_expert(m, ids=None):
    from oracle.moe import moe_expert
    ids = u8(m["ids"] if ids is None else ids)
    r = moe_expert(bf16_np(m["x"]), ids, m["weights"].cpu().numpy().astype(np.float64), u8(m["w13"]),
                   u8(m["c13"]), u8(m["w2"]), u8(m["c2"]))
    W2 = dequant_experts_bf16(u8(m["w2"]), u8(m["c2"]))
    T, topk = ids.shape
    den = np.zeros_like(r["out"])
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            if 0 <= e < m["E"]:
                den[t] += abs(float(m["weights"][t, j])) * np.linalg.norm(W2[e], axis=1) * np.linalg.norm(r["act"][t, j])
    r["den"] = den
    return r


def gpu_expert(m, ids=None, status=None):
    dev = cuda_device()
    ensure_built()
    w13 = mx.mx_pack_weights(m["w13"].to(dev), m["c13"].to(dev), "e2m1", mx.MX_PACK_GATE_UP)
    w2 = mx.mx_pack_weights(m["w2"].to(dev), m["c2"].to(dev), "e2m1", 0)
    ids = m["ids"] if ids is None else ids
    y = mx.mxfp4_moe_expert(m["x"].to(dev), ids.to(dev), m["weights"].to(dev), w13, w2, dev_status=status)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


@pytest.mark.parametrize("E,I,H,T,topk", [(8, 160, 256, 13, 3), (5, 192, 160, 9, 2), (4, 256, 2080, 33, 4)])
def test_expert_matches_oracle(E, I, H, T, topk):
    m = inputs.moe_expert(E=E, I=I, H=H, T=T, topk=topk, seed=E + I)
    ids = m["ids"].clone()
    ids[T // 2, 0] = -1                  # a skipped slot
    y = gpu_expert(m, ids)
    ref = oracle_expert(m, ids)
    err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
    assert err <= TOL, err


def test_expert_invalid_id_status():
    dev = cuda_device()
    m = inputs.moe_expert(E=4, I=160, H=256, T=5, topk=2, seed=1)
    ids = m["ids"].clone()
    ids[2, 1] = 77
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    y = gpu_expert(m, ids, status)
    assert int(status.item()) == MX_ERR_EXPERT_ID
    ref = oracle_expert(m, ids)
    assert np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0)) <= TOL


def test_expert_refuses_plain_w13():
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_expert(E=2, I=160, H=256, T=2, topk=1, seed=2)
    w13 = mx.mx_pack_weights(m["w13"].to(dev), m["c13"].to(dev), "e2m1", 0)
    w2 = mx.mx_pack_weights(m["w2"].to(dev), m["c2"].to(dev), "e2m1", 0)
    with pytest.raises(mx.MxError):
        mx.mxfp4_moe_expert(m["x"].to(dev), m["ids"].to(dev), m["weights"].to(dev), w13, w2)


def test_expert_full_size_sampled_tokens():
    """E=64, I=2048, H=4096, T=64, top-8 (the gate/up GEMM of the bench, then
    SwiGLU, the down projection and the combine): two tokens checked in full."""
    from oracle.moe import silu
    m = inputs.moe_expert()
    y = gpu_expert(m)
    xv, ids, wts = bf16_np(m["x"]), u8(m["ids"]), m["weights"].numpy().astype(np.float64)
    I = m["I"]
    for t in (0, 37):
        out = np.zeros(m["H"])
        den = np.zeros(m["H"])
        for j in range(m["topk"]):
            e = int(ids[t, j])
            W13 = bf16_value(bf16_rne_bits(dequant_values(u8(m["w13"][e]), u8(m["c13"][e]), "e2m1", 2 * I, m["H"])))
            y13 = W13 @ xv[t]
            act = bf16_value(bf16_rne_bits(silu(y13[:I]) * y13[I:]))
            W2 = bf16_value(bf16_rne_bits(dequant_values(u8(m["w2"][e]), u8(m["c2"][e]), "e2m1", m["H"], I)))
            out += wts[t, j] * (W2 @ act)
            den += abs(wts[t, j]) * np.linalg.norm(W2, axis=1) * np.linalg.norm(act)
        err = np.max(np.abs(y[t] - out) / den)
        assert err <= TOL, (t, err)


def test_moe_single_k_step_and_k_32():
    """K = 128 (one K step, N below one row tile) and K = 32 (one block, padded
    to a step)."""
    assert check_moe(inputs.moe_gate_up(E=2, N=64, K=128, T=3, topk=1, seed=6)) == 0
    assert check_moe(inputs.moe_gate_up(E=3, N=40, K=32, T=5, topk=2, seed=9)) == 0


# ---------------------------------------------------------------- W4A8 (MXFP4 x MXFP8 activations)

def check_w4a8(m, ids=None):
    from oracle.moe import moe_linear_w4a8
    dev = cuda_device()
    ensure_built()
    ids = m["ids"] if ids is None else ids
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    y = mx.mxfp4_moe_linear_w4a8(m["x"].to(dev), ids.to(dev), p, dev_status=status)
    torch.cuda.synchronize()
    y = y.float().cpu().numpy()
    xv = bf16_np(m["x"])
    idn = u8(ids)
    r = moe_linear_w4a8(xv, idn, u8(m["w"]), u8(m["codes"]))
    E = m["E"]
    K = xv.shape[1]
    for t in range(idn.shape[0]):
        for j in range(idn.shape[1]):
            e = int(idn[t, j])
            if 0 <= e < E:
                W = dequant_values(u8(m["w"])[e], u8(m["codes"])[e], "e2m1", m["N"], K)
                err = normalized_error(y[t, j][None], r["y"][t, j][None], r["A"][t][None], W)
                assert err <= TOL, (t, j, err)
                # exact products, f32 sums, one bf16 rounding: far inside the tolerance
                den = np.linalg.norm(W, axis=1) * np.linalg.norm(r["A"][t])
                assert np.all(np.abs(y[t, j] - r["y"][t, j]) <= 2.0 ** -8 * np.abs(r["y"][t, j]) + 1e-5 * den)
            else:
                assert np.all(y[t, j] == 0)
    return int(status.item())


def test_w4a8_small_with_invalid_ids():
    m = inputs.moe_gate_up(E=8, N=256, K=512, T=13, topk=3, seed=21)
    ids = m["ids"].clone()
    ids[4, 1] = -1
    assert check_w4a8(m, ids) == 0
    ids[6, 2] = 99
    assert check_w4a8(m, ids) == MX_ERR_EXPERT_ID


def test_w4a8_ragged_rows_and_k():
    assert check_w4a8(inputs.moe_gate_up(E=5, N=136, K=2080, T=9, topk=2, seed=22)) == 0


def test_w4a8_several_passes_of_pairs():
    """75 pairs on one expert: three 32-pair passes (the last one ragged)."""
    m = inputs.moe_gate_up(E=4, N=200, K=384, T=75, topk=2, seed=23)
    ids = torch.full((75, 2), 1, dtype=torch.int32)
    ids[:, 0] = torch.tensor([0, 2, 3], dtype=torch.int32).repeat(25)
    assert check_w4a8(m, ids) == 0


def test_w4a8_full_size_sampled():
    from oracle.quant import quantize_act
    from oracle.linear import expand_codes
    from oracle.formats import e4m3_decode
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_gate_up()
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    y = mx.mxfp4_moe_linear_w4a8(m["x"].to(dev), m["ids"].to(dev), p)
    torch.cuda.synchronize()
    y = y.float().cpu().numpy()
    xv = bf16_np(m["x"])
    xq, xc = quantize_act(xv)
    A = e4m3_decode(xq) * expand_codes(xc, xv.shape[0], xv.shape[1])
    rng = np.random.default_rng(24)
    wb, cb, ids = u8(m["w"]), u8(m["codes"]), u8(m["ids"])
    for _ in range(48):
        t, j = int(rng.integers(0, 64)), int(rng.integers(0, 8))
        ns = np.sort(rng.choice(4096, size=64, replace=False))
        e = int(ids[t, j])
        Wd = dequant_values(wb[e, ns], cb[e, ns], "e2m1", len(ns), 4096)
        ref = Wd @ A[t]
        err = normalized_error(y[t, j, ns][None], ref[None], A[t][None], Wd)
        assert err <= TOL, (t, j, err)


# ---------------------------------------------------------------- wide passes (prefill sizes)

def test_w4a8_wide_passes():
    """Enough pairs an expert for the wide passes (128 pairs each): ragged
    counts, a ragged last pass, ragged rows and K."""
    m = inputs.moe_gate_up(E=4, N=200, K=416, T=300, topk=2, seed=31)
    assert check_w4a8(m) == 0


def test_a16w4_wide_passes_and_invalid_ids():
    """A16W4 with 64-pair wide passes (hi and lo stacked), with invalid ids."""
    m = inputs.moe_gate_up(E=3, N=136, K=288, T=150, topk=2, seed=32)
    ids = m["ids"].clone()
    ids[5, 1] = -1
    assert check_moe(m, ids) == 0


def test_expert_wide_passes():
    """The full expert at prefill-like pair counts (wide passes in both
    projections, I = 96 not a multiple of 128)."""
    m = inputs.moe_expert(E=4, I=96, H=256, T=160, topk=2, seed=33)
    ids = m["ids"].clone()
    ids[7, 0] = -1
    y = gpu_expert(m, ids)
    ref = oracle_expert(m, ids)
    err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
    assert err <= TOL, err


def test_many_pairs_routing_path():
    """More pairs than one routing chunk (4096): the many-CTA routing (count,
    scan, stable scatter) with invalid ids, under both activation forms."""
    m = inputs.moe_gate_up(E=5, N=64, K=128, T=2300, topk=2, seed=41)
    ids = m["ids"].clone()
    ids[17, 0] = -1
    ids[2222, 1] = -1
    assert check_moe(m, ids) == 0
    assert check_w4a8(m, ids) == 0
    ids[1000, 1] = 9
    assert check_w4a8(m, ids) == MX_ERR_EXPERT_ID


def test_expert_many_pairs():
    """The full expert past one routing chunk (4200 pairs): many-CTA routing,
    activation rows split once per token and per pair, wide passes."""
    m = inputs.moe_expert(E=4, I=64, H=128, T=2100, topk=2, seed=42)
    ids = m["ids"].clone()
    ids[5, 1] = -1
    y = gpu_expert(m, ids)
    ref = oracle_expert(m, ids)
    err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
    assert err <= TOL, err


@pytest.mark.parametrize("N", [300, 456, 584])
def test_wide_passes_odd_and_even_row_tiles(N):
    """Prefill pair counts with 3, 4 and 5 ragged 128-row weight tiles: an even
    count runs the two-tile items (two accumulators on one activation stage),
    an odd count the one-tile items; both activation forms."""
    m = inputs.moe_gate_up(E=3, N=N, K=544, T=200, topk=2, seed=50 + N)
    ids = m["ids"].clone()
    ids[3, 0] = -1
    assert check_w4a8(m, ids) == 0
    assert check_moe(m, ids) == 0


def test_w4a8_prefill_size_sampled():
    """The W4A8 prefill workload itself (E=64, N=K=4096, T=4096, top-8: wide
    two-tile passes, many-CTA routing, per-token activation rows) on sampled
    (token, slot, rows) against the oracle's quantized activation."""
    from oracle.quant import quantize_act
    from oracle.linear import expand_codes
    from oracle.formats import e4m3_decode
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_gate_up(T=4096)
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    y = mx.mxfp4_moe_linear_w4a8(m["x"].to(dev), m["ids"].to(dev), p)
    torch.cuda.synchronize()
    xv = bf16_np(m["x"])
    rng = np.random.default_rng(25)
    wb, cb, ids = u8(m["w"]), u8(m["codes"]), u8(m["ids"])
    for _ in range(32):
        t, j = int(rng.integers(0, 4096)), int(rng.integers(0, 8))
        xq, xc = quantize_act(xv[t:t + 1])
        a = (e4m3_decode(xq) * expand_codes(xc, 1, 4096))[0]
        ns = np.sort(rng.choice(4096, size=64, replace=False))
        e = int(ids[t, j])
        Wd = dequant_values(wb[e, ns], cb[e, ns], "e2m1", len(ns), 4096)
        got = y[t, j, torch.from_numpy(ns).to(dev)].float().cpu().numpy()
        err = normalized_error(got[None], (Wd @ a)[None], a[None], Wd)
        assert err <= TOL, (t, j, err)


def test_decode_split_k():
    """Few pairs on few experts (decode): the K steps of each (expert, row
    tile) are split over several CTAs (17 steps into uneven ranges), partial
    sums added in range order by the finishing kernel; both activation forms,
    an invalid id, and the full expert (SiLU-and-mul and f32 outputs)."""
    m = inputs.moe_gate_up(E=64, N=256, K=2080, T=2, topk=8, seed=61)
    ids = m["ids"].clone()
    ids[1, 3] = -1
    assert check_moe(m, ids) == 0
    assert check_w4a8(m, ids) == 0
    e = inputs.moe_expert(E=32, I=128, H=256, T=1, topk=8, seed=62)
    y = gpu_expert(e, e["ids"])
    ref = oracle_expert(e, e["ids"])
    err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
    assert err <= TOL, err


@pytest.mark.parametrize("n_act", [1, 5, 19, 28, 56, 57, 58, 64])
def test_decode_split_over_active_experts(n_act):
    """The decode K split is chosen on the device from the number of active
    experts: 64 pairs spread over exactly n_act experts (N = 1024, eight row
    tiles an expert; K = 1024, eight K steps) reach every choice on a
    152-SM part, unsplit ones among them (56 and 57 experts fill whole rounds
    of resident CTAs), and one expert with four passes of pairs.  Both
    activation forms against the oracle, per pair, the 1e-2 gate and the
    per-element bound."""
    from oracle.moe import moe_linear_w4a8
    E, N, K, T, topk = 64, 1024, 1024, 8, 8
    m = inputs.moe_gate_up(E=E, N=N, K=K, T=T, topk=topk, seed=300 + n_act)
    rng = np.random.default_rng(n_act)
    chosen = rng.permutation(E)[:n_act]
    ids = torch.from_numpy(chosen[np.arange(T * topk) % n_act].reshape(T, topk).astype(np.int32))
    dev = cuda_device()
    ensure_built()
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    xv = bf16_np(m["x"])
    idn = u8(ids)
    r8 = moe_linear_w4a8(xv, idn, u8(m["w"]), u8(m["codes"]))
    W = {int(e): dequant_values(u8(m["w"])[e], u8(m["codes"])[e], "e2m1", N, K) for e in chosen}
    for form in ("a16w4", "w4a8"):
        fn = mx.mxfp4_moe_linear if form == "a16w4" else mx.mxfp4_moe_linear_w4a8
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        y = fn(m["x"].to(dev), ids.to(dev), p, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        y = y.float().cpu().numpy()
        c = 5e-5 if form == "a16w4" else 1e-5
        for t in range(T):
            a = xv[t] if form == "a16w4" else r8["A"][t]
            for j in range(topk):
                Wd = W[int(idn[t, j])]
                ref = Wd @ a
                err = normalized_error(y[t, j][None], ref[None], a[None], Wd)
                assert err <= TOL, (form, t, j, err)
                den = np.linalg.norm(Wd, axis=1) * np.linalg.norm(a)
                assert np.all(np.abs(y[t, j] - ref) <= 2.0 ** -8 * np.abs(ref) + c * den), (form, t, j)


@pytest.mark.parametrize("T", [9, 32])
def test_sixteen_row_form_above_decode_sizes(T):
    """More than 64 pairs on experts that average at most half a 16-row pass
    (E=64, top-8, T=9 or 32: 72 or 256 pairs, 2 P <= 8 E), so the A16W4 and
    MXFP8 calls take the 16-row narrow form with the routing kernel's arrays
    (no K split, no routing of its own); an expert with more than 8 pairs
    takes two passes.  Ragged N (3 row tiles, the last partial) and K (two
    steps and a tail), an invalid id."""
    m = inputs.moe_gate_up(E=64, N=320, K=352, T=T, topk=8, seed=400 + T)
    ids = m["ids"].clone()
    ids[T - 1, 5] = -1
    ids[0, :] = torch.arange(8, dtype=torch.int32)       # experts 0..7 ...
    ids[1, :] = torch.arange(8, dtype=torch.int32)       # ... twice more,
    ids[2, :] = torch.arange(8, dtype=torch.int32)       # so some hold > 8 pairs at T=32
    assert check_moe(m, ids) == 0
    assert check_w4a8(m, ids) == 0


def test_decode_inputs_written_just_before_each_call():
    """Decode calls read the ids (and, through the activation kernel, x) that
    a device copy on the same stream wrote right before each call, six calls
    back to back with no synchronization between them: the expert kernel,
    which routes from the ids before its dependency wait, must see each
    call's own ids.  Both activation forms and the full expert, against the
    oracle per call."""
    from oracle.moe import moe_linear_w4a8
    dev = cuda_device()
    ensure_built()
    E, N, K, T, topk = 32, 256, 512, 2, 8
    m = inputs.moe_gate_up(E=E, N=N, K=K, T=T, topk=topk, seed=500)
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    g = torch.Generator().manual_seed(501)
    n = 6
    ids_h = [torch.randperm(E, generator=g)[: T * topk].reshape(T, topk).to(torch.int32) for _ in range(n)]
    x_h = [torch.randn((T, K), generator=g).to(torch.bfloat16) for _ in range(n)]
    ids_src = [t.to(dev) for t in ids_h]
    x_src = [t.to(dev) for t in x_h]
    ids_d = torch.empty((T, topk), dtype=torch.int32, device=dev)
    x_d = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    work = torch.empty(mx.mxfp4_moe_workspace_size(T, topk, E, N, K), dtype=torch.uint8, device=dev)
    W = dequant_experts_bf16(u8(m["w"]), u8(m["codes"]))
    for form, fn in (("a16w4", mx.mxfp4_moe_linear), ("w4a8", mx.mxfp4_moe_linear_w4a8)):
        torch.cuda.synchronize()
        outs = []
        for k in range(n):
            ids_d.copy_(ids_src[k])
            x_d.copy_(x_src[k])
            outs.append(fn(x_d, ids_d, p, workspace=work))
        torch.cuda.synchronize()
        for k in range(n):
            y = outs[k].float().cpu().numpy()
            xv = bf16_np(x_h[k])
            idn = u8(ids_h[k])
            if form == "a16w4":
                ref = moe_linear(xv, idn, u8(m["w"]), u8(m["codes"]), wdeq=W)
                A = xv
            else:
                r = moe_linear_w4a8(xv, idn, u8(m["w"]), u8(m["codes"]))
                ref, A = r["y"], r["A"]
            for t in range(T):
                for j in range(topk):
                    err = normalized_error(y[t, j][None], ref[t, j][None], A[t][None], W[int(idn[t, j])])
                    assert err <= TOL, (form, k, t, j, err)
    # the full expert: both projections at decode size
    e = inputs.moe_expert(E=16, I=128, H=256, T=T, topk=topk, seed=502)
    w13 = mx.mx_pack_weights(e["w13"].to(dev), e["c13"].to(dev), "e2m1", mx.MX_PACK_GATE_UP)
    w2 = mx.mx_pack_weights(e["w2"].to(dev), e["c2"].to(dev), "e2m1", 0)
    wts = e["weights"].to(dev)
    ids_e = [torch.randperm(16, generator=g)[: T * topk].reshape(T, topk).to(torch.int32) for _ in range(n)]
    ids_e_src = [t.to(dev) for t in ids_e]
    x_e_src = e["x"].to(dev)
    torch.cuda.synchronize()
    outs = []
    for k in range(n):
        ids_d.copy_(ids_e_src[k])
        outs.append(mx.mxfp4_moe_expert(x_e_src, ids_d, wts, w13, w2))
    torch.cuda.synchronize()
    for k in range(n):
        ref = oracle_expert(e, ids_e[k])
        y = outs[k].float().cpu().numpy()
        err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
        assert err <= TOL, (k, err)


def test_more_items_than_resident_ctas():
    """More (expert, row tile) items than resident CTAs (64 experts x 8 tiles
    over 3 CTAs an SM, a partly filled last round), ragged N and K, an invalid
    id, both activation forms, and the full expert."""
    m = inputs.moe_gate_up(E=64, N=1000, K=544, T=64, topk=8, seed=71)
    ids = m["ids"].clone()
    ids[9, 2] = -1
    assert check_moe(m, ids) == 0
    assert check_w4a8(m, ids) == 0
    e = inputs.moe_expert(E=64, I=512, H=1024, T=64, topk=8, seed=72)
    y = gpu_expert(e, e["ids"])
    ref = oracle_expert(e, e["ids"])
    err = np.max(np.abs(y - ref["out"]) / np.where(ref["den"] > 0, ref["den"], 1.0))
    assert err <= TOL, err


@pytest.mark.parametrize("T", [2, 300])
def test_every_id_invalid(T):
    """No pair routed anywhere (every id -1): no active expert, no pass, no
    split item; every output row is zero and the status is OK, at a decode
    size (split-K path) and a prefill size (wide passes), both activation forms
    and the full expert."""
    m = inputs.moe_gate_up(E=8, N=256, K=256, T=T, topk=2, seed=80 + T)
    ids = torch.full_like(m["ids"], -1)
    assert check_moe(m, ids) == 0
    assert check_w4a8(m, ids) == 0
    e = inputs.moe_expert(E=4, I=64, H=128, T=T, topk=2, seed=82 + T)
    status = torch.full((1,), -1, dtype=torch.int32, device=cuda_device())
    y = gpu_expert(e, torch.full_like(e["ids"], -1), status)
    assert np.all(y == 0) and int(status.item()) == 0


def test_zero_tokens():
    """T = 0: every MoE entry returns at once with an empty output."""
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_gate_up(E=4, N=128, K=128, T=1, topk=2, seed=90)
    p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
    x = m["x"][:0].to(dev)
    ids = m["ids"][:0].to(dev)
    assert mx.mxfp4_moe_linear(x, ids, p).shape == (0, 2, 128)
    assert mx.mxfp4_moe_linear_w4a8(x, ids, p).shape == (0, 2, 128)
    torch.cuda.synchronize()


# ---------------------------------------------------------------- the layer sweep's experts

@pytest.fixture(scope="module")
def sweep_experts():
    """E=256 experts of N=4096 rows, K=7168, top-8 routing of up to 256 tokens
    (3.8 GB of expert bytes, drawn on the device by the seeded generator)."""
    dev = cuda_device()
    ensure_built()
    m = inputs.moe_gate_up(E=256, N=4096, K=7168, T=256, topk=8, seed=5, device=dev)
    p = mx.mx_pack_weights(m["w"], m["codes"], "e2m1")
    torch.cuda.synchronize()
    yield m, p
    del p
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 2, 8, 256])
@pytest.mark.parametrize("form", ["a16w4", "w4a8"])
def test_sweep_experts_sampled(sweep_experts, T, form):
    """The layer sweep's expert shape (E=256, N=4096, K=7168, top-8) at decode
    token counts (K steps split over several CTAs, 56 steps into uneven
    ranges) and at T=256, against the oracle on sampled (token, slot, rows):
    the 1e-2 gate and the per-element bound 2^-8 |y_ref| + c ||w|| ||x||
    (c = 1e-5 for MXFP8 activations; 5e-5 for bf16 activations, which carry
    the hi/lo splitting term)."""
    from oracle.quant import quantize_act
    from oracle.linear import expand_codes
    from oracle.formats import e4m3_decode
    m, p = sweep_experts
    dev = cuda_device()
    K = 7168
    x = m["x"][:T].contiguous()
    ids = m["ids"][:T].contiguous()
    fn = mx.mxfp4_moe_linear if form == "a16w4" else mx.mxfp4_moe_linear_w4a8
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    y = fn(x, ids, p, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xv = bf16_np(x)
    idn = u8(ids)
    rng = np.random.default_rng(100 + T)
    pairs = [(t, j) for t in range(T) for j in range(8)]
    if len(pairs) > 40:
        pairs = [pairs[i] for i in rng.choice(len(pairs), size=40, replace=False)]
    c = 5e-5 if form == "a16w4" else 1e-5
    for t, j in pairs:
        e = int(idn[t, j])
        ns = np.sort(rng.choice(4096, size=48, replace=False))
        ns_d = torch.from_numpy(ns).to(dev)
        wb = m["w"][e].index_select(0, ns_d).cpu().numpy()
        cb = m["codes"][e].index_select(0, ns_d).cpu().numpy()
        Wd = dequant_values(wb, cb, "e2m1", len(ns), K)
        if form == "a16w4":
            a = xv[t]
        else:
            xq, xc = quantize_act(xv[t:t + 1])
            a = (e4m3_decode(xq) * expand_codes(xc, 1, K))[0]
        ref = Wd @ a
        got = y[t, j].index_select(0, ns_d).float().cpu().numpy()
        err = normalized_error(got[None], ref[None], a[None], Wd)
        assert err <= TOL, (t, j, err)
        den = np.linalg.norm(Wd, axis=1) * np.linalg.norm(a)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + c * den), (t, j)


def test_a16w4_wide_dynamic_range_blocks():
    """bf16 activations whose 32-element blocks span many binades, where the
    hi + lo MXFP8 pieces lose their smallest elements: bf16 subnormals next to
    values near 1, single outliers 2^20 above and 2^-20 below the rest of
    their block, blocks at 2^-120 and 2^100, and ordinary N(0,1) blocks.  Each
    token takes one pattern so that its norm is set by it.  Per element,
    |y - y_ref| <= 2^-8 |y_ref| + 5e-5 ||w|| ||x|| (the bound of the hi/lo
    reading: the pieces miss at most 2^-21.8 of a block's max |x| a value)."""
    K, T = 2048, 6
    m = inputs.moe_gate_up(E=4, N=256, K=K, T=T, topk=2, seed=12)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((T, K))
    blocks = x.reshape(T, K // 32, 32)
    # token 0: every block holds bf16 subnormals (2^-130 .. 2^-133) next to N(0,1) values
    sub = rng.integers(1, 8, size=(K // 32, 8)) * 2.0 ** -133 * rng.choice([-1.0, 1.0], size=(K // 32, 8))
    blocks[0, :, :8] = sub
    # token 1: one element of every block 2^20 above the rest
    blocks[1, :, 5] *= 2.0 ** 20
    # token 2: one element of every block 2^-20 below the rest
    blocks[2, :, 7] *= 2.0 ** -20
    # token 3: a tiny token (2^-120 scale) with one 2^20 outlier in every fourth block
    blocks[3] *= 2.0 ** -120
    blocks[3, ::4, 0] *= 2.0 ** 20
    # token 4: a huge token (2^100 scale)
    blocks[4] *= 2.0 ** 100
    # token 5: blocks alternate between the patterns above
    blocks[5, 0::4, 3] *= 2.0 ** 20
    blocks[5, 1::4, :16] *= 2.0 ** -125
    blocks[5, 2::4, 9] *= 2.0 ** -20
    m["x"] = torch.from_numpy(x).float().to(torch.bfloat16)
    xv = bf16_np(m["x"])
    assert np.any((np.abs(xv[0]) < 2.0 ** -126) & (xv[0] != 0))   # subnormals survived the cast
    y = gpu_moe(m)
    W = dequant_experts_bf16(u8(m["w"]), u8(m["codes"]))
    ids = u8(m["ids"])
    ref = moe_linear(xv, ids, u8(m["w"]), u8(m["codes"]), wdeq=W)
    for t in range(T):
        for j in range(2):
            e = int(ids[t, j])
            den = np.linalg.norm(W[e].astype(np.float64), axis=1) * np.linalg.norm(xv[t])
            assert normalized_error(y[t, j][None], ref[t, j][None], xv[t][None], W[e]) <= TOL, (t, j)
            bound = 2.0 ** -8 * np.abs(ref[t, j]) + 5e-5 * den
            assert np.all(np.abs(y[t, j] - ref[t, j]) <= bound), (t, j, float(np.max(np.abs(y[t, j] - ref[t, j]) / den)))

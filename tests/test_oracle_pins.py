"""Pins for the CPU oracle: each checks it against something other than itself.

* numpy fp64 brute force over ALL experts (independent routing by a full
  lexicographic sort, textbook softmax and SwiGLU) on tiny inputs;
* closed forms (E[U] for uniform routing, softmax identities, exact special
  cases: k = 1, k = E, E = 1);
* invariants (grouping is a stable permutation, per-route == dedup bitwise,
  linearity in the down weights);
* the dedup table printed on the FreeToken #46 page (unique experts / reuse)
  and its traffic model.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import accounting, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_from_bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def rand_bf16(rng, shape, sigma):
    t = torch.from_numpy((rng.standard_normal(shape) * sigma).astype(np.float32))
    return synth.bf16_bits(t.to(torch.bfloat16))


def ref_order(l):
    """Full order of experts by (logit descending, id ascending)."""
    E = l.shape[0]
    return np.lexsort((np.arange(E), -l.astype(np.float64)))


# --------------------------------------------------------------------- router
@pytest.mark.parametrize("B,H,E", [(4, 64, 8), (3, 72, 5), (1, 2048, 16)])
def test_router_matches_fp64_within_fp32_bound(B, H, E):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((B, H)).astype(np.float32)
    w = rand_bf16(rng, (E, H), 0.05)
    bias = rng.standard_normal(E).astype(np.float32)
    got = oracle.router(x, w, bias)
    wf = f32_from_bf16(w).astype(np.float64)
    ref = x.astype(np.float64) @ wf.T + bias
    bound = (H + 2) * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(wf).T + np.abs(bias)) * 1.01
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


def test_router_bf16_x_equals_widened_fp32():
    rng = np.random.default_rng(2)
    xb = rand_bf16(rng, (5, 64), 1.0)
    w = rand_bf16(rng, (8, 64), 0.02)
    a = oracle.router(xb, w)
    b = oracle.router(f32_from_bf16(xb), w)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(8, 2), (17, 3), (256, 8), (128, 2), (256, 6)])
def test_topk_ids_match_full_lexicographic_sort(E, k):
    rng = np.random.default_rng(E * 10 + k)
    lg = rng.standard_normal((40, E)).astype(np.float32)
    # plant exact ties: copy some logits onto other experts
    for t in range(0, 40, 3):
        a, b = rng.integers(0, E, 2)
        lg[t, b] = lg[t, a]
    lg[5, :] = 0.25  # all equal
    ids, w = oracle.topk(lg, k)
    for t in range(40):
        assert list(ids[t]) == list(ref_order(lg[t])[:k])


def test_topk_ties_go_to_the_lower_id():
    lg = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0]], np.float32)
    ids, _ = oracle.topk(lg, 3)
    assert list(ids[0]) == [1, 2, 4]
    ids, _ = oracle.topk(lg, 4)
    assert list(ids[0]) == [1, 2, 4, 3]


@pytest.mark.parametrize("E,k", [(8, 2), (256, 8), (64, 5)])
def test_topk_weights_are_softmax_of_selected_logits(E, k):
    rng = np.random.default_rng(7)
    lg = (rng.standard_normal((50, E)) * 3).astype(np.float32)
    ids, w = oracle.topk(lg, k)
    sel = np.take_along_axis(lg.astype(np.float64), ids.astype(np.int64), axis=1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(w - ref)) <= 1e-6
    assert np.max(np.abs(w.astype(np.float64).sum(1) - 1.0)) <= 1e-6
    # weights come out in descending order with the ids
    assert np.all(np.diff(w, axis=1) <= 1e-7)


def test_topk_k1_gives_weight_exactly_one_and_argmax():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((30, 12)).astype(np.float32)
    ids, w = oracle.topk(lg, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(lg, axis=1))


def test_topk_k_equals_E_is_the_full_softmax():
    rng = np.random.default_rng(4)
    E = 16
    lg = rng.standard_normal((10, E)).astype(np.float32)
    ids, w = oracle.topk(lg, E)
    l64 = lg.astype(np.float64)
    p = np.exp(l64 - l64.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for t in range(10):
        assert list(ids[t]) == list(ref_order(lg[t]))
        assert np.max(np.abs(w[t] - p[t, ids[t]])) <= 1e-6


# ------------------------------------------------------------------- grouping
@pytest.mark.parametrize("B,k,E", [(4, 2, 8), (64, 8, 256), (1, 2, 128), (128, 6, 256), (7, 3, 5)])
def test_group_is_a_stable_counting_sort(B, k, E):
    rng = np.random.default_rng(B + k + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    offsets, ridx, uniq = oracle.group(ids, E)
    flat = ids.reshape(-1)
    assert offsets[0] == 0 and offsets[E] == B * k
    assert np.all(np.diff(offsets) >= 0)
    assert np.array_equal(np.sort(ridx), np.arange(B * k))
    # brute force: a stable argsort of the flat ids is the same permutation
    assert np.array_equal(ridx, np.argsort(flat, kind="stable"))
    for e in range(E):
        seg = ridx[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
        assert (offsets[e + 1] - offsets[e]) == np.count_nonzero(flat == e)
    assert np.array_equal(uniq, np.unique(flat))


def _uniform_unique_counts(B, draws, seed):
    """U per draw for the uniform workload: logits i.i.d. N(0,1) -> oracle top-k -> group."""
    E, k = 256, 8
    rng = np.random.default_rng(seed)
    us = []
    for _ in range(draws):
        lg = rng.standard_normal((B, E)).astype(np.float32)
        ids, _ = oracle.topk(lg, k)
        _, _, uniq = oracle.group(ids, E)
        us.append(len(uniq))
    return np.array(us)


@pytest.mark.parametrize("B", [4, 8, 16, 32, 64])
def test_unique_experts_follow_the_closed_form(B):
    us = _uniform_unique_counts(B, 300, seed=B)
    mean = accounting.expected_unique(256, 8, B)
    se = us.std(ddof=1) / np.sqrt(len(us)) + 1e-9
    assert abs(us.mean() - mean) <= 4.5 * se + 0.05


def test_unique_counts_printed_on_the_dedup_page_are_plausible_draws():
    tab = json.load(open(os.path.join(GOLDEN, "freetoken46_dedup_table.json")))
    for bs, routes, unique, reuse, *_ in tab["rows"]:
        assert routes == bs * 8
        # the page's reuse column is routes / unique, rounded to 2 decimals
        assert round(routes / unique, 2) == pytest.approx(reuse, abs=0.006)
        us = _uniform_unique_counts(bs, 400, seed=1000 + bs)
        lo, hi = np.quantile(us, [0.0005, 0.9995])
        assert lo - 2 <= unique <= hi + 2, (bs, unique, lo, hi)


def test_traffic_model_reproduces_the_printed_predictions():
    tab = json.load(open(os.path.join(GOLDEN, "freetoken46_dedup_table.json")))
    for reuse, pred in tab["traffic_model"]["predicted"]:
        assert round(accounting.traffic_model_speedup(reuse), 2) == pytest.approx(pred, abs=1e-9)
    # 9.00 MB per expert on the PR page is 6*H*I bf16 bytes at H=2048, I=768
    assert accounting.layer_bytes(2048, 768, 256, 1) - 2 * 256 * 2048 == 9 * 2 ** 20


# -------------------------------------------------------------------- experts
def _fp64_bruteforce_layer(x, wr, gate_up, down, k, bias=None):
    """Independent fp64 layer: all E experts on every token, combined with a
    top-k mask from a full lexicographic sort of the logits."""
    xf = x.astype(np.float64) if x.dtype != np.uint16 else f32_from_bf16(x).astype(np.float64)
    W = f32_from_bf16(wr).astype(np.float64)
    G = f32_from_bf16(gate_up).astype(np.float64)
    D = f32_from_bf16(down).astype(np.float64)
    B = xf.shape[0]
    E, twoI, _ = G.shape
    I = twoI // 2
    logits = xf @ W.T + (0 if bias is None else bias.astype(np.float64))
    y = np.zeros_like(xf)
    ids = np.zeros((B, k), np.int64)
    margins = np.zeros(B)
    for t in range(B):
        order = np.lexsort((np.arange(E), -logits[t]))
        sel = order[:k]
        ids[t] = sel
        srt = np.sort(logits[t])[::-1]
        margins[t] = srt[k - 1] - srt[k] if k < E else np.inf
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        wsel = p[sel] / p[sel].sum()
        outs = []
        for e in range(E):  # every expert, masked afterwards
            g = G[e, :I] @ xf[t]
            u = G[e, I:] @ xf[t]
            h = g / (1.0 + np.exp(-g)) * u
            outs.append(D[e] @ h)
        mask = np.zeros(E)
        mask[sel] = wsel
        y[t] = sum(mask[e] * outs[e] for e in range(E))
    return y, ids, margins


@pytest.mark.parametrize("x_bf16", [False, True])
def test_layer_matches_fp64_bruteforce_on_the_tiny_workload(x_bf16):
    w = synth.TINY
    lw = synth.make_layer(w, 0, seed=0)
    x = synth.make_x(w, 0, seed=0)
    if x_bf16:
        x = x.to(torch.bfloat16)
    xn = synth.bf16_bits(x) if x_bf16 else x.numpy()
    wr, gu, dn = (synth.bf16_bits(lw[n]) for n in ("w_router", "gate_up", "down"))
    y, ids, wts, _ = oracle.layer(xn, wr, gu, dn, w.top_k)
    yref, idref, margins = _fp64_bruteforce_layer(xn, wr, gu, dn, w.top_k)
    assert np.all(margins > 1e-5)
    assert np.array_equal(ids, idref)
    scale = np.max(np.abs(yref))
    assert np.max(np.abs(y - yref)) <= 2e-5 * scale


def test_layer_with_bias_matches_fp64_bruteforce():
    rng = np.random.default_rng(11)
    B, H, I, E, k = 6, 32, 16, 12, 3
    x = rng.standard_normal((B, H)).astype(np.float32)
    wr = rand_bf16(rng, (E, H), H ** -0.5)
    gu = rand_bf16(rng, (E, 2 * I, H), 0.1)
    dn = rand_bf16(rng, (E, H, I), 0.1)
    bias = synth.zipf_bias(E, 3).numpy()
    y, ids, _, _ = oracle.layer(x, wr, gu, dn, k, bias=bias)
    yref, idref, margins = _fp64_bruteforce_layer(x, wr, gu, dn, k, bias=bias)
    ok = margins > 1e-5
    assert ok.sum() >= B - 1
    assert np.array_equal(ids[ok], idref[ok])
    assert np.max(np.abs(y[ok] - yref[ok])) <= 2e-5 * np.max(np.abs(yref))


def test_per_route_and_dedup_orders_are_bit_identical():
    rng = np.random.default_rng(5)
    B, H, I, E, k = 24, 48, 24, 6, 3  # heavy expert reuse
    x = rng.standard_normal((B, H)).astype(np.float32)
    wr = rand_bf16(rng, (E, H), 0.2)
    gu = rand_bf16(rng, (E, 2 * I, H), 0.05)
    dn = rand_bf16(rng, (E, H, I), 0.05)
    y0, ids0, w0, _ = oracle.layer(x, wr, gu, dn, k, mode=oracle.PER_ROUTE)
    y1, ids1, w1, _ = oracle.layer(x, wr, gu, dn, k, mode=oracle.DEDUP)
    assert np.array_equal(ids0, ids1) and np.array_equal(w0, w1)
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))


def test_single_expert_is_a_textbook_swiglu_mlp():
    rng = np.random.default_rng(6)
    B, H, I = 5, 40, 24
    x = rng.standard_normal((B, H)).astype(np.float32)
    wr = rand_bf16(rng, (1, H), 0.1)
    gu = rand_bf16(rng, (1, 2 * I, H), 0.1)
    dn = rand_bf16(rng, (1, H, I), 0.1)
    y, ids, w, _ = oracle.layer(x, wr, gu, dn, 1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    Wg = f32_from_bf16(gu[0, :I]).astype(np.float64)
    Wu = f32_from_bf16(gu[0, I:]).astype(np.float64)
    Wd = f32_from_bf16(dn[0]).astype(np.float64)
    a = x.astype(np.float64) @ Wg.T
    ref = ((a / (1 + np.exp(-a))) * (x.astype(np.float64) @ Wu.T)) @ Wd.T
    assert np.max(np.abs(y - ref)) <= 1e-5 * np.max(np.abs(ref))


def test_doubling_down_doubles_y_exactly():
    rng = np.random.default_rng(8)
    B, H, I, E, k = 4, 64, 32, 8, 2
    x = rng.standard_normal((B, H)).astype(np.float32)
    wr = rand_bf16(rng, (E, H), 0.1)
    gu = rand_bf16(rng, (E, 2 * I, H), 0.05)
    dn = rand_bf16(rng, (E, H, I), 0.05)
    dn2 = synth.bf16_bits(torch.from_numpy(f32_from_bf16(dn) * 2).to(torch.bfloat16))
    y1, *_ = oracle.layer(x, wr, gu, dn, k)
    y2, *_ = oracle.layer(x, wr, gu, dn2, k)
    assert np.array_equal(y2, 2 * y1)


def test_gate_and_up_halves_are_not_interchangeable():
    """Swapping the two halves of gate_up must change y (SiLU is applied to
    the gate half only) -- guards the row layout against a silent swap."""
    rng = np.random.default_rng(9)
    B, H, I, E, k = 3, 32, 16, 4, 2
    x = rng.standard_normal((B, H)).astype(np.float32)
    wr = rand_bf16(rng, (E, H), 0.1)
    gu = rand_bf16(rng, (E, 2 * I, H), 0.3)
    dn = rand_bf16(rng, (E, H, I), 0.1)
    swapped = np.concatenate([gu[:, I:], gu[:, :I]], axis=1)
    y, *_ = oracle.layer(x, wr, gu, dn, k)
    ys, *_ = oracle.layer(x, wr, swapped, dn, k)
    yref, _, _ = _fp64_bruteforce_layer(x, wr, gu, dn, k)
    assert np.max(np.abs(y - yref)) < np.max(np.abs(ys - yref))


# ---------------------------------------------------------------------- stack
def test_stack_python_and_c_drivers_agree_and_add_the_residual():
    rng = np.random.default_rng(10)
    B, H, I, E, k, L = 2, 64, 32, 8, 2, 3
    layers = []
    for _ in range(L):
        layers.append({"w_router": rand_bf16(rng, (E, H), 0.1),
                       "gate_up": rand_bf16(rng, (E, 2 * I, H), 0.05),
                       "down": rand_bf16(rng, (E, H, I), 0.05)})
    x = rng.standard_normal((B, H)).astype(np.float32)
    xa, ida = oracle.stack(x, layers, k)
    xb, idb = oracle.stack_c(x, layers, k)
    assert np.array_equal(xa, xb) and np.array_equal(ida, idb)
    # one layer by hand: x1 = x0 + y(x0) in fp32
    y0, *_ = oracle.layer(x, layers[0]["w_router"], layers[0]["gate_up"], layers[0]["down"], k)
    x1, _ = oracle.stack(x, layers[:1], k)
    assert np.array_equal(x1, (x + y0).astype(np.float32))


def test_oracle_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.group(np.array([[0, 9]], np.int32), 8)


# -------------------------------------------------------------------- RMSNorm
def _fp64_rmsnorm(x, g, eps):
    xf = x.astype(np.float64)
    return xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + eps) * g.astype(np.float64)


def test_rmsnorm_matches_fp64_within_fp32_rounding():
    rng = np.random.default_rng(21)
    for B, H in ((1, 64), (3, 2048), (5, 72)):
        x = (rng.standard_normal((B, H)) * rng.uniform(0.1, 10.0)).astype(np.float32)
        g = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
        a = oracle.rmsnorm(x, g, 1e-6)
        ref = _fp64_rmsnorm(x, g, 1e-6)
        assert np.max(np.abs(a - ref)) <= 1e-5 * np.max(np.abs(ref))


def test_rmsnorm_with_unit_weights_gives_unit_rms_and_ignores_scale():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    ones = np.ones(256, np.float32)
    a = oracle.rmsnorm(x, ones, 0.0)
    assert np.allclose(np.sqrt(np.mean(a.astype(np.float64) ** 2, axis=1)), 1.0, atol=1e-6)
    # scaling the input by a power of two changes nothing (eps = 0: every step
    # is exact under the scaling)
    assert np.array_equal(oracle.rmsnorm(x * 8.0, ones, 0.0), a)
    # the weights multiply each column
    g = np.linspace(0.5, 1.5, 256).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), a * g, rtol=1e-6, atol=0)


def test_prenorm_stack_adds_the_layer_of_the_normalised_input_to_the_raw_input():
    """x1 = x0 + MoE(rmsnorm(x0)): checked against the fp64 brute-force layer
    applied to the fp64 norm, and the C and Python drivers agree bitwise."""
    rng = np.random.default_rng(23)
    B, H, I, E, k, L, eps = 3, 64, 32, 8, 2, 3, 1e-6
    layers = []
    for _ in range(L):
        layers.append({"w_router": rand_bf16(rng, (E, H), 0.1),
                       "gate_up": rand_bf16(rng, (E, 2 * I, H), 0.05),
                       "down": rand_bf16(rng, (E, H, I), 0.05),
                       "norm": (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)})
    x = (3.0 * rng.standard_normal((B, H))).astype(np.float32)
    xa, ida = oracle.stack_norm(x, layers, k, eps)
    xb, idb = oracle.stack_norm_c(x, layers, k, eps)
    assert np.array_equal(xa, xb) and np.array_equal(ida, idb)
    x1, id1 = oracle.stack_norm(x, layers[:1], k, eps)
    a64 = _fp64_rmsnorm(x, layers[0]["norm"], eps)
    yref, idref, margins = _fp64_bruteforce_layer(a64, layers[0]["w_router"], layers[0]["gate_up"],
                                                  layers[0]["down"], k)
    ok = margins > 1e-5
    assert np.array_equal(id1[0][ok], idref[ok])
    ref = x.astype(np.float64) + yref
    assert np.max(np.abs(x1[ok] - ref[ok])) <= 2e-5 * np.max(np.abs(yref))
    # without the norm the layer sees a different input: the norm is applied
    xs, _ = oracle.stack(x, layers[:1], k)
    assert not np.allclose(xs, x1)


# ------------------------------------------------------- block-scaled FP8
def test_fp8_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8).reshape(1, 256)
    # one 1 x 256 matrix, two blocks of columns, unit scales
    dq = oracle.dequant_fp8_block(codes, np.ones((1, 2), np.float32))
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dq), nan) and nan.sum() == 2  # S.1111.111
    assert np.array_equal(dq[~nan], ref[~nan])
    assert float(np.nanmax(dq)) == 448.0 and float(dq[0, 1]) == 2.0 ** -9  # largest; smallest subnormal


def test_fp8_block_scales_apply_per_128_block():
    rng = np.random.default_rng(31)
    R, C = 200, 300  # ragged blocks at both edges
    codes = rng.integers(0, 126, size=(R, C)).astype(np.uint8)  # finite positive codes
    scale = rng.uniform(0.5, 2.0, size=(2, 3)).astype(np.float32)
    dq = oracle.dequant_fp8_block(codes, scale)
    base = oracle.dequant_fp8_block(codes, np.ones((2, 3), np.float32))
    for br in range(2):
        for bc in range(3):
            blk = np.s_[128 * br:128 * (br + 1), 128 * bc:128 * (bc + 1)]
            assert np.array_equal(dq[blk], (base[blk] * scale[br, bc]).astype(np.float32))


def test_fp8_block_round_trip_error_is_within_the_format_bound():
    w = synth.normal_bf16((2, 384, 256), 0.02, 0, 99, 0, "cpu")
    q, s = synth.quantize_fp8_block(w)
    wf = w.to(torch.float32).numpy()
    for e in range(2):
        dq = oracle.dequant_fp8_block(q[e].numpy(), s[e].numpy())
        # 3 mantissa bits: a normal code is within 2^-4 of its value; the
        # subnormals (below 2^-6 of the block's scale) within 2^-10 * scale
        sc = np.repeat(np.repeat(s[e].numpy(), 128, 0), 128, 1)[:384, :256]
        assert np.all(np.abs(dq - wf[e]) <= np.maximum(2.0 ** -4 * np.abs(wf[e]), 2.0 ** -10 * sc) + 1e-12)


def test_fp8_layer_is_the_bf16_layer_on_the_dequantised_weights():
    """The expert pass on fp32 weights (the FP8 path's dequantised weights)
    against the fp64 brute force on the same weights, and close to the bf16
    layer it was quantised from."""
    w = synth.TINY
    lw = synth.make_layer_fp8(w, 0, seed=0)
    x = synth.make_x(w, 0, seed=0).numpy()
    wr = synth.bf16_bits(lw["w_router"])
    gq = {e: oracle.dequant_fp8_block(lw["gate_up_q"][e].numpy(), lw["gate_up_scale"][e].numpy()) for e in range(w.E)}
    dq = {e: oracle.dequant_fp8_block(lw["down_q"][e].numpy(), lw["down_scale"][e].numpy()) for e in range(w.E)}
    lo = oracle.router(x, wr)
    ids, wts = oracle.topk(lo, w.top_k)
    y8 = oracle.experts(x, gq, dq, ids, wts, w.E)
    # fp64 brute force over the dequantised weights (routing fixed by the router)
    y64 = np.zeros_like(x, dtype=np.float64)
    for t in range(w.B):
        for j in range(w.top_k):
            e = ids[t, j]
            G = gq[e].astype(np.float64)
            g = G[:w.I] @ x[t]
            u = G[w.I:] @ x[t]
            h = g / (1.0 + np.exp(-g)) * u
            y64[t] += wts[t, j] * (dq[e].astype(np.float64) @ h)
    assert np.max(np.abs(y8 - y64)) <= 2e-5 * np.max(np.abs(y64))
    ybf = oracle.experts(x, synth.bf16_bits(lw["gate_up"]), synth.bf16_bits(lw["down"]), ids, wts, w.E)
    assert np.max(np.abs(y8 - ybf)) <= 0.1 * np.max(np.abs(ybf))  # quantisation noise, not a different layer


# ---------------------------------------------------------------- NVFP4
# E2M1 by its definition: sign, 2 exponent bits biased by 1, 1 mantissa bit;
# exponent 0 is the subnormal 0.m (so 0 and 0.5)
def _e2m1_by_definition(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = 0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -v if s else v


def test_nvfp4_decodes_every_code_and_its_nibble():
    codes = np.arange(16, dtype=np.uint8)
    # two elements a byte: element 2i in the low nibble of byte i
    packed = (codes[0::2] | (codes[1::2] << 4)).reshape(1, 8)
    one = np.array([[0x38]], np.uint8)  # E4M3 1.0: exponent 7 (the bias), mantissa 0
    dq = oracle.dequant_nvfp4(packed, one, 1.0)
    expect = np.array([_e2m1_by_definition(int(c)) for c in codes], np.float32).reshape(1, 16)
    assert np.array_equal(dq, expect)
    assert dq[0, :8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_nvfp4_block_and_matrix_scales_apply_per_16_elements():
    rng = np.random.default_rng(41)
    R, C = 5, 96
    codes = rng.integers(0, 16, size=(R, C)).astype(np.uint8)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    bs = rng.integers(0x08, 0x77, size=(R, C // 16)).astype(np.uint8)  # finite E4M3 codes
    gs = 0.3125
    dq = oracle.dequant_nvfp4(packed, bs, gs)
    bsf = torch.from_numpy(bs.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    el = np.vectorize(_e2m1_by_definition)(codes.astype(np.int64))
    ref = (el * np.repeat(bsf, 16, axis=1) * gs).astype(np.float32)  # exact up to one rounding
    assert np.array_equal(dq, ref)


def test_nvfp4_round_trip_is_within_half_a_code_step():
    w = synth.normal_bf16((2, 96, 256), 0.02, 0, 98, 0, "cpu")
    q, bs, gs = synth.quantize_nvfp4(w)
    wf = w.to(torch.float32).numpy()
    for e in range(2):
        dq = oracle.dequant_nvfp4(q[e].numpy(), bs[e].numpy(), float(gs[e]))
        unit = np.repeat(torch.from_numpy(bs[e].numpy().copy()).view(torch.float8_e4m3fn)
                         .to(torch.float32).numpy(), 16, axis=1) * float(gs[e])
        v = np.abs(wf[e]) / unit
        # half the gap to the neighbouring E2M1 magnitude, or the excess over 6
        half_gap = np.where(v < 2.0, 0.25, np.where(v < 4.0, 0.5, 1.0))
        bound = np.maximum(half_gap, v - 6.0) * unit
        assert np.all(np.abs(dq - wf[e]) <= bound * (1 + 1e-6) + 1e-12)


def test_nvfp4_layer_on_the_dequantised_weights():
    """The expert pass on the NVFP4 path's dequantised fp32 weights against
    the fp64 brute force on the same weights."""
    w = synth.TINY
    lw = synth.make_layer_nvfp4(w, 0, seed=0)
    x = synth.make_x(w, 0, seed=0).numpy()
    wr = synth.bf16_bits(lw["w_router"])
    gq = {e: oracle.dequant_nvfp4(lw["gate_up_q4"][e].numpy(), lw["gate_up_bs"][e].numpy(),
                                  float(lw["gate_up_gs"][e])) for e in range(w.E)}
    dq = {e: oracle.dequant_nvfp4(lw["down_q4"][e].numpy(), lw["down_bs"][e].numpy(),
                                  float(lw["down_gs"][e])) for e in range(w.E)}
    lo = oracle.router(x, wr)
    ids, wts = oracle.topk(lo, w.top_k)
    y4 = oracle.experts(x, gq, dq, ids, wts, w.E)
    y64 = np.zeros_like(x, dtype=np.float64)
    for t in range(w.B):
        for j in range(w.top_k):
            e = ids[t, j]
            G = gq[e].astype(np.float64)
            g = G[:w.I] @ x[t]
            u = G[w.I:] @ x[t]
            y64[t] += wts[t, j] * (dq[e].astype(np.float64) @ (g / (1.0 + np.exp(-g)) * u))
    assert np.max(np.abs(y4 - y64)) <= 2e-5 * np.max(np.abs(y64))

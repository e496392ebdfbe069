"""Helpers shared by the GPU parity tests: seeded cases, oracle calls and the
comparison rules.

Rules (applied element by element):
  * expert ids: bit-exact, except tokens whose oracle logit margin between the
    k-th and (k+1)-th expert is below NEAR_TIE -- those are counted and their
    outputs are compared against the oracle re-run with the GPU's ids;
  * grouped route list (offsets, route_idx, unique): bit-exact;
  * logits: within twice the fp32 dot-product bound (H+8) * 2^-24 * |x|.|W|;
  * routing weights: within 1e-5 absolute;
  * y: max |err| <= 2e-3 * max |y_oracle|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_decode_layer_gemv_gb300 import synth

NEAR_TIE = 1e-5
Y_TOL = 2e-3
W_TOL = 1e-5


def f32_from_bf16(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def np_x(x: torch.Tensor):
    """x as the oracle takes it: fp32 array, or raw bf16 bits."""
    if x.dtype == torch.bfloat16:
        return synth.bf16_bits(x)
    return x.detach().cpu().numpy().astype(np.float32)


def margins(logits: np.ndarray, k: int) -> np.ndarray:
    s = -np.sort(-logits.astype(np.float64), axis=1)
    if k >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def logit_bound(x_np, wr_bits, H):
    xf = f32_from_bf16(x_np) if x_np.dtype == np.uint16 else x_np
    return 2 * (H + 8) * 2.0 ** -24 * (np.abs(xf).astype(np.float64) @ np.abs(f32_from_bf16(wr_bits)).astype(np.float64).T) + 1e-30


def check_route(x, wr, bias, k, ids_g, w_g, logits_g):
    """Compare GPU routing with the oracle; returns (oracle ids, exempt mask)."""
    xn = np_x(x)
    wrn = synth.bf16_bits(wr)
    bn = None if bias is None else bias.detach().cpu().numpy()
    lo = oracle.router(xn, wrn, bn)
    ids_o, w_o = oracle.topk(lo, k)
    lg = logits_g.cpu().numpy()
    assert np.all(np.isfinite(lg))
    bound = logit_bound(xn, wrn, wr.shape[1])
    if bn is not None:
        bound = bound + 2 * 2.0 ** -24 * np.abs(bn)
    assert np.all(np.abs(lg - lo) <= bound), float(np.max(np.abs(lg - lo) - bound))
    exempt = margins(lo, k) < NEAR_TIE
    ig = ids_g.cpu().numpy()
    ok = ~exempt
    # ids must match where the margin is clear (order inside the top-k too,
    # unless two selected logits are within NEAR_TIE of each other)
    srt = -np.sort(-lo.astype(np.float64), axis=1)[:, :k]
    inner_tie = np.any(np.diff(srt, axis=1) > -NEAR_TIE, axis=1) if k > 1 else np.zeros(len(lo), bool)
    strict = ok & ~inner_tie
    assert np.array_equal(ig[strict], ids_o[strict])
    assert np.array_equal(np.sort(ig[ok], axis=1), np.sort(ids_o[ok], axis=1))
    wg = w_g.cpu().numpy()
    assert np.max(np.abs(wg[strict] - w_o[strict]), initial=0.0) <= W_TOL
    return ids_o, exempt


def check_y(y_g, y_o):
    y_g = y_g.detach().cpu().numpy()
    assert np.all(np.isfinite(y_g))
    scale = float(np.max(np.abs(y_o)))
    err = float(np.max(np.abs(y_g - y_o)))
    assert err <= Y_TOL * scale, (err, scale, err / max(scale, 1e-30))
    return err / max(scale, 1e-30)


def layer_weights_np(lw):
    return {"w_router": synth.bf16_bits(lw["w_router"]), "gate_up": synth.bf16_bits(lw["gate_up"]),
            "down": synth.bf16_bits(lw["down"]),
            "bias": None if lw.get("bias") is None else lw["bias"].detach().cpu().numpy()}


def oracle_weights_for(logits_o, ids_use):
    """The oracle's routing weights for a given choice of experts: oracle.topk
    on the oracle's logits with every expert outside the choice masked to
    -inf (its softmax term is then exactly 0, so the renormalised weights are
    those of the chosen experts), returned in the order of ids_use."""
    lo = np.asarray(logits_o, np.float32)
    ids_use = np.asarray(ids_use)
    B, k = ids_use.shape
    rows = np.arange(B)[:, None]
    masked = np.full_like(lo, -np.inf)
    masked[rows, ids_use] = lo[rows, ids_use]
    ids_m, w_m = oracle.topk(masked, k)
    w = np.empty((B, k), np.float32)
    for t in range(B):
        pos = {int(e): j for j, e in enumerate(ids_m[t])}
        w[t] = [w_m[t, pos[int(e)]] for e in ids_use[t]]
    return w


def oracle_layer_following(x, lw_np, k, ids_gpu, residual=None):
    """Oracle layer using the GPU's ids where they differ only on near ties
    (their weights from the oracle as well, for the GPU's choice)."""
    xn = np_x(x)
    lo = oracle.router(xn, lw_np["w_router"], lw_np["bias"])
    ids_o, w_o = oracle.topk(lo, k)
    ex = margins(lo, k) < NEAR_TIE
    ids = ids_o.copy()
    if ex.any():
        ig = ids_gpu.cpu().numpy()
        ids[ex] = ig[ex]
        w_o[ex] = oracle_weights_for(lo[ex], ids[ex])
    E = lw_np["w_router"].shape[0]
    y = oracle.experts(xn, lw_np["gate_up"], lw_np["down"], ids, w_o, E, residual=residual)
    return y, ids, int(ex.sum())


def check_layer_routing(x, wr, bias, k, ids_g, w_g, logits_o=None):
    """The ids and routing weights a forward call itself returned, against the
    oracle: ids in order (as a set where two selected logits are within
    NEAR_TIE; exempt where the k-th/(k+1)-th margin is), and the weights of
    the GPU's choice within W_TOL of the oracle's weights for that choice.
    Returns the number of exempt (near-tie) tokens."""
    xn = np_x(x)
    lo = logits_o if logits_o is not None else oracle.router(
        xn, synth.bf16_bits(wr), None if bias is None else bias.detach().cpu().numpy())
    ids_o, _ = oracle.topk(lo, k)
    ex = margins(lo, k) < NEAR_TIE
    srt = -np.sort(-lo.astype(np.float64), axis=1)[:, :k]
    inner = np.any(np.diff(srt, axis=1) > -NEAR_TIE, axis=1) if k > 1 else np.zeros(len(lo), bool)
    ig = ids_g.cpu().numpy()
    strict = ~ex & ~inner
    assert np.array_equal(ig[strict], ids_o[strict])
    assert np.array_equal(np.sort(ig[~ex], axis=1), np.sort(ids_o[~ex], axis=1))
    wg = w_g.cpu().numpy()
    w_for = oracle_weights_for(lo, ig)
    assert np.max(np.abs(wg - w_for), initial=0.0) <= W_TOL, float(np.max(np.abs(wg - w_for)))
    return int(ex.sum())


def check_grouping(api, ws, ids_g, B, H, I, E, k):
    """The grouped route list the layer left in its workspace, bit-exact
    against the oracle's counting sort of the layer's own ids."""
    off, ridx, uniq, nu = api.workspace_grouping(ws, B, H, I, E, k)
    off_o, ridx_o, uniq_o = oracle.group(ids_g.cpu().numpy(), E)
    assert np.array_equal(off.cpu().numpy(), off_o)
    assert np.array_equal(ridx.cpu().numpy(), ridx_o)
    n = int(nu.item())
    assert n == len(uniq_o)
    assert np.array_equal(uniq.cpu().numpy()[:n], uniq_o)

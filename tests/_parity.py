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


def oracle_layer_following(x, lw_np, k, ids_gpu, residual=None):
    """Oracle layer using the GPU's ids where they differ only on near ties."""
    xn = np_x(x)
    lo = oracle.router(xn, lw_np["w_router"], lw_np["bias"])
    ids_o, w_o = oracle.topk(lo, k)
    ex = margins(lo, k) < NEAR_TIE
    ids = ids_o.copy()
    if ex.any():
        ig = ids_gpu.cpu().numpy()
        ids[ex] = ig[ex]
        # weights for the GPU's choice: softmax of the chosen logits, renormalised
        for t in np.nonzero(ex)[0]:
            l = lo[t]
            m = np.max(l)
            p = np.exp((l - m).astype(np.float32)).astype(np.float32)
            p = p / p.sum(dtype=np.float32)
            sel = p[ids[t]]
            w_o[t] = sel / sel.sum(dtype=np.float32)
    E = lw_np["w_router"].shape[0]
    y = oracle.experts(xn, lw_np["gate_up"], lw_np["down"], ids, w_o, E, residual=residual)
    return y, ids, int(ex.sum())

"""CPU oracle for the MoE decode layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and the two share no
code: this wrapper marshals numpy arrays into ``moe_oracle.c`` and nothing
else.

Every function follows the plain definition of the layer (see the header of
``moe_oracle.c`` for the pages and sections each step comes from).  The pins
that tie it to something other than itself are in ``tests/test_oracle_pins.py``.
Parity status per function: router, top-k, grouping, experts, combine and the
stack are all pinned (brute force / closed forms / invariants); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PER_ROUTE = 0
DEDUP = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so with gcc (portable flags only)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_router.argtypes = [P, i, P, P, i, i, i, P]
            lib.oracle_topk.argtypes = [P, i, i, i, P, P]
            lib.oracle_group.argtypes = [P, i, i, i, P, P, P, P]
            lib.oracle_experts.argtypes = [P, i, P, P, P, P, i, i, i, i, i, i, P, P, P, P]
            lib.oracle_layer.argtypes = [P, i, P, P, P, P, i, i, i, i, i, i, P, P, P, P, P]
            lib.oracle_stack.argtypes = [i, P, P, P, P, i, i, i, i, i, i, P, P]
            lib.oracle_rmsnorm.argtypes = [P, P, i, i, ctypes.c_float, P]
            lib.oracle_experts_w.argtypes = [P, i, P, P, i, P, P, i, i, i, i, i, i, P, P, P, P]
            lib.oracle_dequant_fp8_block.argtypes = [P, P, i, i, P]
            lib.oracle_dequant_nvfp4.argtypes = [P, P, ctypes.c_float, i, i, P]
            lib.oracle_stack_norm.argtypes = [i, P, P, P, P, P, ctypes.c_float, i, i, i, i, i, i, P, P]
            for f in ("oracle_router", "oracle_topk", "oracle_group", "oracle_experts",
                      "oracle_layer", "oracle_stack", "oracle_rmsnorm", "oracle_stack_norm",
                      "oracle_experts_w", "oracle_dequant_fp8_block", "oracle_dequant_nvfp4"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def _x_arg(x):
    """x as fp32 (dtype 0) or raw bf16 bits in uint16 (dtype 1)."""
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), 1
    return np.ascontiguousarray(x, dtype=np.float32), 0


def router(x, w_router, bias=None):
    """logits[B,E] (fp32) = x . W_r^T (+bias), sums in h order."""
    xa, xd = _x_arg(x)
    wr = np.ascontiguousarray(w_router, dtype=np.uint16)
    B, H = xa.shape
    E = wr.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((B, E), np.float32)
    _check(_load().oracle_router(_ptr(xa), xd, _ptr(wr), _ptr(b), B, H, E, _ptr(out)), "router")
    return out


def topk(logits, k):
    """(ids[B,k] int32 in descending-logit order, w[B,k] fp32 renormalised)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    B, E = lg.shape
    ids = np.empty((B, k), np.int32)
    w = np.empty((B, k), np.float32)
    _check(_load().oracle_topk(_ptr(lg), B, E, k, _ptr(ids), _ptr(w)), "topk")
    return ids, w


def group(ids, E):
    """Stable counting sort -> (offsets[E+1], route_idx[R], unique[U])."""
    ia = np.ascontiguousarray(ids, dtype=np.int32)
    B, k = ia.shape
    offsets = np.empty(E + 1, np.int32)
    ridx = np.empty(max(B * k, 1), np.int32)
    uniq = np.empty(E, np.int32)
    nu = np.zeros(1, np.int32)
    _check(_load().oracle_group(_ptr(ia), B, k, E, _ptr(offsets), _ptr(ridx), _ptr(uniq), _ptr(nu)),
           "group")
    return offsets, ridx[:B * k].copy(), uniq[:int(nu[0])].copy()


def _expert_ptrs(gate_up, down, E):
    """Per-expert host pointer tables and the weight type (0: bf16 bit
    patterns in uint16, 1: fp32).  gate_up/down may be full [E,...] arrays or
    dicts {e: array} holding only the experts that are needed."""
    gp = (ctypes.c_void_p * E)()
    dp = (ctypes.c_void_p * E)()
    keep = []
    wtype = None
    for e in range(E):
        if isinstance(gate_up, dict):
            g = gate_up.get(e)
            d = down.get(e)
        else:
            g, d = gate_up[e], down[e]
        if g is not None:
            t = 1 if np.asarray(g).dtype == np.float32 else 0
            wtype = t if wtype is None else wtype
            if t != wtype:
                raise ValueError("expert weights of one call must share a type")
            dt = np.float32 if t == 1 else np.uint16
            g = np.ascontiguousarray(g, dtype=dt)
            d = np.ascontiguousarray(d, dtype=dt)
            keep += [g, d]
            gp[e] = g.ctypes.data
            dp[e] = d.ctypes.data
    return gp, dp, keep, (wtype or 0)


def experts(x, gate_up, down, ids, w, E, mode=DEDUP, residual=None, return_parts=False):
    """y[B,H] = sum_j w[t,j] * down_e(SiLU(gate_e x) * up_e x) (+ residual)."""
    xa, xd = _x_arg(x)
    B, H = xa.shape
    ia = np.ascontiguousarray(ids, dtype=np.int32)
    wa = np.ascontiguousarray(w, dtype=np.float32)
    k = ia.shape[1]
    g0 = gate_up[int(ia.flat[0])] if isinstance(gate_up, dict) and B > 0 else gate_up[0]
    I = g0.shape[0] // 2
    gp, dp, keep, wtype = _expert_ptrs(gate_up, down, E)
    res = None if residual is None else np.ascontiguousarray(residual, dtype=np.float32)
    y = np.empty((B, H), np.float32)
    hr = np.empty((max(B * k, 1), I), np.float32)
    orr = np.empty((max(B * k, 1), H), np.float32)
    _check(_load().oracle_experts_w(_ptr(xa), xd, ctypes.addressof(gp), ctypes.addressof(dp), wtype,
                                    _ptr(ia), _ptr(wa), B, H, I, E, k, mode, _ptr(res), _ptr(y),
                                    _ptr(hr), _ptr(orr)), "experts")
    del keep
    if return_parts:
        return y, hr[:B * k], orr[:B * k]
    return y


def dequant_fp8_block(q, scale):
    """Block-scaled FP8 (E4M3 codes [R, C] uint8, fp32 scales [ceil(R/128),
    ceil(C/128)]) -> fp32 [R, C]: decode(q) * scale of the code's block."""
    qa = np.ascontiguousarray(q, dtype=np.uint8)
    sa = np.ascontiguousarray(scale, dtype=np.float32)
    R, C = qa.shape
    if sa.shape != ((R + 127) // 128, (C + 127) // 128):
        raise ValueError(f"scale shape {sa.shape} for codes {qa.shape}")
    out = np.empty((R, C), np.float32)
    _check(_load().oracle_dequant_fp8_block(_ptr(qa), _ptr(sa), R, C, _ptr(out)), "dequant_fp8_block")
    return out


def dequant_nvfp4(q, bscale, gscale):
    """NVFP4 (E2M1 codes packed two a byte [R, C/2] uint8, element 2i in the
    low nibble; E4M3 scales of 16-element row blocks [R, C/16] uint8; one
    fp32 scale) -> fp32 [R, C]: e2m1(q) * e4m3(bscale) * gscale."""
    qa = np.ascontiguousarray(q, dtype=np.uint8)
    ba = np.ascontiguousarray(bscale, dtype=np.uint8)
    R, C2 = qa.shape
    C = 2 * C2
    if C % 16 or ba.shape != (R, C // 16):
        raise ValueError(f"block scales {ba.shape} for codes {qa.shape}")
    out = np.empty((R, C), np.float32)
    _check(_load().oracle_dequant_nvfp4(_ptr(qa), _ptr(ba), ctypes.c_float(float(gscale)), R, C, _ptr(out)),
           "dequant_nvfp4")
    return out


def layer(x, w_router, gate_up, down, k, bias=None, mode=DEDUP, residual=None):
    """Full layer: returns (y, ids, w, logits)."""
    logits = router(x, w_router, bias)
    ids, w = topk(logits, k)
    E = logits.shape[1]
    y = experts(x, gate_up, down, ids, w, E, mode=mode, residual=residual)
    return y, ids, w, logits


def stack(x, layers, k, mode=DEDUP):
    """x <- x + layer_l(x) for each layer dict {w_router, gate_up, down, bias}.
    Returns (x_out, ids[L,B,k])."""
    xa = np.array(x, dtype=np.float32, copy=True)
    all_ids = []
    for lw in layers:
        y, ids, _, _ = layer(xa, lw["w_router"], lw["gate_up"], lw["down"], k,
                             bias=lw.get("bias"), mode=mode, residual=xa)
        xa = y
        all_ids.append(ids)
    return xa, np.stack(all_ids) if all_ids else np.zeros((0,) + xa.shape[:1] + (k,), np.int32)


def rmsnorm(x, g, eps):
    """a[B,H] = x * (1/sqrt(mean_h x^2 + eps)) * g, fp32, sum of squares in h order."""
    xa = np.ascontiguousarray(x, dtype=np.float32)
    ga = np.ascontiguousarray(g, dtype=np.float32)
    B, H = xa.shape
    a = np.empty((B, H), np.float32)
    _check(_load().oracle_rmsnorm(_ptr(xa), _ptr(ga), B, H, float(eps), _ptr(a)), "rmsnorm")
    return a


def stack_norm(x, layers, k, eps, mode=DEDUP):
    """Pre-norm stack: x <- x + layer_l(rmsnorm_l(x)) for each layer dict
    {w_router, gate_up, down, bias, norm}.  Returns (x_out, ids[L,B,k])."""
    xa = np.array(x, dtype=np.float32, copy=True)
    all_ids = []
    for lw in layers:
        a = rmsnorm(xa, lw["norm"], eps)
        y, ids, _, _ = layer(a, lw["w_router"], lw["gate_up"], lw["down"], k,
                             bias=lw.get("bias"), mode=mode, residual=xa)
        xa = y
        all_ids.append(ids)
    return xa, np.stack(all_ids) if all_ids else np.zeros((0,) + xa.shape[:1] + (k,), np.int32)


def stack_norm_c(x, layers, k, eps, mode=DEDUP):
    """The same pre-norm stack driven by the C loop (oracle_stack_norm)."""
    xa = np.array(x, dtype=np.float32, copy=True)
    L = len(layers)
    B, H = xa.shape
    E = layers[0]["w_router"].shape[0]
    I = layers[0]["gate_up"].shape[1] // 2
    wr = (ctypes.c_void_p * L)()
    bs = (ctypes.c_void_p * L)()
    nw = (ctypes.c_void_p * L)()
    gp = (ctypes.c_void_p * (L * E))()
    dp = (ctypes.c_void_p * (L * E))()
    keep = []
    for l, lw in enumerate(layers):
        a = np.ascontiguousarray(lw["w_router"], dtype=np.uint16)
        n = np.ascontiguousarray(lw["norm"], dtype=np.float32)
        keep += [a, n]
        wr[l] = a.ctypes.data
        nw[l] = n.ctypes.data
        if lw.get("bias") is not None:
            b = np.ascontiguousarray(lw["bias"], dtype=np.float32)
            keep.append(b)
            bs[l] = b.ctypes.data
        g = np.ascontiguousarray(lw["gate_up"], dtype=np.uint16)
        d = np.ascontiguousarray(lw["down"], dtype=np.uint16)
        keep += [g, d]
        for e in range(E):
            gp[l * E + e] = g[e].ctypes.data
            dp[l * E + e] = d[e].ctypes.data
    ids = np.empty((L, B, k), np.int32)
    _check(_load().oracle_stack_norm(L, ctypes.addressof(wr), ctypes.addressof(bs), ctypes.addressof(gp),
                                     ctypes.addressof(dp), ctypes.addressof(nw), float(eps), B, H, I, E, k, mode,
                                     _ptr(xa), _ptr(ids)), "stack_norm")
    del keep
    return xa, ids


def stack_c(x, layers, k, mode=DEDUP):
    """The same stack driven by the C loop (oracle_stack) -- used to pin the
    Python stack driver and for CPU timing."""
    xa = np.array(x, dtype=np.float32, copy=True)
    L = len(layers)
    B, H = xa.shape
    E = layers[0]["w_router"].shape[0]
    I = layers[0]["gate_up"].shape[1] // 2
    wr = (ctypes.c_void_p * L)()
    bs = (ctypes.c_void_p * L)()
    gp = (ctypes.c_void_p * (L * E))()
    dp = (ctypes.c_void_p * (L * E))()
    keep = []
    for l, lw in enumerate(layers):
        a = np.ascontiguousarray(lw["w_router"], dtype=np.uint16)
        keep.append(a)
        wr[l] = a.ctypes.data
        if lw.get("bias") is not None:
            b = np.ascontiguousarray(lw["bias"], dtype=np.float32)
            keep.append(b)
            bs[l] = b.ctypes.data
        g = np.ascontiguousarray(lw["gate_up"], dtype=np.uint16)
        d = np.ascontiguousarray(lw["down"], dtype=np.uint16)
        keep += [g, d]
        for e in range(E):
            gp[l * E + e] = g[e].ctypes.data
            dp[l * E + e] = d[e].ctypes.data
    ids = np.empty((L, B, k), np.int32)
    _check(_load().oracle_stack(L, ctypes.addressof(wr), ctypes.addressof(bs), ctypes.addressof(gp),
                                ctypes.addressof(dp), B, H, I, E, k, mode, _ptr(xa), _ptr(ids)),
           "stack")
    del keep
    return xa, ids

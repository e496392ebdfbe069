"""Byte and reuse accounting for the benchmark and the tests (host logic).

Nothing here is part of the layer's arithmetic: these are the formulas the
measurement uses to turn a time into GB/s and to check reuse figures.
"""
from __future__ import annotations

import math


def expected_unique(E: int, k: int, B: int) -> float:
    """E[U] for B tokens each choosing a uniformly random k-subset of E experts."""
    return E * (1.0 - (1.0 - k / E) ** B)


def layer_bytes(H: int, I: int, E: int, unique: int) -> int:
    """Algorithmic weight bytes of one layer step: the bf16 router plus each
    unique selected expert once (gate_up 2I*H + down H*I, bf16)."""
    return 2 * E * H + unique * 6 * I * H


def traffic_model_speedup(reuse: float) -> float:
    """Speedup when only the gate_up pass (2/3 of an expert's bytes) is
    deduplicated: 1 / (2/3 / reuse + 1/3) -- the traffic model printed on the
    FreeToken #46 page (commit message)."""
    return 1.0 / ((2.0 / 3.0) / reuse + 1.0 / 3.0)


def sigma_logit(w) -> float:
    return w.sigma_router * math.sqrt(w.H)


def layer_bytes_fp8(H: int, I: int, E: int, unique: int) -> int:
    """The same for block-scaled FP8 experts: the bf16 router plus each unique
    selected expert's E4M3 codes (3I*H bytes) and fp32 block scales (one per
    128 x 128 block of gate_up [2I, H] and down [H, I])."""
    nb = lambda n: (n + 127) // 128
    scales = 4 * (nb(2 * I) * nb(H) + nb(H) * nb(I))
    return 2 * E * H + unique * (3 * I * H + scales)


def layer_bytes_nvfp4(H: int, I: int, E: int, unique: int) -> int:
    """The same for NVFP4 experts: the bf16 router plus each unique selected
    expert's E2M1 codes (3I*H / 2 bytes), E4M3 block scales (one byte per 16
    weights) and two fp32 matrix scales."""
    return 2 * E * H + unique * (3 * I * H // 2 + 3 * I * H // 16 + 8)

"""Seeded synthetic inputs for the MoE decode layer.

This module only draws random numbers: it holds none of the layer's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Recipe (every tensor has its own generator stream, seeded from
``(seed, tensor_id, expert)``):

* x:            N(0, 1), fp32 (bf16 for the prefill-sized workload);
                tensor_id 1000 + step.
* W_router[l]:  N(0, sigma_r) rounded to bf16 (round-to-nearest-even);
                tensor_id 10 + 3l.  sigma_r = 0.02, or 1/sqrt(H) for the
                uniform/skewed routing workloads, so that the logits are
                ~N(0, 1) given x.
* gate_up[l]:   [E, 2I, H], N(0, 0.02) -> bf16; tensor_id 11 + 3l; one
                stream per expert, so an expert can be regenerated alone.
* down[l]:      [E, H, I], N(0, 0.02) -> bf16; tensor_id 12 + 3l.
* bias (skewed routing only): b_e = 2 * log(1 / rank_e ** 1.1) with rank a
                seeded random permutation of 1..E (tensor_id 1).
* norm[l] (pre-norm stacks only): RMSNorm weights 1 + 0.1 * N(0, 1), fp32;
                tensor_id 5000 + l.

Small cases are generated on the CPU and copied to the device; the
full-size workloads are generated directly on the GPU by torch's own
generator (the values then depend on the device, so each case records
which device drew it).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    I: int
    E: int
    top_k: int
    layers: int = 1
    sigma_router: float = 0.02
    sigma_expert: float = 0.02
    x_bf16: bool = False
    zipf_bias: bool = False
    residual: bool = False
    batches: tuple = field(default_factory=tuple)

    def with_batch(self, B: int) -> "Workload":
        return Workload(self.name, B, self.H, self.I, self.E, self.top_k, self.layers,
                        self.sigma_router, self.sigma_expert, self.x_bf16, self.zipf_bias,
                        self.residual, self.batches)


# The five workloads the layer is measured and checked on.
TINY = Workload("tiny_b4_h64_i32_e8_k2", B=4, H=64, I=32, E=8, top_k=2)
STACK = Workload("stack30_b1_h2048_i768_e128_k2", B=1, H=2048, I=768, E=128, top_k=2,
                 layers=30, residual=True)
UNIFORM = Workload("uniform_e256_k8_h2048_i768", B=64, H=2048, I=768, E=256, top_k=8,
                   sigma_router=2048 ** -0.5, batches=(1, 4, 8, 16, 32, 64))
SKEWED = Workload("skewed_zipf_e256_k6_h2048_i768", B=128, H=2048, I=768, E=256, top_k=6,
                  sigma_router=2048 ** -0.5, zipf_bias=True, batches=(1, 16, 64, 128))
PREFILL = Workload("prefill_b512_e256_k8_h4096_i1536", B=512, H=4096, I=1536, E=256, top_k=8,
                   x_bf16=True)
# The dense counterpart of the stack: one expert, top-1 (a plain SwiGLU MLP per
# layer, routing weight 1), with I = 2 x 768 so that a layer streams the same
# active weight bytes as a top-2 layer of the MoE stack.  The layer output
# scales as sigma^3 * sqrt(I) (times sqrt(sum w^2) for the MoE: about 0.71
# for two experts); sigma = 0.016 gives the dense layer the MoE layer's
# output scale (0.02^3 * sqrt(768) * 0.71 = 0.016^3 * sqrt(1536)), so that
# the 30-layer residual stream stays O(1) as it does for the MoE stack.
DENSE = Workload("dense_stack30_b1_h2048_i1536", B=1, H=2048, I=1536, E=1, top_k=1, layers=30,
                 sigma_expert=0.016, residual=True)

WORKLOADS = {w.name: w for w in (TINY, STACK, UNIFORM, SKEWED, PREFILL, DENSE)}


def _gen(seed: int, tensor_id: int, sub: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    # a fixed mixing of the three integers into one 63-bit seed
    s = (seed * 0x9E3779B1 + tensor_id * 0x85EBCA77 + sub * 0xC2B2AE3D + 0x27D4EB2F) % (2 ** 63 - 1)
    g.manual_seed(s)
    return g


def normal_bf16(shape, sigma, seed, tensor_id, sub, device) -> torch.Tensor:
    g = _gen(seed, tensor_id, sub, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * sigma).to(torch.bfloat16)


def make_layer(w: Workload, layer: int = 0, seed: int = 0, device="cpu"):
    """Weights of one layer as torch tensors on ``device``."""
    E, H, I = w.E, w.H, w.I
    wr = normal_bf16((E, H), w.sigma_router, seed, 10 + 3 * layer, 0, device)
    gate_up = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
    down = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        gate_up[e] = normal_bf16((2 * I, H), w.sigma_expert, seed, 11 + 3 * layer, e, device)
        down[e] = normal_bf16((H, I), w.sigma_expert, seed, 12 + 3 * layer, e, device)
    bias = zipf_bias(E, seed).to(device) if w.zipf_bias else None
    return {"w_router": wr, "gate_up": gate_up, "down": down, "bias": bias}


def quantize_fp8_block(w: torch.Tensor, block: int = 128):
    """Block-scaled FP8 copy of a weight matrix [..., R, C] (input
    preparation, not the layer's arithmetic): per block of block x block
    elements the fp32 scale amax / 448 (448 = the largest E4M3 value; a zero
    block gets scale 1), the codes round(w / scale) to float8_e4m3fn by
    torch.  Returns (codes uint8 [..., R, C], scales fp32 [..., ceil(R/b),
    ceil(C/b)])."""
    wf = w.to(torch.float32)
    *lead, R, C = wf.shape
    nbr, nbc = (R + block - 1) // block, (C + block - 1) // block
    pad = torch.zeros(*lead, nbr * block, nbc * block, dtype=torch.float32, device=w.device)
    pad[..., :R, :C] = wf
    blocks = pad.reshape(*lead, nbr, block, nbc, block)
    amax = blocks.abs().amax(dim=(-3, -1))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale[..., :, None, :, None]).reshape(*lead, nbr * block, nbc * block)[..., :R, :C]
    codes = q.contiguous().to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.contiguous()


def make_layer_fp8(w: Workload, layer: int = 0, seed: int = 0, device="cpu"):
    """A layer of the recipe with its expert weights in block-scaled FP8:
    the bf16 weights of make_layer, quantised per 128 x 128 block."""
    lw = make_layer(w, layer, seed=seed, device=device)
    gq, gs = quantize_fp8_block(lw["gate_up"])
    dq, ds = quantize_fp8_block(lw["down"])
    lw.update({"gate_up_q": gq, "gate_up_scale": gs, "down_q": dq, "down_scale": ds})
    return lw


# E2M1 magnitudes by code (bits: exponent, mantissa) and the midpoints between
# neighbours, for round-to-nearest (a value on a midpoint takes the smaller code)
_E2M1 = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_nvfp4(w: torch.Tensor):
    """[E, R, C] weights -> NVFP4: E2M1 codes packed two a byte [E, R, C/2]
    uint8 (element 2i of a row in the low nibble), E4M3 scales of 16-element
    row blocks [E, R, C/16] uint8, one fp32 scale per matrix [E]:
    gs = amax / (448 * 6), block scale = e4m3(block amax / 6 / gs), code =
    nearest E2M1 of w / (block scale * gs), clamped to +-6."""
    E, R, C = w.shape
    if C % 16:
        raise ValueError("NVFP4 rows need a multiple of 16 elements")
    dev = w.device
    mid = torch.tensor(_E2M1_MID, dtype=torch.float32, device=dev)
    q = torch.empty((E, R, C // 2), dtype=torch.uint8, device=dev)
    bs = torch.empty((E, R, C // 16), dtype=torch.uint8, device=dev)
    gs = torch.empty(E, dtype=torch.float32)
    for e in range(E):  # one matrix at a time: bounded temporaries
        wf = w[e].to(torch.float32)
        g = float(wf.abs().amax()) / (448.0 * 6.0)
        g = g if g > 0.0 else 1.0
        blk = wf.view(R, C // 16, 16)
        s = (blk.abs().amax(-1) / 6.0 / g).clamp(max=448.0)
        s8 = s.to(torch.float8_e4m3fn)
        sf = s8.to(torch.float32)
        v = blk / torch.where(sf > 0, sf, torch.ones_like(sf)).unsqueeze(-1) / g
        mag = torch.bucketize(v.abs().clamp(max=6.0), mid).to(torch.uint8)  # 0..7
        code = mag | ((v < 0) & (mag > 0)).to(torch.uint8) << 3
        code = code.view(R, C)
        q[e] = code[:, 0::2] | (code[:, 1::2] << 4)
        bs[e] = s8.view(torch.uint8)
        gs[e] = g
    return q, bs, gs.to(dev)


def make_layer_nvfp4(w: Workload, layer: int = 0, seed: int = 0, device="cpu"):
    """A layer of the recipe with its expert weights in NVFP4: the bf16 weights
    of make_layer, quantised per 16-element row block."""
    lw = make_layer(w, layer, seed=seed, device=device)
    gq, gb, gg = quantize_nvfp4(lw["gate_up"])
    dq, db, dg = quantize_nvfp4(lw["down"])
    lw.update({"gate_up_q4": gq, "gate_up_bs": gb, "gate_up_gs": gg,
               "down_q4": dq, "down_bs": db, "down_gs": dg})
    return lw


def norm_weights(H: int, layer: int = 0, seed: int = 0, device="cpu") -> torch.Tensor:
    """RMSNorm weights of layer l: 1 + 0.1 * N(0, 1), fp32 (tensor_id 5000 + l)."""
    g = _gen(seed, 5000 + layer, 0, device)
    return 1.0 + 0.1 * torch.randn(H, generator=g, device=device, dtype=torch.float32)


def zipf_bias(E: int, seed: int = 0) -> torch.Tensor:
    """b_e = 2*log(1/rank_e^1.1), rank a seeded permutation of 1..E (fp32)."""
    g = _gen(seed, 1, 0, "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (2.0 * torch.log(1.0 / rank ** 1.1)).to(torch.float32)


def make_x(w: Workload, step: int = 0, seed: int = 0, device="cpu", B: int | None = None):
    B = w.B if B is None else B
    g = _gen(seed, 1000 + step, 0, device)
    x = torch.randn((B, w.H), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16) if w.x_bf16 else x


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (CPU copy)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)

"""NVFP4 expert weights (E2M1 codes two a byte, an E4M3 scale per 16
elements, an fp32 scale per matrix) through the persistent decode kernel
and, for larger batches, the CUDA-core phase kernels, against the oracle on
the dequantised weights."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import synth
from _parity import NEAR_TIE, check_y, margins, np_x, oracle_weights_for

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _nvfp4_layers(w, L, seed):
    return [synth.make_layer_nvfp4(w, l, seed=seed, device=DEV) for l in range(L)]


def _oracle_walk(x0, layers, k, ids_gpu):
    """The oracle's stack on the dequantised experts, following the GPU's ids
    only on near ties; ids compared in order where the margins are clear."""
    x = x0.cpu().numpy().astype(np.float32)
    for l, lw in enumerate(layers):
        wr = synth.bf16_bits(lw["w_router"])
        bias = None if lw.get("bias") is None else lw["bias"].cpu().numpy()
        lo = oracle.router(x, wr, bias)
        ids_o, w_o = oracle.topk(lo, k)
        ex = margins(lo, k) < NEAR_TIE
        ig = ids_gpu[l].cpu().numpy()
        srt = -np.sort(-lo.astype(np.float64), axis=1)[:, :k]
        inner = np.any(np.diff(srt, axis=1) > -NEAR_TIE, axis=1) if k > 1 else np.zeros(len(lo), bool)
        strict = ~ex & ~inner
        assert np.array_equal(ig[strict], ids_o[strict]), l
        ids = np.where(ex[:, None], ig, ids_o)
        if ex.any():
            w_o[ex] = oracle_weights_for(lo[ex], ids[ex])
        gq, dq = {}, {}
        for e in np.unique(ids):
            e = int(e)
            gq[e] = oracle.dequant_nvfp4(lw["gate_up_q4"][e].cpu().numpy(), lw["gate_up_bs"][e].cpu().numpy(),
                                         float(lw["gate_up_gs"][e]))
            dq[e] = oracle.dequant_nvfp4(lw["down_q4"][e].cpu().numpy(), lw["down_bs"][e].cpu().numpy(),
                                         float(lw["down_gs"][e]))
        x = oracle.experts(x, gq, dq, ids, w_o, wr.shape[0], residual=x)
    return x


@pytest.mark.parametrize("B,H,I,E,k,L", [
    (1, 256, 128, 16, 2, 3),
    (4, 512, 256, 32, 4, 2),
    (2, 256, 512, 8, 2, 2),    # I > H/2: ring stages of fewer than four down rows
    (3, 384, 160, 5, 3, 2),    # rows of 12 and 5 scale blocks
])
def test_nvfp4_stack_matches_oracle_on_dequantised_weights(cuda_lib, B, H, I, E, k, L):
    w = synth.Workload("nvfp4", B=B, H=H, I=I, E=E, top_k=k, layers=L, sigma_router=H ** -0.5, sigma_expert=0.05)
    layers = _nvfp4_layers(w, L, seed=B + I)
    sw = cuda_lib.StackWeightsNVFP4(layers)
    x0 = synth.make_x(w, 0, seed=B + I, device=DEV)
    x = x0.clone()
    ids = torch.empty((L, B, k), dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    cuda_lib.stack_forward_nvfp4_(x, sw, k, ids_out=ids, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_y(x, _oracle_walk(x0, layers, k, ids))


def test_nvfp4_30_layer_stack_at_full_size(cuda_lib):
    w = synth.STACK
    layers = _nvfp4_layers(w, w.layers, seed=0)
    for lw in layers:  # only the codes and scales stay on the device
        lw.pop("gate_up")
        lw.pop("down")
    torch.cuda.empty_cache()
    sw = cuda_lib.StackWeightsNVFP4(layers)
    x0 = synth.make_x(w, 0, seed=0, device=DEV)
    x = x0.clone()
    ids = torch.empty((w.layers, 1, w.top_k), dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    n0 = cuda_lib.launch_count()
    cuda_lib.stack_forward_nvfp4_(x, sw, w.top_k, ids_out=ids, status=st)
    torch.cuda.synchronize()
    assert cuda_lib.launch_count() - n0 == 1
    assert int(st.item()) == 0
    check_y(x, _oracle_walk(x0, layers, w.top_k, ids))
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,H,I,E,k,L,flags", [
    (9, 256, 128, 16, 2, 2, 0),        # beyond the decode kernel: the phase kernels layer by layer
    (24, 384, 160, 12, 3, 2, 0),       # 16-element blocks across 128-column boundaries
    (64, 512, 256, 32, 8, 1, 0),       # a uniform-routing batch shape, top-8
    (3, 256, 128, 16, 2, 2, 2),        # MOE_F_UNFUSED below the decode kernel's limit
])
def test_nvfp4_phase_kernels_match_oracle_on_dequantised_weights(cuda_lib, B, H, I, E, k, L, flags):
    """Batches beyond the decode kernel (and MOE_F_UNFUSED) run the CUDA-core
    phase kernels on the E2M1 codes with their block and matrix scales."""
    w = synth.Workload("nvfp4", B=B, H=H, I=I, E=E, top_k=k, layers=L, sigma_router=H ** -0.5,
                       sigma_expert=0.05)
    layers = _nvfp4_layers(w, L, seed=B + I)
    sw = cuda_lib.StackWeightsNVFP4(layers)
    x0 = synth.make_x(w, 0, seed=B + I, device=DEV)
    x = x0.clone()
    ids = torch.empty((L, B, k), dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    cuda_lib.stack_forward_nvfp4_(x, sw, k, flags=flags, ids_out=ids, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_y(x, _oracle_walk(x0, layers, k, ids))

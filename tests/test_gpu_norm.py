"""Pre-norm stacks (x <- x + layer(RMSNorm(x))) on the GPU against the CPU
oracle: the norm fused into the persistent decode kernel's router and
residual add, and the layer-by-layer path with a norm kernel."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import synth
from _parity import NEAR_TIE, check_y, margins, np_x, oracle_layer_following

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6


def _layers(w, L, seed):
    out = []
    for l in range(L):
        lw = synth.make_layer(w, l, seed=seed, device=DEV)
        lw["norm"] = synth.norm_weights(w.H, l, seed=seed, device=DEV)
        out.append(lw)
    return out


def _np(lw):
    return {"w_router": synth.bf16_bits(lw["w_router"]), "gate_up": synth.bf16_bits(lw["gate_up"]),
            "down": synth.bf16_bits(lw["down"]),
            "bias": None if lw.get("bias") is None else lw["bias"].cpu().numpy()}


def _oracle_walk(x0, layers, k, ids_gpu):
    """The oracle's pre-norm stack, following the GPU's ids only on near ties;
    ids compared in order where the margins are clear."""
    x = x0.cpu().numpy().astype(np.float32)
    for l, lw in enumerate(layers):
        lnp = _np(lw)
        a = oracle.rmsnorm(x, lw["norm"].cpu().numpy(), EPS)
        lo = oracle.router(a, lnp["w_router"], lnp["bias"])
        ids_o, _ = oracle.topk(lo, k)
        ex = margins(lo, k) < NEAR_TIE
        ig = ids_gpu[l].cpu().numpy()
        if k > 1:
            srt = -np.sort(-lo.astype(np.float64), axis=1)[:, :k]
            inner = np.any(np.diff(srt, axis=1) > -NEAR_TIE, axis=1)
        else:
            inner = np.zeros(len(lo), bool)
        strict = ~ex & ~inner
        assert np.array_equal(ig[strict], ids_o[strict]), l
        y, _, _ = oracle_layer_following(torch.from_numpy(a), lnp, k, ids_gpu[l], residual=x)
        x = y
    return x


@pytest.mark.parametrize("B,H,I,E,k,L,flags", [
    (1, 256, 96, 16, 2, 3, 0),      # decode kernel, norm fused
    (4, 512, 128, 32, 4, 2, 0),     # decode kernel, four tokens
    (3, 72, 40, 5, 3, 2, 0),        # ragged H and I
    (9, 256, 64, 12, 3, 2, 0),      # beyond the decode kernel: norm kernel + tensor-core phases
    (9, 256, 64, 12, 3, 2, 8),      # MOE_F_NO_TC: norm kernel + fused CUDA-core layer
    (24, 256, 128, 8, 2, 2, 64),    # MOE_F_SPLIT_TC: norm kernel + tensor cores + streaming GEMV
    (2, 256, 96, 16, 2, 2, 2),      # MOE_F_UNFUSED
])
def test_prenorm_stack_matches_oracle(cuda_lib, B, H, I, E, k, L, flags):
    w = synth.Workload("norm", B=B, H=H, I=I, E=E, top_k=k, layers=L, sigma_router=H ** -0.5,
                       sigma_expert=0.05)
    layers = _layers(w, L, seed=B + H)
    sw = cuda_lib.StackWeights(layers)
    x0 = 2.0 * synth.make_x(w, 0, seed=B + H, device=DEV)  # not unit scale: the norm matters
    x = x0.clone()
    ids = torch.empty((L, B, k), dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    cuda_lib.stack_forward_norm_(x, sw, k, eps=EPS, flags=flags, ids_out=ids, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x_o = _oracle_walk(x0, layers, k, ids)
    check_y(x, x_o)


def test_prenorm_30_layer_stack_at_full_size(cuda_lib):
    """The headline stack's shape (B=1, H=2048, I=768, E=128, top-2, 30
    layers) as a pre-norm stack: one launch of the decode kernel."""
    w = synth.STACK
    path, _ = cuda_lib.forward_path(w.B, w.H, w.I, w.E, w.top_k, L=w.layers)
    assert path == cuda_lib.PATH_DECODE
    layers = _layers(w, w.layers, seed=0)
    sw = cuda_lib.StackWeights(layers)
    x0 = synth.make_x(w, 0, seed=0, device=DEV)
    x = x0.clone()
    ids = torch.empty((w.layers, 1, w.top_k), dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    n0 = cuda_lib.launch_count()
    cuda_lib.stack_forward_norm_(x, sw, w.top_k, eps=EPS, ids_out=ids, status=st)
    torch.cuda.synchronize()
    assert cuda_lib.launch_count() - n0 == 1
    assert int(st.item()) == 0
    x_o = _oracle_walk(x0, layers, w.top_k, ids)
    check_y(x, x_o)
    del layers
    torch.cuda.empty_cache()

"""The tensor-core (tcgen05) grouped GEMM path against the CPU oracle.

By default every chosen expert runs as a grouped GEMM on the tensor cores;
with MOE_F_SPLIT_TC only the experts chosen by at least MOE_TC_MIN_ROUTES
routes do, the rest stream through the CUDA-core GEMV.  Shapes cover
several M tiles, K steps, token tiles (more than 128 routes on one expert)
and both activation dtypes.
"""
import numpy as np
import pytest
import torch

from moe_decode_layer_gemv_gb300 import synth
from _parity import check_y, layer_weights_np, oracle_layer_following

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, I, E, k, seed, x_bf16=False, skew=False):
    w = synth.Workload("tc", B=B, H=H, I=I, E=E, top_k=k, sigma_router=H ** -0.5, sigma_expert=0.05,
                       x_bf16=x_bf16, zipf_bias=skew)
    lw = {n: (v.to(DEV) if v is not None else None) for n, v in synth.make_layer(w, 0, seed=seed).items()}
    x = synth.make_x(w, 0, seed=seed).to(DEV)
    return lw, x


@pytest.mark.parametrize("B,H,I,E,k,x_bf16", [
    (16, 256, 128, 4, 2, False),
    (40, 512, 192, 6, 3, False),
    (64, 2048, 768, 8, 4, False),
    (24, 1024, 256, 5, 2, True),
    (300, 256, 64, 3, 2, False),   # > 128 routes on one expert: several token tiles
])
def test_forced_tensor_core_layer_matches_oracle(cuda_lib, B, H, I, E, k, x_bf16):
    lw, x = _case(B, H, I, E, k, seed=B + I, x_bf16=x_bf16)
    st = cuda_lib.new_status()
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k,
                                       flags=cuda_lib.MOE_F_FORCE_TC, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    rel = check_y(y, y_o)
    assert rel < 1e-4  # hi/lo split activations keep near-fp32 accuracy


def test_split_dispatch_skewed_routing(cuda_lib):
    """MOE_F_SPLIT_TC with skewed routing: popular experts (>= 8 routes) on
    the tensor cores, the rest on the CUDA-core streaming GEMV, in one layer."""
    B, H, I, E, k = 96, 1024, 256, 32, 4
    lw, x = _case(B, H, I, E, k, seed=4, skew=True)
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                       flags=cuda_lib.MOE_F_SPLIT_TC)
    torch.cuda.synchronize()
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=E)
    assert counts.max() >= cuda_lib.TC_MIN_ROUTES and (counts[counts > 0] < cuda_lib.TC_MIN_ROUTES).any()
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    check_y(y, y_o)


@pytest.mark.parametrize("B,E,k", [(15, 16, 4), (96, 32, 4)])
def test_default_runs_every_expert_on_the_tensor_cores(cuda_lib, B, E, k):
    """By default every chosen expert -- popular or not -- takes the
    tensor-core GEMM: the result is the forced one, bit for bit, and matches
    the oracle."""
    H, I = 1024, 256
    lw, x = _case(B, H, I, E, k, seed=4, skew=True)
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"])
    yf, idsf, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                         flags=cuda_lib.MOE_F_FORCE_TC | cuda_lib.MOE_F_SPLIT_TC)
    torch.cuda.synchronize()
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=E)
    assert counts.max() >= cuda_lib.TC_MIN_ROUTES and (counts[counts > 0] < cuda_lib.TC_MIN_ROUTES).any()
    assert torch.equal(ids, idsf) and torch.equal(y, yf)
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    check_y(y, y_o)


def test_tensor_core_and_gemv_paths_agree(cuda_lib):
    B, H, I, E, k = 128, 2048, 768, 16, 4
    lw, x = _case(B, H, I, E, k, seed=9)
    ya, ia, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k,
                                       flags=cuda_lib.MOE_F_FORCE_TC)
    yb, ib, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k,
                                       flags=cuda_lib.MOE_F_NO_TC)
    torch.cuda.synchronize()
    assert torch.equal(ia, ib)
    assert float((ya - yb).abs().max()) <= 1e-4 * float(yb.abs().max())


@pytest.mark.parametrize("split", [False, True])
def test_hot_expert_l2_policy_leaves_results_unchanged(cuda_lib, split):
    """MOE_F_HOT_L2 only changes the L2 eviction priority of the weight
    copies (evict_last for the experts with >= 8 routes, evict_first for
    the rest), on the tensor cores or the streaming GEMV: the layer's
    outputs are bit-identical with and without it."""
    B, H, I, E, k = 96, 1024, 256, 32, 4
    lw, x = _case(B, H, I, E, k, seed=6, skew=True)
    base = cuda_lib.MOE_F_SPLIT_TC if split else 0
    y0, i0, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                       flags=base)
    y1, i1, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                       flags=base | cuda_lib.MOE_F_HOT_L2)
    torch.cuda.synchronize()
    assert torch.equal(i0, i1) and torch.equal(y0, y1)
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, i1)
    check_y(y1, y_o)


@pytest.mark.parametrize("x_bf16", [False, True])
def test_unequal_items_snake_order_and_per_item_stages(cuda_lib, x_bf16):
    """A launch whose segments differ widely in size (one expert with more
    than 96 of the 128 tokens beside experts with at most 32): the GEMM
    ranks its segments by size, deals the items in a snake, and (fp32
    activations) packs two k-steps into a stage for the small experts'
    items.  The layer still matches the oracle and the CUDA-core path."""
    B, H, I, E, k = 128, 1024, 256, 64, 4
    lw, x = _case(B, H, I, E, k, seed=11, x_bf16=x_bf16, skew=True)
    y, ids, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"])
    yg, idsg, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                         flags=cuda_lib.MOE_F_NO_TC)
    torch.cuda.synchronize()
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=E)
    assert counts.max() > 96 and ((counts > 0) & (counts <= 32)).any()
    assert torch.equal(ids, idsg)
    assert float((y - yg).abs().max()) <= 1e-4 * float(yg.abs().max())
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    rel = check_y(y, y_o)
    assert rel < 1e-4

"""GPU path vs the CPU oracle, through the C ABI, on seeded inputs.

Sizes span several tiles with ragged tails; the workloads' own shapes are
covered at full size (sampled or whole where the oracle is fast enough).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import synth
from _parity import (check_grouping, check_layer_routing, check_route, check_y, layer_weights_np, np_x,
                     oracle_layer_following)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def make_case(B, H, I, E, k, seed=0, sigma_r=None, bias=False, x_bf16=False, device="cpu"):
    w = synth.Workload("case", B=B, H=H, I=I, E=E, top_k=k,
                       sigma_router=sigma_r if sigma_r is not None else H ** -0.5,
                       sigma_expert=0.02 if H >= 512 else 0.1, x_bf16=x_bf16, zipf_bias=bias)
    lw = synth.make_layer(w, 0, seed=seed, device=device)
    x = synth.make_x(w, 0, seed=seed, device=device)
    return w, {n: (v.to(DEV) if v is not None else None) for n, v in lw.items()}, x.to(DEV)


SHAPES = [
    # B, H, I, E, k
    (4, 64, 32, 8, 2),       # the tiny workload
    (1, 2048, 768, 128, 2),  # one layer of the 30-layer stack
    (5, 72, 40, 5, 3),       # ragged H and I (not multiples of 256), E < 32
    (13, 264, 24, 17, 4),    # ragged everything
    (9, 128, 64, 6, 6),      # top_k == E
    (3, 128, 64, 1, 1),      # one expert: a dense SwiGLU MLP
    (40, 256, 128, 12, 3),   # heavy reuse: many tokens per expert (> 8 per pass)
]


@pytest.mark.parametrize("B,H,I,E,k", SHAPES)
def test_route_parity(cuda_lib, B, H, I, E, k):
    _, lw, x = make_case(B, H, I, E, k, seed=B + H)
    ids, w, logits = cuda_lib.route(x, lw["w_router"], k)
    torch.cuda.synchronize()
    check_route(x, lw["w_router"], None, k, ids, w, logits)


@pytest.mark.parametrize("B,H,I,E,k", SHAPES)
def test_group_parity_bit_exact(cuda_lib, B, H, I, E, k):
    rng = np.random.default_rng(B * 7 + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    off_o, ridx_o, uniq_o = oracle.group(ids, E)
    st = cuda_lib.new_status()
    off, ridx, uniq, nu = cuda_lib.group_by_expert(torch.from_numpy(ids).to(DEV), E, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(off.cpu().numpy(), off_o)
    assert np.array_equal(ridx.cpu().numpy(), ridx_o)
    n = int(nu.item())
    assert n == len(uniq_o)
    assert np.array_equal(uniq.cpu().numpy()[:n], uniq_o)


@pytest.mark.parametrize("B", [1, 64, 300, 1024])
def test_group_parity_large_batches(cuda_lib, B):
    E, k = 256, 8
    rng = np.random.default_rng(B)
    # skewed: popular experts repeat heavily
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(B)]).astype(np.int32)
    off_o, ridx_o, uniq_o = oracle.group(ids, E)
    off, ridx, uniq, nu = cuda_lib.group_by_expert(torch.from_numpy(ids).to(DEV), E)
    torch.cuda.synchronize()
    assert np.array_equal(off.cpu().numpy(), off_o)
    assert np.array_equal(ridx.cpu().numpy(), ridx_o)
    assert np.array_equal(uniq.cpu().numpy()[:int(nu.item())], uniq_o)


def test_group_flags_bad_and_duplicate_ids(cuda_lib):
    ids = torch.tensor([[0, 3], [2, 9], [1, 1]], dtype=torch.int32, device=DEV)
    st = cuda_lib.new_status()
    cuda_lib.group_by_expert(ids, 8, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & cuda_lib.MOE_DEV_BAD_EXPERT_ID
    assert s & cuda_lib.MOE_DEV_DUP_EXPERT


@pytest.mark.parametrize("B,H,I,E,k", SHAPES)
@pytest.mark.parametrize("flags", [0, 2, 1])  # fused, unfused, no-dedup
def test_layer_parity(cuda_lib, B, H, I, E, k, flags):
    _, lw, x = make_case(B, H, I, E, k, seed=3 * B + I)
    st = cuda_lib.new_status()
    ws = cuda_lib.new_workspace(B, H, I, E, k)
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, flags=flags,
                                       workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lnp = layer_weights_np(lw)
    y_o, _, _ = oracle_layer_following(x, lnp, k, ids)
    check_y(y, y_o)
    # the routing and grouping this layer call itself used
    check_layer_routing(x, lw["w_router"], None, k, ids, w)
    if not flags & cuda_lib.MOE_F_NO_DEDUP:
        check_grouping(cuda_lib, ws, ids, B, H, I, E, k)
    ids_g, w_g, logits_g = cuda_lib.route(x, lw["w_router"], k)
    check_route(x, lw["w_router"], None, k, ids_g, w_g, logits_g)
    assert torch.equal(ids_g, ids)


def test_layer_with_bias_and_residual(cuda_lib):
    B, H, I, E, k = 16, 256, 96, 24, 6
    _, lw, x = make_case(B, H, I, E, k, seed=5, bias=True)
    res = torch.randn(B, H, device=DEV)
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw["bias"],
                                       residual=res)
    torch.cuda.synchronize()
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids, residual=res.cpu().numpy())
    check_y(y, y_o)
    check_layer_routing(x, lw["w_router"], lw["bias"], k, ids, w)


def test_bf16_activations(cuda_lib):
    B, H, I, E, k = 20, 512, 64, 16, 4
    _, lw, x = make_case(B, H, I, E, k, seed=9, x_bf16=True)
    assert x.dtype == torch.bfloat16
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k)
    torch.cuda.synchronize()
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    check_y(y, y_o)


def test_expert_forward_on_oracle_routing(cuda_lib):
    """moe_expert_forward fed the oracle's own routing and grouping."""
    B, H, I, E, k = 24, 320, 48, 10, 3
    _, lw, x = make_case(B, H, I, E, k, seed=12)
    lnp = layer_weights_np(lw)
    lo = oracle.router(np_x(x), lnp["w_router"])
    ids_o, w_o = oracle.topk(lo, k)
    off, ridx, uniq = oracle.group(ids_o, E)
    uniq_full = np.full(E, -1, np.int32)
    uniq_full[:len(uniq)] = uniq
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    grouping = (t(off), t(ridx), t(uniq_full), t(np.array([len(uniq)], np.int32)))
    for flags in (0, 1):
        y = cuda_lib.expert_forward(x, lw["gate_up"], lw["down"], t(ids_o), t(w_o), grouping, flags=flags)
        torch.cuda.synchronize()
        y_o = oracle.experts(np_x(x), lnp["gate_up"], lnp["down"], ids_o, w_o, E)
        check_y(y, y_o)


def test_dedup_and_no_dedup_agree(cuda_lib):
    B, H, I, E, k = 32, 512, 128, 8, 4
    _, lw, x = make_case(B, H, I, E, k, seed=21)
    y0, i0, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, flags=0)
    y1, i1, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, flags=1)
    torch.cuda.synchronize()
    assert torch.equal(i0, i1)
    assert torch.allclose(y0, y1, rtol=0, atol=1e-5 * float(y0.abs().max()))


def test_empty_batch_is_a_no_op(cuda_lib):
    B, H, I, E, k = 0, 64, 32, 8, 2
    _, lw, _ = make_case(4, H, I, E, k)
    x = torch.empty((0, H), device=DEV)
    y, ids, w = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k)
    torch.cuda.synchronize()
    assert y.shape == (0, H)


def test_deterministic_across_calls(cuda_lib):
    B, H, I, E, k = 64, 2048, 768, 256, 8
    _, lw, x = make_case(B, H, I, E, k, seed=1)
    ya, ia, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k)
    yb, ib, _ = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k)
    torch.cuda.synchronize()
    assert torch.equal(ia, ib) and torch.equal(ya, yb)


@pytest.mark.parametrize("B,k,E", [(1, 2, 128), (4, 8, 256), (3, 6, 256), (2, 8, 64)])
def test_persistent_decode_kernel_is_stable_over_repeated_runs(cuda_lib, B, k, E):
    """The small-batch layer runs in one persistent kernel whose phases hand
    data over through device-wide barriers; a missing ordering would show up
    as an occasional wrong token.  Many seeds, compared with the phase-by-phase
    CUDA-core kernels (each checked against the oracle above; fp32 throughout,
    like the persistent kernel, so the two agree to 1e-5)."""
    H, I = 2048, 768
    w = synth.Workload("rep", B=B, H=H, I=I, E=E, top_k=k, sigma_router=H ** -0.5)
    lw = synth.make_layer(w, 0, seed=7, device=DEV)
    for step in range(40):
        x = synth.make_x(w, step, seed=7, device=DEV)
        y0, i0, w0 = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k)
        y1, i1, w1 = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k,
                                            flags=cuda_lib.MOE_F_UNFUSED | cuda_lib.MOE_F_NO_TC)
        torch.cuda.synchronize()
        assert torch.equal(i0, i1), step
        assert float((w0 - w1).abs().max()) <= 1e-6
        assert float((y0 - y1).abs().max()) <= 1e-5 * float(y1.abs().max()), step


def test_persistent_stack_is_stable_over_repeated_runs(cuda_lib):
    H, I, E, k, L = 2048, 768, 128, 2, 6
    w = synth.Workload("rep", B=1, H=H, I=I, E=E, top_k=k, layers=L)
    layers = [synth.make_layer(w, l, seed=3, device=DEV) for l in range(L)]
    sw = cuda_lib.StackWeights(layers)
    for step in range(30):
        x = synth.make_x(w, step, seed=3, device=DEV)
        xa, ia = cuda_lib.stack_forward(x, sw, k)
        xb, ib = cuda_lib.stack_forward(x, sw, k, flags=cuda_lib.MOE_F_UNFUSED | cuda_lib.MOE_F_NO_TC)
        torch.cuda.synchronize()
        assert torch.equal(ia, ib), step
        assert float((xa - xb).abs().max()) <= 1e-5 * float(xb.abs().max()), step


def test_stack_captured_in_a_cuda_graph(cuda_lib):
    """No host synchronisation anywhere in a stack forward: the whole call
    (the workspace clear and the persistent kernel) is captured into a CUDA
    graph, and each replay gives the direct call's result on new inputs."""
    H, I, E, k, L = 2048, 768, 128, 2, 4
    w = synth.Workload("graph", B=1, H=H, I=I, E=E, top_k=k, layers=L)
    layers = [synth.make_layer(w, l, seed=5, device=DEV) for l in range(L)]
    sw = cuda_lib.StackWeights(layers)
    ws = cuda_lib.new_workspace(1, H, I, E, k, DEV)
    st = cuda_lib.new_status(DEV)
    xbuf = torch.empty((1, H), dtype=torch.float32, device=DEV)
    ids = torch.empty((L, 1, k), dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        xbuf.copy_(synth.make_x(w, 0, seed=5, device=DEV))
        cuda_lib.stack_forward_(xbuf, sw, k, ids_out=ids, workspace=ws, status=st, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.stack_forward_(xbuf, sw, k, ids_out=ids, workspace=ws, status=st,
                                stream=torch.cuda.current_stream())
    for step in range(1, 4):
        x = synth.make_x(w, step, seed=5, device=DEV)
        xbuf.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        xr, ir = cuda_lib.stack_forward(x, sw, k)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(ids, ir), step
        assert torch.equal(xbuf, xr), step

"""The five workloads at full size, in the launch configuration the benchmark
times (the fused persistent kernel), against the CPU oracle.

Weights are drawn on the GPU by torch's generator (synth recipe) and the
oracle reads back exactly the tensors it needs: every router, and the
experts its own routing selects.  Where the oracle would take minutes
(prefill-sized layer), outputs are sampled token by token.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import accounting, synth
from _parity import (NEAR_TIE, check_grouping, check_layer_routing, check_route, check_y, margins, np_x,
                     oracle_layer_following)

pytestmark = pytest.mark.gpu
DEV = "cuda"


class LazyExperts(dict):
    """{e: uint16 array} filled on demand from a device tensor [E, ...]."""

    def __init__(self, dev_tensor):
        super().__init__()
        self.t = dev_tensor

    def need(self, ids):
        for e in np.unique(ids):
            e = int(e)
            if e not in self:
                self[e] = synth.bf16_bits(self.t[e])
        return self


def oracle_layer_lazy(x, lw, k, ids_gpu, residual=None, tokens=None):
    """Oracle y for the given tokens (all by default), fetching only the
    selected experts; near ties follow the GPU's ids."""
    xn = np_x(x)
    wr = synth.bf16_bits(lw["w_router"])
    bias = None if lw.get("bias") is None else lw["bias"].cpu().numpy()
    lo = oracle.router(xn, wr, bias)
    ids_o, w_o = oracle.topk(lo, k)
    ex = margins(lo, k) < NEAR_TIE
    ig = ids_gpu.cpu().numpy()
    tok = np.arange(xn.shape[0]) if tokens is None else np.asarray(tokens)
    lnp = {"w_router": wr, "bias": bias,
           "gate_up": LazyExperts(lw["gate_up"]), "down": LazyExperts(lw["down"])}
    ids_use = np.where(ex[:, None], ig, ids_o)
    lnp["gate_up"].need(ids_use[tok])
    lnp["down"].need(ids_use[tok])
    sub = {"w_router": wr, "bias": bias, "gate_up": lnp["gate_up"], "down": lnp["down"]}
    res = None if residual is None else residual[tok]
    xs = x[torch.as_tensor(tok, device=x.device)]
    y, _, n_ex = oracle_layer_following(xs, sub, k, ids_gpu[torch.as_tensor(tok, device=x.device)],
                                        residual=res)
    return y, ids_o, ex


def run_layer(cuda_lib, w, lw, x, flags=0):
    """The layer in the benchmark's launch configuration; also checks the
    routing weights it returned and the grouping it left in its workspace."""
    st = cuda_lib.new_status()
    B = x.shape[0]
    ws = cuda_lib.new_workspace(B, w.H, w.I, w.E, w.top_k)
    y, ids, rw = cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], w.top_k,
                                        bias=lw.get("bias"), workspace=ws, status=st, flags=flags)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_layer_routing(x, lw["w_router"], lw.get("bias"), w.top_k, ids, rw)
    check_grouping(cuda_lib, ws, ids, B, w.H, w.I, w.E, w.top_k)
    return y, ids, rw


@pytest.fixture(scope="module")
def uniform_layer():
    w = synth.UNIFORM
    lw = synth.make_layer(w, 0, seed=0, device=DEV)
    yield w, lw
    del lw
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", synth.UNIFORM.batches)
def test_uniform_routing_layer(cuda_lib, uniform_layer, B):
    w, lw = uniform_layer
    x = synth.make_x(w, 0, seed=0, device=DEV, B=B)
    y, ids, rw = run_layer(cuda_lib, w, lw, x)
    ids_r, w_r, lg = cuda_lib.route(x, lw["w_router"], w.top_k)
    torch.cuda.synchronize()
    check_route(x, lw["w_router"], None, w.top_k, ids_r, w_r, lg)
    y_o, _, ex = oracle_layer_lazy(x, lw, w.top_k, ids)
    check_y(y, y_o)
    U = len(np.unique(ids.cpu().numpy()))
    # unique count inside a generous band around the closed form
    assert abs(U - accounting.expected_unique(256, 8, B)) <= 6 * np.sqrt(max(B, 1)) + 2


@pytest.mark.parametrize("B", [5, 16, 64])
def test_uniform_layer_split_dispatch(cuda_lib, uniform_layer, B):
    """MOE_F_SPLIT_TC: the experts with fewer than MOE_TC_MIN_ROUTES routes
    stream through the CUDA-core grouped GEMV, the others (if any) take the
    tensor cores."""
    w, lw = uniform_layer
    x = synth.make_x(w, 0, seed=B, device=DEV, B=B)
    y, ids, rw = run_layer(cuda_lib, w, lw, x, flags=cuda_lib.MOE_F_SPLIT_TC)
    y_o, _, ex = oracle_layer_lazy(x, lw, w.top_k, ids)
    check_y(y, y_o)


@pytest.fixture(scope="module")
def skewed_layer():
    w = synth.SKEWED
    lw = synth.make_layer(w, 0, seed=0, device=DEV)
    yield w, lw
    del lw
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", synth.SKEWED.batches)
def test_skewed_routing_layer(cuda_lib, skewed_layer, B):
    w, lw = skewed_layer
    x = synth.make_x(w, 0, seed=0, device=DEV, B=B)
    y, ids, rw = run_layer(cuda_lib, w, lw, x)
    y_o, _, ex = oracle_layer_lazy(x, lw, w.top_k, ids)
    check_y(y, y_o)
    # the grouped route list of the layer's own ids, bit-exact
    off, ridx, uniq, nu = cuda_lib.group_by_expert(ids, w.E)
    torch.cuda.synchronize()
    off_o, ridx_o, uniq_o = oracle.group(ids.cpu().numpy(), w.E)
    assert np.array_equal(off.cpu().numpy(), off_o) and np.array_equal(ridx.cpu().numpy(), ridx_o)
    assert np.array_equal(uniq.cpu().numpy()[:int(nu.item())], uniq_o)


def test_prefill_sized_layer_every_row(cuda_lib):
    """All 512 tokens of the prefill-sized layer (every expert's tensor-core
    tiles) against the oracle, which evaluates the whole layer here."""
    w = synth.PREFILL
    lw = synth.make_layer(w, 0, seed=0, device=DEV)
    x = synth.make_x(w, 0, seed=0, device=DEV)
    y, ids, rw = run_layer(cuda_lib, w, lw, x)
    ids_r, w_r, lg = cuda_lib.route(x, lw["w_router"], w.top_k)
    torch.cuda.synchronize()
    check_route(x, lw["w_router"], None, w.top_k, ids_r, w_r, lg)
    y_o, _, _ = oracle_layer_lazy(x, lw, w.top_k, ids)
    check_y(y, y_o)
    del lw
    torch.cuda.empty_cache()


def test_stack_of_30_layers_end_to_end(cuda_lib):
    w = synth.STACK
    layers = [synth.make_layer(w, l, seed=0, device=DEV) for l in range(w.layers)]
    x0 = synth.make_x(w, 0, seed=0, device=DEV)
    st = cuda_lib.new_status()
    xs = cuda_lib.StackWeights(layers)
    x_out, ids = cuda_lib.stack_forward(x0, xs, w.top_k, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # oracle walks the same 30 layers, following the GPU only on near ties
    x = x0.clone()
    n_ties = 0
    for l, lw in enumerate(layers):
        y_o, ids_o, ex = oracle_layer_lazy(x, lw, w.top_k, ids[l], residual=x.cpu().numpy())
        n_ties += int(ex.sum())
        ig = ids[l].cpu().numpy()
        # in order (descending logit), unless the two selected logits are
        # within the near-tie margin of each other
        lo = oracle.router(np_x(x), synth.bf16_bits(lw["w_router"]))
        srt = -np.sort(-lo.astype(np.float64), axis=1)[:, :w.top_k]
        inner = np.any(np.diff(srt, axis=1) > -NEAR_TIE, axis=1)
        strict = ~ex & ~inner
        assert np.array_equal(ig[strict], ids_o[strict]), l
        assert np.array_equal(np.sort(ig[~ex], 1), np.sort(ids_o[~ex], 1)), l
        x = torch.from_numpy(y_o).to(DEV)
    check_y(x_out, x.cpu().numpy())
    del layers
    torch.cuda.empty_cache()


def test_dense_stack_of_30_layers_end_to_end(cuda_lib):
    """The dense counterpart of the stack (one expert, top-1: a SwiGLU MLP
    per layer with routing weight 1) through the same stack entry point,
    layer by layer against the oracle and end to end."""
    w = synth.DENSE
    layers = [synth.make_layer(w, l, seed=0, device=DEV) for l in range(w.layers)]
    x0 = synth.make_x(w, 0, seed=0, device=DEV)
    st = cuda_lib.new_status()
    x_out, ids = cuda_lib.stack_forward(x0, cuda_lib.StackWeights(layers), w.top_k, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ids.abs().sum()) == 0  # the only expert, every layer
    lnp = [{"w_router": synth.bf16_bits(lw["w_router"]), "gate_up": synth.bf16_bits(lw["gate_up"]),
            "down": synth.bf16_bits(lw["down"])} for lw in layers]
    x_o, ids_o = oracle.stack(x0.cpu().numpy(), lnp, w.top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    check_y(x_out, x_o)
    del layers
    torch.cuda.empty_cache()

"""moe_expert_forward_noalloc: the expert pass for callers that cannot
allocate device memory.

Some callers cannot call cudaMalloc at all -- code inside a CUDA graph that
is being captured, an allocator hook, a runtime with a fixed memory budget --
so the library offers one expert-pass entry point whose scratch is a fixed
array inside the library.  Its results must match the oracle (and the
workspace version of the same pass).  Two calls in a row, with different
problems, check that the shared array's leftover contents from one call never
leak into the next; the size limit is checked at the exact fit and just past
it.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_layer_gemv_gb300 import synth
from _parity import Y_TOL, check_y, layer_weights_np, np_x

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, I, E, k, seed):
    w = synth.Workload("noalloc", B=B, H=H, I=I, E=E, top_k=k, sigma_router=H ** -0.5,
                       sigma_expert=0.05)
    lw = {n: (v.to(DEV) if v is not None else None) for n, v in synth.make_layer(w, 0, seed=seed).items()}
    x = synth.make_x(w, 0, seed=seed).to(DEV)
    return lw, x


def _oracle_routing(lw, x, k):
    """The oracle's routing and grouping, as device tensors for the call."""
    lnp = layer_weights_np(lw)
    E = lnp["w_router"].shape[0]
    lo = oracle.router(np_x(x), lnp["w_router"])
    ids_o, w_o = oracle.topk(lo, k)
    off, ridx, uniq = oracle.group(ids_o, E)
    uniq_full = np.full(E, -1, np.int32)
    uniq_full[:len(uniq)] = uniq
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    grouping = (t(off), t(ridx), t(uniq_full), t(np.array([len(uniq)], np.int32)))
    return lnp, ids_o, w_o, t(ids_o), t(w_o), grouping


def _check_against_oracle(api, lw, x, k):
    lnp, ids_o, w_o, ids, w, grouping = _oracle_routing(lw, x, k)
    st = api.new_status()
    y = torch.full((x.shape[0], x.shape[1]), float("nan"), device=DEV)
    api.expert_forward_noalloc(x, lw["gate_up"], lw["down"], ids, w, grouping, out=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    E = lnp["w_router"].shape[0]
    y_o = oracle.experts(np_x(x), lnp["gate_up"], lnp["down"], ids_o, w_o, E)
    check_y(y, y_o)
    return y


def _check_against_workspace_version(api, lw, x, k):
    E = lw["w_router"].shape[0]
    ids, w, _ = api.route(x, lw["w_router"], k)
    grouping = api.group_by_expert(ids, E)
    st = api.new_status()
    ref = api.expert_forward(x, lw["gate_up"], lw["down"], ids, w, grouping, status=st)
    y = torch.full_like(ref, float("nan"))
    api.expert_forward_noalloc(x, lw["gate_up"], lw["down"], ids, w, grouping, out=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    r = ref.cpu().numpy()
    g = y.cpu().numpy()
    assert np.all(np.isfinite(g))
    assert float(np.max(np.abs(g - r))) <= Y_TOL * float(np.max(np.abs(r)))


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(cuda_lib):
    # first call: 192 routes (h and o take about 0.55 MB of the array); the
    # second, a different and smaller problem, reuses the array with the
    # first call's values still in it
    lw, x = _case(48, 512, 192, 16, 4, seed=3)
    _check_against_oracle(cuda_lib, lw, x, 4)
    lw2, x2 = _case(5, 264, 40, 9, 3, seed=4)
    _check_against_oracle(cuda_lib, lw2, x2, 3)
    _check_against_workspace_version(cuda_lib, lw2, x2, 3)


def test_noalloc_accepts_a_problem_that_fills_its_array_exactly(cuda_lib):
    # R = 1024 routes, H = I = 2048: h [R, I] and o [R, H] in fp32 take
    # 8 MiB each, the whole 16 MiB array
    B, H, I, E, k = 128, 2048, 2048, 16, 8
    assert 4 * B * k * I + 4 * B * k * H == cuda_lib.NOALLOC_SCRATCH_BYTES
    lw, x = _case(B, H, I, E, k, seed=5)
    _check_against_workspace_version(cuda_lib, lw, x, k)


def _raw_call(api, B, H, I, E, k, flags=0):
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    p = dummy.data_ptr()
    return api._lib.moe_expert_forward_noalloc(p, 0, p, p, p, p, p, p, p, p, B, H, I, E, k, None, p, flags,
                                               None, None)


def test_noalloc_rejects_problems_larger_than_its_array(cuda_lib):
    # one step (8 columns of I) past the exact fit, and far past it: refused
    # before anything is enqueued (the dummy pointers are never read)
    assert _raw_call(cuda_lib, 128, 2048, 2056, 16, 8) == cuda_lib.MOE_ERR_WORKSPACE
    assert _raw_call(cuda_lib, 1024, 4096, 1536, 256, 8) == cuda_lib.MOE_ERR_WORKSPACE


def test_noalloc_refuses_the_tensor_core_flag(cuda_lib):
    assert _raw_call(cuda_lib, 4, 64, 32, 8, 2, flags=cuda_lib.MOE_F_FORCE_TC) == cuda_lib.MOE_ERR_UNSUPPORTED

"""moe_expert_forward_noalloc against moe_expert_forward.

Some callers cannot call cudaMalloc at all -- code inside a CUDA graph that
is being captured, an allocator hook, a runtime with a fixed memory budget --
so the library offers one expert-pass entry point whose scratch is a fixed
array inside the library.  Its results must match the workspace version.
Two calls in a row (with different problems) check that the shared array's
leftover contents from one call never leak into the next.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from moe_decode_layer_gemv_gb300 import synth
from _parity import Y_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, I, E, k, seed):
    w = synth.Workload("noalloc", B=B, H=H, I=I, E=E, top_k=k, sigma_router=H ** -0.5,
                       sigma_expert=0.05)
    lw = {n: (v.to(DEV) if v is not None else None) for n, v in synth.make_layer(w, 0, seed=seed).items()}
    x = synth.make_x(w, 0, seed=seed).to(DEV)
    return lw, x


def _compare(api, lw, x, k):
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


def test_noalloc_matches_workspace_version_on_two_calls_in_a_row(cuda_lib):
    # first call: many routes (fills much of the array); second: a different,
    # smaller problem that reuses the array with stale contents in it
    lw, x = _case(48, 512, 192, 16, 4, seed=3)
    _compare(cuda_lib, lw, x, 4)
    lw2, x2 = _case(5, 264, 40, 9, 3, seed=4)
    _compare(cuda_lib, lw2, x2, 3)


def test_noalloc_rejects_problems_larger_than_its_array(cuda_lib):
    B, H, I, E, k = 1024, 4096, 1536, 256, 8  # 4*R*(H+I) bytes >> 16 MiB
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    rc = cuda_lib._lib.moe_expert_forward_noalloc(
        dummy.data_ptr(), 0, dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
        dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), B, H, I, E, k, None,
        dummy.data_ptr(), 0, None, None)
    assert rc == cuda_lib.MOE_ERR_WORKSPACE

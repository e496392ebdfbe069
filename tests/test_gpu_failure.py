"""Failure detection on the GPU without a GPU fault: the device-wide
barriers of the persistent kernels are bounded waits.  With the injection
hook on, each barrier waits for arrivals that never come; the wait runs out
(about a second), the kernel records MOE_DEV_TIMEOUT in the status word and
returns, and the context stays usable -- the same call then runs clean and
matches the oracle."""
import time

import pytest
import torch

from moe_decode_layer_gemv_gb300 import synth
from _parity import check_y, layer_weights_np, oracle_layer_following

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(B, H, I, E, k, seed):
    w = synth.Workload("case", B=B, H=H, I=I, E=E, top_k=k, sigma_router=H ** -0.5, sigma_expert=0.05)
    lw = synth.make_layer(w, 0, seed=seed, device=DEV)
    x = synth.make_x(w, 0, seed=seed, device=DEV)
    return lw, x


def _timed_out_then_clean(api, run):
    st = api.new_status()
    api.inject_barrier_stall(1)
    try:
        t0 = time.perf_counter()
        run(st)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        api.inject_barrier_stall(0)
    assert int(st.item()) & api.MOE_DEV_TIMEOUT, int(st.item())
    assert elapsed < 60.0
    st2 = api.new_status()
    out = run(st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    return out


@pytest.mark.parametrize("B,flags", [(1, 0), (4, 0), (24, 8)])  # decode kernel x2, general fused kernel
def test_layer_barrier_timeout_reports_and_recovers(cuda_lib, B, flags):
    H, I, E, k = 256, 96, 16, 2
    lw, x = _case(B, H, I, E, k, seed=B)

    def run(st):
        return cuda_lib.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, flags=flags, status=st)

    y, ids, _ = _timed_out_then_clean(cuda_lib, run)
    y_o, _, _ = oracle_layer_following(x, layer_weights_np(lw), k, ids)
    check_y(y, y_o)


def test_stack_barrier_timeout_reports_and_recovers(cuda_lib):
    w = synth.Workload("stack3", B=1, H=512, I=128, E=32, top_k=2, layers=3, residual=True,
                       sigma_router=512 ** -0.5, sigma_expert=0.05)
    layers = [synth.make_layer(w, l, seed=1, device=DEV) for l in range(3)]
    sw = cuda_lib.StackWeights(layers)
    x = synth.make_x(w, 0, seed=1, device=DEV)

    def run(st):
        return cuda_lib.stack_forward(x, sw, w.top_k, status=st)

    xa, ia = _timed_out_then_clean(cuda_lib, run)
    xb, ib = cuda_lib.stack_forward(x, sw, w.top_k, flags=cuda_lib.MOE_F_UNFUSED | cuda_lib.MOE_F_NO_TC)
    torch.cuda.synchronize()
    assert torch.equal(ia, ib)
    assert float((xa - xb).abs().max()) <= 1e-5 * float(xb.abs().max())


def test_stack_flags_router_values_beyond_the_fixed_point_range(cuda_lib):
    """The decode kernel sums the router's per-CTA partial logits in counted
    fixed-point words; a partial beyond their range is clamped and reported
    (MOE_DEV_RANGE), never a wait that runs out, and the next call is clean."""
    w = synth.Workload("stack2", B=1, H=512, I=128, E=32, top_k=2, layers=2, residual=True,
                       sigma_router=512 ** -0.5, sigma_expert=0.05)
    layers = [synth.make_layer(w, l, seed=2, device=DEV) for l in range(2)]
    sw = cuda_lib.StackWeights(layers)
    x = synth.make_x(w, 0, seed=2, device=DEV)
    st = cuda_lib.new_status()
    t0 = time.perf_counter()
    cuda_lib.stack_forward(x * 1e8, sw, w.top_k, status=st)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    v = int(st.item())
    assert v & cuda_lib.MOE_DEV_RANGE, v
    assert v & ~(cuda_lib.MOE_DEV_RANGE | cuda_lib.MOE_DEV_NONFINITE) == 0, v
    st2 = cuda_lib.new_status()
    cuda_lib.stack_forward(x, sw, w.top_k, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0

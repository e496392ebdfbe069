"""The Python binding on the CPU: it marshals arguments only, so every check
it makes happens before any launch, and it never computes a result itself
(a CPU tensor is refused, not evaluated)."""
import re
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    from moe_decode_layer_gemv_gb300 import build
    build.build()
    from moe_decode_layer_gemv_gb300 import api as a
    return a


def test_binding_names_every_declared_entry_point(api):
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    declared = set(re.findall(r"^\s*(?:const\s+)?(?:\w+\s+)*\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M))
    assert declared == set(api.EXPORTED)


def test_cpu_tensors_are_refused_not_computed(api):
    B, H, I, E, k = 2, 64, 32, 8, 2
    x = torch.zeros(B, H)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    gu = torch.zeros(E, 2 * I, H, dtype=torch.bfloat16)
    dn = torch.zeros(E, H, I, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.layer_forward(x, wr, gu, dn, k)
    with pytest.raises(TypeError):  # x must be fp32 or bf16
        api.layer_forward(x.double(), wr, gu, dn, k)


def test_every_entry_point_checks_its_tensors_before_any_launch(api):
    B, H, I, E, k = 2, 64, 32, 8, 2
    x = torch.zeros(B, H)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.route(x, wr, k)
    with pytest.raises(ValueError):
        api.group_by_expert(torch.zeros(B, k, dtype=torch.int32), E)
    with pytest.raises(ValueError):
        api.stack_forward_(x, None, k)
    gu = torch.zeros(E, 2 * I, H, dtype=torch.bfloat16)
    dn = torch.zeros(E, H, I, dtype=torch.bfloat16)
    ids = torch.zeros(B, k, dtype=torch.int32)
    grouping = tuple(torch.zeros(n, dtype=torch.int32) for n in (E + 1, B * k, E, 1))
    with pytest.raises(ValueError):
        api.expert_forward(x, gu, dn, ids, torch.zeros(B, k), grouping)
    with pytest.raises(ValueError):
        api.expert_forward_noalloc(x, gu, dn, ids, torch.zeros(B, k), grouping)
    with pytest.raises(TypeError):  # x must be fp32 or bf16
        api.route(x.double(), wr, k)


def test_host_errors_raise_with_their_status(api):
    with pytest.raises(api.MoeError) as e:
        api.workspace_bytes(4, 2048, 768, 300, 8)  # E above the maximum
    assert e.value.code == api.MOE_ERR_INVALID_ARG
    with pytest.raises(api.MoeError):
        api.inject_barrier_stall(-1)
    api.inject_barrier_stall(0)


def test_workspace_grows_with_the_batch(api):
    a = api.workspace_bytes(1, 2048, 768, 128, 2)
    b = api.workspace_bytes(64, 2048, 768, 256, 8)
    assert 0 < a < b
    # at least the per-route scratch: h [R, I] and o [R, H] in fp32
    assert b >= 64 * 8 * (768 + 2048) * 4


def test_status_strings_name_the_device_bits(api):
    assert "timed out" in api.status_string(api.MOE_DEV_TIMEOUT)
    assert api.status_string(api.MOE_OK)


def test_mismatched_shapes_are_refused_before_any_launch(api):
    """A buffer shorter than the problem needs would be read or written out
    of bounds on the device: every shape is checked in the binding first."""
    B, H, I, E, k = 3, 64, 32, 8, 2
    x = torch.zeros(B, H)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    gu = torch.zeros(E, 2 * I, H, dtype=torch.bfloat16)
    dn = torch.zeros(E, H, I, dtype=torch.bfloat16)
    ids = torch.zeros(B, k, dtype=torch.int32)
    rw = torch.zeros(B, k)
    grouping = tuple(torch.zeros(n, dtype=torch.int32) for n in (E + 1, B * k, E, 1))
    shape = "shape"
    with pytest.raises(ValueError, match=shape):  # gate_up's H disagrees with x
        api.layer_forward(x, wr, gu[:, :, :32], dn, k)
    with pytest.raises(ValueError, match=shape):  # down's I disagrees with gate_up
        api.layer_forward(x, wr, gu, dn[:, :, :16], k)
    with pytest.raises(ValueError, match=shape):  # router rows != E
        api.layer_forward(x, wr[:4], gu, dn, k)
    with pytest.raises(ValueError, match=shape):  # out too small
        api.layer_forward(x, wr, gu, dn, k, out=torch.zeros(B - 1, H))
    with pytest.raises(ValueError, match=shape):  # ids_out of the wrong top_k
        api.layer_forward(x, wr, gu, dn, k, ids_out=torch.zeros(B, k + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match=shape):  # bias of the wrong length
        api.route(x, wr, k, bias=torch.zeros(E - 1))
    for bad in ((torch.zeros(E, dtype=torch.int32),) + grouping[1:],          # offsets [E] < E+1
                grouping[:1] + (torch.zeros(B * k - 1, dtype=torch.int32),) + grouping[2:],  # route_idx
                grouping[:3] + (torch.zeros(0, dtype=torch.int32),)):         # num_unique
        with pytest.raises(ValueError, match=shape):
            api.expert_forward(x, gu, dn, ids, rw, bad)
        with pytest.raises(ValueError, match=shape):
            api.expert_forward_noalloc(x, gu, dn, ids, rw, bad)
    with pytest.raises(ValueError, match=shape):  # route_w of the wrong shape
        api.expert_forward(x, gu, dn, ids, rw[:, :1], grouping)
    with pytest.raises(ValueError, match="required"):
        api.expert_forward_noalloc(x, gu, dn, None, rw, grouping)
    with pytest.raises(ValueError, match=shape):  # residual too small
        api.expert_forward(x, gu, dn, ids, rw, grouping, residual=torch.zeros(B, H // 2))

"""The C ABI library builds, loads and exports every entry point declared in
include/moe.h; host-side argument checks reject bad calls before any CUDA
work is enqueued (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

from moe_decode_layer_gemv_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?(?:\w+\s+)*\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "moe_layer_forward" in names and "moe_stack_forward" in names
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes_host_only(lib):
    n = ctypes.c_size_t(0)
    lib.moe_workspace_bytes.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
    assert lib.moe_workspace_bytes(64, 2048, 768, 256, 8, ctypes.byref(n)) == 0
    # scratch holds at least h [R, I] and o [R, H] in fp32
    assert n.value >= 512 * (768 + 2048) * 4
    assert lib.moe_workspace_bytes(4, 2048, 768, 300, 8, ctypes.byref(n)) == -1  # E too large
    assert lib.moe_workspace_bytes(4, 2048, 768, 256, 9, ctypes.byref(n)) == -1  # top_k too large
    assert lib.moe_workspace_bytes(4, 2044, 768, 256, 8, ctypes.byref(n)) == -1  # H % 8
    assert lib.moe_workspace_bytes(4, 2048, 768, 4, 5, ctypes.byref(n)) == -1   # top_k > E
    assert lib.moe_workspace_bytes(2048, 2048, 768, 256, 8, ctypes.byref(n)) == -1  # B > max


def test_bad_arguments_are_rejected_before_any_launch(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.moe_route.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, ctypes.c_size_t, P, P]
    good = P(0x10000)
    odd = P(0x10004)
    # null x
    assert lib.moe_route(None, 0, good, None, 4, 64, 8, 2, good, good, good, None, 0, None, None) == -1
    # misaligned pointer
    assert lib.moe_route(odd, 0, good, None, 4, 64, 8, 2, good, good, good, None, 0, None, None) == -1
    # unknown dtype
    assert lib.moe_route(good, 7, good, None, 4, 64, 8, 2, good, good, good, None, 0, None, None) == -1
    # no logits buffer and no workspace
    assert lib.moe_route(good, 0, good, None, 4, 64, 8, 2, good, good, None, None, 0, None, None) == -4
    lib.moe_group_by_expert.argtypes = [P, I, I, I, P, P, P, P, P, P]
    assert lib.moe_group_by_expert(good, 4, 0, 8, good, good, good, good, None, None) == -1
    lib.moe_stack_forward.argtypes = [I, P, P, P, P, I, I, I, I, I, P, P, ctypes.c_uint32, P,
                                      ctypes.c_size_t, P, P]
    assert lib.moe_stack_forward(0, None, None, None, None, 1, 64, 32, 8, 2, good, None, 0, good, 1 << 20,
                                 None, None) == -1


def test_injection_hook_range_checked(lib):
    lib.moe_inject_barrier_stall.argtypes = [ctypes.c_int]
    assert lib.moe_inject_barrier_stall(-1) == -1
    assert lib.moe_inject_barrier_stall(1025) == -1
    assert lib.moe_inject_barrier_stall(0) == 0


def test_status_strings(lib):
    lib.moe_status_string.restype = ctypes.c_char_p
    assert b"invalid" in lib.moe_status_string(-1)
    assert b"workspace" in lib.moe_status_string(-4)
    assert b"timed out" in lib.moe_status_string(1)


def test_binding_constants_match_the_header():
    """Every integer constant of include/moe.h that the Python binding mirrors
    (as MOE_X or as X) has the header's value."""
    from moe_decode_layer_gemv_gb300 import api
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    checked = 0
    for name, val in re.findall(r"^#define\s+(MOE_\w+)\s+(-?\d+)u?\b", src, flags=re.M):
        for attr in (name, name[len("MOE_"):]):
            if hasattr(api, attr):
                assert getattr(api, attr) == int(val), name
                checked += 1
                break
    assert checked >= 15 and api.MOE_F_SPLIT_TC == 64 and api.TC_MIN_ROUTES == 8

"""Python binding of libmoe.so -- argument marshalling only.

Every step of the layer runs in the CUDA library; this module allocates the
output tensors and the workspace with torch (device memory and streams are
all torch is used for) and passes raw pointers through the C ABI declared in
``include/moe.h``.  It raises ImportError when the library has not been
built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

if not os.path.exists(_build.LIB):
    raise ImportError(f"{_build.LIB} is missing: build it first with "
                      "moe_decode_layer_gemv_gb300.build.build()")

_lib = ctypes.CDLL(_build.LIB)
LIB_PATH = _build.LIB

_P = ctypes.c_void_p
_I = ctypes.c_int
_U = ctypes.c_uint32
_S = ctypes.c_size_t

_lib.moe_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_S)]
_lib.moe_route.argtypes = [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P, _P]
_lib.moe_group_by_expert.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
_lib.moe_expert_forward.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                    _P, _P, _U, _P, _S, _P, _P]
_lib.moe_expert_forward_noalloc.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                            _I, _P, _P, _U, _P, _P]
_lib.moe_layer_forward.argtypes = [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _U,
                                   _P, _S, _P, _P]
_lib.moe_stack_forward.argtypes = [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _U, _P, _S, _P, _P]
_lib.moe_stack_forward_fp8.argtypes = [_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _U, _P, _S, _P,
                                       _P]
_lib.moe_stack_forward_nvfp4.argtypes = [_I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _U, _P,
                                         _S, _P, _P]
_lib.moe_stack_forward_norm.argtypes = [_I, _P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _I, _I, _I, _P, _P, _U,
                                        _P, _S, _P, _P]
_lib.moe_workspace_grouping.argtypes = [_P, _S, _I, _I, _I, _I, _I, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                        ctypes.POINTER(_P), ctypes.POINTER(_P)]
_lib.moe_forward_path.argtypes = [_I, _I, _I, _I, _I, _I, _U, ctypes.POINTER(_I), ctypes.POINTER(_I)]
_lib.moe_forward_path.restype = ctypes.c_int
_lib.moe_launch_count.argtypes = []
_lib.moe_launch_count.restype = ctypes.c_ulonglong
_lib.moe_set_trace_buffer.argtypes = [_P, _I]
_lib.moe_set_trace_buffer.restype = ctypes.c_int
_lib.moe_inject_barrier_stall.argtypes = [_I]
_lib.moe_inject_barrier_stall.restype = ctypes.c_int
_lib.moe_status_string.argtypes = [_I]
_lib.moe_status_string.restype = ctypes.c_char_p
for _f in ("moe_workspace_bytes", "moe_route", "moe_group_by_expert", "moe_expert_forward",
           "moe_expert_forward_noalloc", "moe_layer_forward", "moe_stack_forward", "moe_stack_forward_norm",
           "moe_stack_forward_fp8", "moe_stack_forward_nvfp4", "moe_workspace_grouping"):
    getattr(_lib, _f).restype = ctypes.c_int

EXPORTED = ("moe_workspace_bytes", "moe_route", "moe_group_by_expert", "moe_expert_forward",
            "moe_expert_forward_noalloc", "moe_layer_forward", "moe_stack_forward", "moe_stack_forward_norm",
            "moe_stack_forward_fp8", "moe_stack_forward_nvfp4", "moe_workspace_grouping",
            "moe_launch_count", "moe_forward_path", "moe_set_trace_buffer",
            "moe_inject_barrier_stall", "moe_status_string")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_WORKSPACE = -4
MOE_DEV_TIMEOUT = 1
MOE_DEV_BAD_EXPERT_ID = 2
MOE_DEV_DUP_EXPERT = 4
MOE_DEV_NONFINITE = 8
MOE_DEV_BAD_ROUTE = 16
MOE_DEV_RANGE = 32
MOE_DT_F32 = 0
MOE_DT_BF16 = 1
MOE_F_NO_DEDUP = 1
MOE_F_UNFUSED = 2
MOE_F_FORCE_TC = 4
MOE_F_NO_TC = 8
MOE_F_NO_PREFETCH = 16
MOE_F_HOT_L2 = 32
MOE_F_SPLIT_TC = 64
TC_MIN_ROUTES = 8
MAX_E, MAX_TOPK, MAX_B, MAX_DIM, MAX_LAYERS = 256, 8, 1024, 16384, 64
NOALLOC_SCRATCH_BYTES = 16 << 20


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code}: {status_string(code)}")
        self.code = code


def status_string(code: int) -> str:
    return _lib.moe_status_string(int(code)).decode()


def _check(rc, fn):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _x_dtype(x):
    if x.dtype == torch.float32:
        return MOE_DT_F32
    if x.dtype == torch.bfloat16:
        return MOE_DT_BF16
    raise TypeError("x must be float32 or bfloat16")


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _opt(t, dtype, name, device):
    """Optional tensor argument: None, or a contiguous CUDA tensor of dtype on
    x's device (a host tensor's address must never reach a kernel)."""
    if t is None:
        return
    if dtype is not None:
        _need(t, dtype, name)
    elif not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, x on {device}")


def _need_x(x):
    _x_dtype(x)
    if x.dim() != 2:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H]")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")


def _shape(t, shape, name):
    """t (when given) must have exactly this shape; None entries match any size.
    Checked before any pointer reaches the library: a short buffer would be
    read or written out of bounds on the device."""
    if t is None:
        return
    if t.dim() != len(shape) or any(s is not None and d != s for d, s in zip(t.shape, shape)):
        want = "[" + ", ".join("*" if s is None else str(s) for s in shape) + "]"
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {want}")


def _at_least(t, n, name):
    if t.dim() != 1 or t.numel() < n:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected 1-D with at least {n} entries")


def _expert_shapes(x, gate_up, down):
    """-> (B, H, I, E) from x [B,H], gate_up [E,2I,H] and down [E,H,I]."""
    if x.dim() != 2:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H]")
    B, H = x.shape
    if gate_up.dim() != 3 or gate_up.shape[1] % 2 or gate_up.shape[2] != H:
        raise ValueError(f"gate_up has shape {tuple(gate_up.shape)}, expected [E, 2I, {H}]")
    E, I = gate_up.shape[0], gate_up.shape[1] // 2
    _shape(down, (E, H, I), "down")
    return B, H, I, E


def set_trace_buffer(buf):
    """Record phase timestamps of the persistent decode kernel into `buf`
    (a CUDA int64 tensor) on every following launch; None turns it off."""
    if buf is None:
        _check(_lib.moe_set_trace_buffer(None, 0), "moe_set_trace_buffer")
    else:
        _need(buf, torch.int64, "trace buffer")
        _check(_lib.moe_set_trace_buffer(_ptr(buf), buf.numel()), "moe_set_trace_buffer")


def inject_barrier_stall(extra_arrivals: int):
    """Fault injection: while > 0 the persistent kernels' device-wide
    barriers wait for arrivals that never come, time out (about a second),
    set MOE_DEV_TIMEOUT in the status word and return; 0 turns it off."""
    _check(_lib.moe_inject_barrier_stall(int(extra_arrivals)), "moe_inject_barrier_stall")


def workspace_bytes(B, H, I, E, top_k) -> int:
    n = _S(0)
    _check(_lib.moe_workspace_bytes(B, H, I, E, top_k, ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def new_workspace(B, H, I, E, top_k, device=None) -> torch.Tensor:
    n = workspace_bytes(B, H, I, E, top_k)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def workspace_grouping(workspace, B, H, I, E, top_k):
    """The grouped route list that the last forward call left in `workspace`
    -> (offsets [E+1], route_idx [B*k], unique [E], num_unique [1]) int32
    views into it (read them after that call has completed)."""
    _need(workspace, torch.uint8, "workspace")
    outs = [_P() for _ in range(4)]
    _check(_lib.moe_workspace_grouping(_ptr(workspace), workspace.numel(), B, H, I, E, top_k,
                                       *[ctypes.byref(o) for o in outs]), "moe_workspace_grouping")
    base = workspace.data_ptr()
    views = []
    for o, n in zip(outs, (E + 1, B * top_k, E, 1)):
        off = o.value - base
        views.append(workspace[off:off + 4 * n].view(torch.int32))
    return tuple(views)


PATH_DECODE, PATH_FUSED, PATH_PHASES = 2, 3, 4
PATH_NAMES = {0: "none", 2: "decode kernel", 3: "fused kernel", 4: "phase kernels"}


def forward_path(B, H, I, E, top_k, L=1, flags=0):
    """-> (path, grid): the kernels a layer (L=1) or stack forward runs for
    this shape on the current device (MOE_PATH_*), and its persistent grid."""
    path, grid = _I(0), _I(0)
    _check(_lib.moe_forward_path(B, H, I, E, top_k, L, flags, ctypes.byref(path), ctypes.byref(grid)),
           "moe_forward_path")
    return path.value, grid.value


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(_lib.moe_launch_count())


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def route(x, w_router, top_k, bias=None, stream=None, status=None):
    """-> (expert_ids [B,k] int32, route_w [B,k] fp32, logits [B,E] fp32)."""
    if x.dim() != 2 or w_router.dim() != 2:
        raise ValueError(f"x {tuple(x.shape)} and w_router {tuple(w_router.shape)} must be [B, H] and [E, H]")
    _shape(w_router, (None, x.shape[1]), "w_router")
    _shape(bias, (w_router.shape[0],), "bias")
    _shape(status, (1,), "status")
    _need_x(x)
    _need(w_router, torch.bfloat16, "w_router")
    _opt(bias, torch.float32, "bias", x.device)
    _opt(status, torch.int32, "status", x.device)
    B, H = x.shape
    E = w_router.shape[0]
    ids = torch.empty((B, top_k), dtype=torch.int32, device=x.device)
    w = torch.empty((B, top_k), dtype=torch.float32, device=x.device)
    logits = torch.empty((B, E), dtype=torch.float32, device=x.device)
    _check(_lib.moe_route(_ptr(x), _x_dtype(x), _ptr(w_router), _ptr(bias), B, H, E, top_k, _ptr(ids),
                          _ptr(w), _ptr(logits), None, 0, _ptr(status), _stream(stream)), "moe_route")
    return ids, w, logits


def group_by_expert(expert_ids, E, stream=None, status=None):
    """-> (offsets [E+1], route_idx [R], unique [E] (first num_unique valid), num_unique [1])."""
    if expert_ids.dim() != 2:
        raise ValueError(f"expert_ids has shape {tuple(expert_ids.shape)}, expected [B, top_k]")
    _shape(status, (1,), "status")
    _need(expert_ids, torch.int32, "expert_ids")
    B, k = expert_ids.shape
    dev = expert_ids.device
    _opt(status, torch.int32, "status", dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ridx = torch.empty(max(B * k, 1), dtype=torch.int32, device=dev)
    uniq = torch.empty(E, dtype=torch.int32, device=dev)
    nu = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_lib.moe_group_by_expert(_ptr(expert_ids), B, k, E, _ptr(offsets), _ptr(ridx), _ptr(uniq),
                                    _ptr(nu), _ptr(status), _stream(stream)), "moe_group_by_expert")
    return offsets, ridx[:B * k], uniq, nu


def _check_expert_args(x, gate_up, down, expert_ids, route_w, grouping, residual, out, status):
    B, H, I, E = _expert_shapes(x, gate_up, down)
    if expert_ids is None or route_w is None:
        raise ValueError("expert_ids and route_w are required")
    if expert_ids.dim() != 2 or expert_ids.shape[0] != B:
        raise ValueError(f"expert_ids has shape {tuple(expert_ids.shape)}, expected [{B}, top_k]")
    k = expert_ids.shape[1]
    _shape(route_w, (B, k), "route_w")
    if grouping is None or len(grouping) != 4 or any(t is None for t in grouping):
        raise ValueError("grouping must be (offsets, route_idx, unique_experts, num_unique)")
    R = B * k
    for t, n, need in zip(grouping, ("offsets", "route_idx", "unique_experts", "num_unique"),
                          (E + 1, R, min(R, E), 1)):
        _at_least(t, need, n)
    _shape(residual, (B, H), "residual")
    _shape(out, (B, H), "out")
    _shape(status, (1,), "status")
    _need_x(x)
    _need(gate_up, torch.bfloat16, "gate_up")
    _need(down, torch.bfloat16, "down")
    dev = x.device
    _opt(expert_ids, torch.int32, "expert_ids", dev)
    _opt(route_w, torch.float32, "route_w", dev)
    for t, n in zip(grouping, ("offsets", "route_idx", "unique_experts", "num_unique")):
        _opt(t, torch.int32, n, dev)
    _opt(residual, torch.float32, "residual", dev)
    _opt(out, torch.float32, "out", dev)
    _opt(status, torch.int32, "status", dev)


def expert_forward(x, gate_up, down, expert_ids, route_w, grouping, residual=None, flags=0,
                   out=None, workspace=None, status=None, stream=None):
    """y [B,H] fp32 = sum_j w * down_e(SiLU(gate_e x) * up_e x) (+ residual)."""
    _check_expert_args(x, gate_up, down, expert_ids, route_w, grouping, residual, out, status)
    _opt(workspace, torch.uint8, "workspace", x.device)
    B, H = x.shape
    E, twoI, _ = gate_up.shape
    I = twoI // 2
    k = expert_ids.shape[1]
    offsets, ridx, uniq, nu = grouping
    y = out if out is not None else torch.empty((B, H), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else new_workspace(B, H, I, E, k, x.device)
    _check(_lib.moe_expert_forward(_ptr(x), _x_dtype(x), _ptr(gate_up), _ptr(down), _ptr(expert_ids),
                                   _ptr(route_w), _ptr(offsets), _ptr(ridx), _ptr(uniq), _ptr(nu), B, H,
                                   I, E, k, _ptr(residual), _ptr(y), flags, _ptr(ws), ws.numel(),
                                   _ptr(status), _stream(stream)), "moe_expert_forward")
    return y


def expert_forward_noalloc(x, gate_up, down, expert_ids, route_w, grouping, residual=None, flags=0,
                           out=None, status=None, stream=None):
    """expert_forward with the library's fixed scratch array instead of a
    workspace: for callers that cannot allocate device memory.  `out` must
    be given by such callers (it is allocated here only for convenience)."""
    _check_expert_args(x, gate_up, down, expert_ids, route_w, grouping, residual, out, status)
    B, H = x.shape
    E, twoI, _ = gate_up.shape
    I = twoI // 2
    k = expert_ids.shape[1]
    offsets, ridx, uniq, nu = grouping
    y = out if out is not None else torch.empty((B, H), dtype=torch.float32, device=x.device)
    _check(_lib.moe_expert_forward_noalloc(_ptr(x), _x_dtype(x), _ptr(gate_up), _ptr(down),
                                           _ptr(expert_ids), _ptr(route_w), _ptr(offsets), _ptr(ridx),
                                           _ptr(uniq), _ptr(nu), B, H, I, E, k, _ptr(residual), _ptr(y),
                                           flags, _ptr(status), _stream(stream)),
           "moe_expert_forward_noalloc")
    return y


def layer_forward(x, w_router, gate_up, down, top_k, bias=None, residual=None, flags=0, out=None,
                  ids_out=None, w_out=None, workspace=None, status=None, stream=None):
    """Whole layer -> (y [B,H] fp32, expert_ids [B,k], route_w [B,k])."""
    B, H, I, E = _expert_shapes(x, gate_up, down)
    _shape(w_router, (E, H), "w_router")
    _shape(bias, (E,), "bias")
    for t, shp, n in ((residual, (B, H), "residual"), (out, (B, H), "out"), (ids_out, (B, top_k), "ids_out"),
                      (w_out, (B, top_k), "w_out"), (status, (1,), "status")):
        _shape(t, shp, n)
    _need_x(x)
    for t, n in ((w_router, "w_router"), (gate_up, "gate_up"), (down, "down")):
        _need(t, torch.bfloat16, n)
    for t, dt, n in ((bias, torch.float32, "bias"), (residual, torch.float32, "residual"),
                     (out, torch.float32, "out"), (ids_out, torch.int32, "ids_out"),
                     (w_out, torch.float32, "w_out"), (workspace, torch.uint8, "workspace"),
                     (status, torch.int32, "status")):
        _opt(t, dt, n, x.device)
    B, H = x.shape
    E, twoI, _ = gate_up.shape
    I = twoI // 2
    dev = x.device
    y = out if out is not None else torch.empty((B, H), dtype=torch.float32, device=dev)
    ids = ids_out if ids_out is not None else torch.empty((B, top_k), dtype=torch.int32, device=dev)
    w = w_out if w_out is not None else torch.empty((B, top_k), dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else new_workspace(B, H, I, E, top_k, dev)
    _check(_lib.moe_layer_forward(_ptr(x), _x_dtype(x), _ptr(w_router), _ptr(bias), _ptr(gate_up),
                                  _ptr(down), B, H, I, E, top_k, _ptr(residual), _ptr(y), _ptr(ids),
                                  _ptr(w), flags, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)),
           "moe_layer_forward")
    return y, ids, w


class StackWeightsFP8:
    """Host pointer tables for moe_stack_forward_fp8: each layer dict holds
    w_router [E,H] bf16, gate_up_q [E,2I,H] / down_q [E,H,I] uint8 E4M3 codes,
    gate_up_scale [E,ceil(2I/128),ceil(H/128)] / down_scale
    [E,ceil(H/128),ceil(I/128)] fp32, and optionally bias [E]."""

    def __init__(self, layers):
        self.layers = layers
        L = self.L = len(layers)
        g = layers[0]["gate_up_q"]
        if g.dim() != 3 or g.shape[1] % 2:
            raise ValueError(f"gate_up_q has shape {tuple(g.shape)}, expected [E, 2I, H]")
        self.E, twoI, self.H = g.shape
        self.I = twoI // 2
        nb = lambda n: (n + 127) // 128
        for l in layers:
            _shape(l["w_router"], (self.E, self.H), "w_router")
            _shape(l["gate_up_q"], (self.E, 2 * self.I, self.H), "gate_up_q")
            _shape(l["down_q"], (self.E, self.H, self.I), "down_q")
            _shape(l["gate_up_scale"], (self.E, nb(2 * self.I), nb(self.H)), "gate_up_scale")
            _shape(l["down_scale"], (self.E, nb(self.H), nb(self.I)), "down_scale")
            _shape(l.get("bias"), (self.E,), "bias")
            _need(l["w_router"], torch.bfloat16, "w_router")
            for n in ("gate_up_q", "down_q"):
                _need(l[n], torch.uint8, n)
            for n in ("gate_up_scale", "down_scale"):
                _need(l[n], torch.float32, n)
        P = lambda name: (ctypes.c_void_p * L)(*[l[name].data_ptr() for l in layers])
        self.wr, self.gq, self.gs, self.dq, self.ds = (P(n) for n in ("w_router", "gate_up_q", "gate_up_scale",
                                                                       "down_q", "down_scale"))
        has_bias = any(l.get("bias") is not None for l in layers)
        self.bias = ((ctypes.c_void_p * L)(*[(l["bias"].data_ptr() if l.get("bias") is not None else None)
                                             for l in layers]) if has_bias else None)


def stack_forward_fp8_(x, stack: StackWeightsFP8, top_k, flags=0, ids_out=None, workspace=None, status=None,
                       stream=None):
    """In place, block-scaled FP8 experts: x [B,H] fp32 <- x + layer_l(x)."""
    if x.dim() != 2 or stack is None or x.shape[1] != stack.H:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H] with H of the stack's weights")
    _shape(ids_out, (stack.L, x.shape[0], top_k), "ids_out")
    _shape(status, (1,), "status")
    _need(x, torch.float32, "x")
    for t, dt, n in ((ids_out, torch.int32, "ids_out"), (workspace, torch.uint8, "workspace"),
                     (status, torch.int32, "status")):
        _opt(t, dt, n, x.device)
    B, H = x.shape
    ws = workspace if workspace is not None else new_workspace(B, H, stack.I, stack.E, top_k, x.device)
    _check(_lib.moe_stack_forward_fp8(stack.L, ctypes.addressof(stack.wr),
                                      ctypes.addressof(stack.bias) if stack.bias is not None else None,
                                      ctypes.addressof(stack.gq), ctypes.addressof(stack.gs),
                                      ctypes.addressof(stack.dq), ctypes.addressof(stack.ds), B, H, stack.I, stack.E,
                                      top_k, _ptr(x), _ptr(ids_out), flags, _ptr(ws), ws.numel(), _ptr(status),
                                      _stream(stream)), "moe_stack_forward_fp8")
    return x


class StackWeightsNVFP4:
    """Host pointer tables for moe_stack_forward_nvfp4: each layer dict holds
    w_router [E,H] bf16, gate_up_q4 [E,2I,H/2] / down_q4 [E,H,I/2] uint8
    (E2M1 codes two a byte, element 2i in the low nibble), gate_up_bs
    [E,2I,H/16] / down_bs [E,H,I/16] uint8 E4M3 block scales, gate_up_gs /
    down_gs [E] fp32 matrix scales, and optionally bias [E]."""

    def __init__(self, layers):
        self.layers = layers
        L = self.L = len(layers)
        g = layers[0]["gate_up_q4"]
        if g.dim() != 3 or g.shape[1] % 2:
            raise ValueError(f"gate_up_q4 has shape {tuple(g.shape)}, expected [E, 2I, H/2]")
        self.E, twoI, h2 = g.shape
        self.I, self.H = twoI // 2, 2 * h2
        for l in layers:
            _shape(l["w_router"], (self.E, self.H), "w_router")
            _shape(l["gate_up_q4"], (self.E, 2 * self.I, self.H // 2), "gate_up_q4")
            _shape(l["down_q4"], (self.E, self.H, self.I // 2), "down_q4")
            _shape(l["gate_up_bs"], (self.E, 2 * self.I, self.H // 16), "gate_up_bs")
            _shape(l["down_bs"], (self.E, self.H, self.I // 16), "down_bs")
            _shape(l["gate_up_gs"], (self.E,), "gate_up_gs")
            _shape(l["down_gs"], (self.E,), "down_gs")
            _shape(l.get("bias"), (self.E,), "bias")
            _need(l["w_router"], torch.bfloat16, "w_router")
            for n in ("gate_up_q4", "down_q4", "gate_up_bs", "down_bs"):
                _need(l[n], torch.uint8, n)
            for n in ("gate_up_gs", "down_gs"):
                _need(l[n], torch.float32, n)
        P = lambda name: (ctypes.c_void_p * L)(*[l[name].data_ptr() for l in layers])
        self.wr, self.gq, self.gb, self.gg, self.dq, self.db, self.dg = (
            P(n) for n in ("w_router", "gate_up_q4", "gate_up_bs", "gate_up_gs", "down_q4", "down_bs", "down_gs"))
        has_bias = any(l.get("bias") is not None for l in layers)
        self.bias = ((ctypes.c_void_p * L)(*[(l["bias"].data_ptr() if l.get("bias") is not None else None)
                                             for l in layers]) if has_bias else None)


def stack_forward_nvfp4_(x, stack: StackWeightsNVFP4, top_k, flags=0, ids_out=None, workspace=None, status=None,
                         stream=None):
    """In place, NVFP4 experts: x [B,H] fp32 <- x + layer_l(x)."""
    if x.dim() != 2 or stack is None or x.shape[1] != stack.H:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H] with H of the stack's weights")
    _shape(ids_out, (stack.L, x.shape[0], top_k), "ids_out")
    _shape(status, (1,), "status")
    _need(x, torch.float32, "x")
    for t, dt, n in ((ids_out, torch.int32, "ids_out"), (workspace, torch.uint8, "workspace"),
                     (status, torch.int32, "status")):
        _opt(t, dt, n, x.device)
    B, H = x.shape
    ws = workspace if workspace is not None else new_workspace(B, H, stack.I, stack.E, top_k, x.device)
    _check(_lib.moe_stack_forward_nvfp4(stack.L, ctypes.addressof(stack.wr),
                                        ctypes.addressof(stack.bias) if stack.bias is not None else None,
                                        ctypes.addressof(stack.gq), ctypes.addressof(stack.gb),
                                        ctypes.addressof(stack.gg), ctypes.addressof(stack.dq),
                                        ctypes.addressof(stack.db), ctypes.addressof(stack.dg), B, H, stack.I,
                                        stack.E, top_k, _ptr(x), _ptr(ids_out), flags, _ptr(ws), ws.numel(),
                                        _ptr(status), _stream(stream)), "moe_stack_forward_nvfp4")
    return x


class StackWeights:
    """Host pointer tables for moe_stack_forward (built once, reused)."""

    def __init__(self, layers):
        self.layers = layers
        L = len(layers)
        self.L = L
        self.wr = (ctypes.c_void_p * L)(*[l["w_router"].data_ptr() for l in layers])
        self.gu = (ctypes.c_void_p * L)(*[l["gate_up"].data_ptr() for l in layers])
        self.dn = (ctypes.c_void_p * L)(*[l["down"].data_ptr() for l in layers])
        has_norm = all(l.get("norm") is not None for l in layers)
        self.norm = ((ctypes.c_void_p * L)(*[l["norm"].data_ptr() for l in layers]) if has_norm else None)
        has_bias = any(l.get("bias") is not None for l in layers)
        self.bias = ((ctypes.c_void_p * L)(*[(l["bias"].data_ptr() if l.get("bias") is not None else None)
                                             for l in layers]) if has_bias else None)
        g = layers[0]["gate_up"]
        if g.dim() != 3 or g.shape[1] % 2:
            raise ValueError(f"gate_up has shape {tuple(g.shape)}, expected [E, 2I, H]")
        self.E, twoI, self.H = g.shape
        self.I = twoI // 2
        for l in layers:
            _shape(l["w_router"], (self.E, self.H), "w_router")
            _shape(l["gate_up"], (self.E, 2 * self.I, self.H), "gate_up")
            _shape(l["down"], (self.E, self.H, self.I), "down")
            _shape(l.get("bias"), (self.E,), "bias")
            _shape(l.get("norm"), (self.H,), "norm")
            if l.get("norm") is not None:
                _need(l["norm"], torch.float32, "norm")
            for n in ("w_router", "gate_up", "down"):
                _need(l[n], torch.bfloat16, n)
            if l.get("bias") is not None:
                _need(l["bias"], torch.float32, "bias")


def stack_forward_(x, stack: StackWeights, top_k, flags=0, ids_out=None, workspace=None, status=None,
                   stream=None):
    """In place: x [B,H] fp32 <- x + layer_l(x) for every layer.  Returns x."""
    if x.dim() != 2 or stack is None or x.shape[1] != stack.H:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H] with H of the stack's weights")
    _shape(ids_out, (stack.L, x.shape[0], top_k), "ids_out")
    _shape(status, (1,), "status")
    _need(x, torch.float32, "x")
    for t, dt, n in ((ids_out, torch.int32, "ids_out"), (workspace, torch.uint8, "workspace"),
                     (status, torch.int32, "status")):
        _opt(t, dt, n, x.device)
    B, H = x.shape
    ws = workspace if workspace is not None else new_workspace(B, H, stack.I, stack.E, top_k, x.device)
    _check(_lib.moe_stack_forward(stack.L, ctypes.addressof(stack.wr),
                                  ctypes.addressof(stack.bias) if stack.bias is not None else None,
                                  ctypes.addressof(stack.gu), ctypes.addressof(stack.dn), B, H, stack.I,
                                  stack.E, top_k, _ptr(x), _ptr(ids_out), flags, _ptr(ws), ws.numel(),
                                  _ptr(status), _stream(stream)), "moe_stack_forward")
    return x


def stack_forward_norm_(x, stack: StackWeights, top_k, eps=1e-6, flags=0, ids_out=None, workspace=None,
                        status=None, stream=None):
    """Pre-norm stack, in place: x <- x + layer_l(RMSNorm_l(x)) for every
    layer (each layer dict carries its "norm" weights [H] fp32).  Returns x."""
    if x.dim() != 2 or stack is None or x.shape[1] != stack.H:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected [B, H] with H of the stack's weights")
    if stack.norm is None:
        raise ValueError("every layer needs its 'norm' weights for a pre-norm stack")
    _shape(ids_out, (stack.L, x.shape[0], top_k), "ids_out")
    _shape(status, (1,), "status")
    _need(x, torch.float32, "x")
    for t, dt, n in ((ids_out, torch.int32, "ids_out"), (workspace, torch.uint8, "workspace"),
                     (status, torch.int32, "status")):
        _opt(t, dt, n, x.device)
    B, H = x.shape
    ws = workspace if workspace is not None else new_workspace(B, H, stack.I, stack.E, top_k, x.device)
    _check(_lib.moe_stack_forward_norm(stack.L, ctypes.addressof(stack.wr),
                                       ctypes.addressof(stack.bias) if stack.bias is not None else None,
                                       ctypes.addressof(stack.gu), ctypes.addressof(stack.dn),
                                       ctypes.addressof(stack.norm), float(eps), B, H, stack.I, stack.E, top_k,
                                       _ptr(x), _ptr(ids_out), flags, _ptr(ws), ws.numel(), _ptr(status),
                                       _stream(stream)), "moe_stack_forward_norm")
    return x


def stack_forward(x, layers, top_k, flags=0, stream=None, status=None):
    """Out of place: returns (x_out, ids [L,B,k])."""
    st = layers if isinstance(layers, StackWeights) else StackWeights(layers)
    xo = x.to(torch.float32).clone()
    ids = torch.empty((st.L, x.shape[0], top_k), dtype=torch.int32, device=x.device)
    stack_forward_(xo, st, top_k, flags=flags, ids_out=ids, status=status, stream=stream)
    return xo, ids

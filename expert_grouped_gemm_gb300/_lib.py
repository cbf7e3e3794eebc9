"""ctypes binding of libmoe_gb300.so: the C ABI of include/moe.h, same names.

Argument marshalling only: each function checks that tensors are contiguous,
on the GPU and of the expected dtype, passes their pointers and the current
CUDA stream, and raises MoeError on a non-OK status. Every step of the layer
runs in the library's kernels. There is no fallback: if the library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_STATE = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_DEVICE_ARG = -7
MOE_BF16 = 0
MOE_F32 = 1
MOE_FROZEN = 1
MOE_RECOMPUTE = 2

EXPORTED = ["moe_workspace_size", "moe_fwd", "moe_select_retained", "moe_bwd", "moe_read_status",
            "moe_last_error", "moe_workspace_entry", "moe_kernel_launches", "moe_timing_enable",
            "moe_timing_read", "moe_route_noalloc", "moe_plan_quota", "moe_selftest_wait", "moe_fwd_decode",
            "moe_selftest_decode_wait"]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"moe status {code}: {msg}")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("F", ctypes.c_int64), ("E", ctypes.c_int64),
                ("k", ctypes.c_int64), ("F_shared", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library once (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    vp, i32p, f32p, i64 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64
    D = ctypes.POINTER(Dims)
    lib.moe_workspace_size.argtypes = [D, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_fwd.argtypes = [D, vp, ctypes.c_size_t, vp] + [vp] * 10 + [i32p, f32p, i32p, i32p, f32p]
    lib.moe_fwd_decode.argtypes = [D, vp, ctypes.c_size_t, vp] + [vp] * 10 + [i32p, f32p, f32p]
    lib.moe_selftest_decode_wait.argtypes = [D, vp, ctypes.c_size_t, vp] + [vp] * 10 + [ctypes.c_int, ctypes.c_int64]
    lib.moe_select_retained.argtypes = [D, vp, ctypes.c_size_t, vp, vp, i32p, i32p, i32p, f32p]
    lib.moe_bwd.argtypes = [D, vp, ctypes.c_size_t, vp, vp, vp, ctypes.c_int] + [vp] * 8
    lib.moe_read_status.argtypes = [vp, vp]
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_workspace_entry.argtypes = [D, ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_route_noalloc.argtypes = [D, vp, vp, vp, vp, i32p, f32p, i32p, i32p, i32p]
    lib.moe_route_noalloc.restype = ctypes.c_int
    lib.moe_plan_quota.argtypes = [D, vp, ctypes.c_size_t, vp, ctypes.c_int64, ctypes.c_int64, i32p, i32p]
    lib.moe_plan_quota.restype = ctypes.c_int
    lib.moe_selftest_wait.argtypes = [vp, ctypes.c_int, ctypes.c_int64, i32p]
    lib.moe_selftest_wait.restype = ctypes.c_int
    lib.moe_kernel_launches.argtypes = []
    lib.moe_kernel_launches.restype = ctypes.c_int64
    lib.moe_timing_enable.argtypes = [ctypes.c_int]
    lib.moe_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
    for name in ["moe_workspace_size", "moe_fwd", "moe_fwd_decode", "moe_selftest_decode_wait", "moe_select_retained",
                 "moe_bwd", "moe_read_status",
                 "moe_workspace_entry", "moe_timing_enable", "moe_timing_read"]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, load().moe_last_error().decode(errors="replace"))


def make_dims(T, H, F, E, k, F_shared=0, dtype="bf16", frozen=False, recompute=False) -> Dims:
    return Dims(T, H, F, E, k, F_shared, MOE_BF16 if dtype in ("bf16", MOE_BF16) else MOE_F32,
                (MOE_FROZEN if frozen else 0) | (MOE_RECOMPUTE if recompute else 0))


def _io_dtype(d: Dims):
    return torch.bfloat16 if d.dtype == MOE_BF16 else torch.float32


def _ptr(t, name, dtype=None, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def moe_workspace_size(dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(dims), ctypes.byref(n)))
    return n.value


def alloc_workspace(dims: Dims, device="cuda") -> torch.Tensor:
    """A uint8 device tensor of moe_workspace_size bytes (torch allocations are 256-byte aligned)."""
    return torch.empty(moe_workspace_size(dims), dtype=torch.uint8, device=device)


def moe_fwd(dims: Dims, ws: torch.Tensor, x, w_router, router_bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
            y, topk_idx=None, topk_w=None, expert_offsets=None, row_of_pair=None, logits=None, stream=None):
    io = _io_dtype(dims)
    rc = load().moe_fwd(
        ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream),
        _ptr(x, "x", io), _ptr(w_router, "w_router", io), _ptr(router_bias, "router_bias", torch.float32, False),
        _ptr(w_gate, "w_gate", io), _ptr(w_up, "w_up", io), _ptr(w_down, "w_down", io),
        _ptr(ws_gate, "ws_gate", io, False), _ptr(ws_up, "ws_up", io, False), _ptr(ws_down, "ws_down", io, False),
        _ptr(y, "y", io),
        _ptr(topk_idx, "topk_idx", torch.int32, False), _ptr(topk_w, "topk_w", torch.float32, False),
        _ptr(expert_offsets, "expert_offsets", torch.int32, False),
        _ptr(row_of_pair, "row_of_pair", torch.int32, False), _ptr(logits, "logits", torch.float32, False))
    _check(rc)


def moe_fwd_decode(dims: Dims, ws: torch.Tensor, x, w_router, router_bias, w_gate, w_up, w_down, ws_gate, ws_up,
                   ws_down, y, topk_idx=None, topk_w=None, logits=None, stream=None):
    """Fused inference forward for 1 <= T <= 16 tokens (bf16); keeps nothing for a backward."""
    io = _io_dtype(dims)
    rc = load().moe_fwd_decode(
        ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream),
        _ptr(x, "x", io), _ptr(w_router, "w_router", io), _ptr(router_bias, "router_bias", torch.float32, False),
        _ptr(w_gate, "w_gate", io), _ptr(w_up, "w_up", io), _ptr(w_down, "w_down", io),
        _ptr(ws_gate, "ws_gate", io, False), _ptr(ws_up, "ws_up", io, False), _ptr(ws_down, "ws_down", io, False),
        _ptr(y, "y", io), _ptr(topk_idx, "topk_idx", torch.int32, False), _ptr(topk_w, "topk_w", torch.float32, False),
        _ptr(logits, "logits", torch.float32, False))
    _check(rc)


def moe_selftest_decode_wait(dims: Dims, ws: torch.Tensor, x, w_router, router_bias, w_gate, w_up, w_down, ws_gate,
                             ws_up, ws_down, y, barrier: int, limit_us: int, stream=None):
    """moe_fwd_decode with grid barrier `barrier` (1..4) unreachable and every wait bounded
    by limit_us: the workspace status word becomes MOE_ERR_TIMEOUT."""
    io = _io_dtype(dims)
    rc = load().moe_selftest_decode_wait(
        ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream),
        _ptr(x, "x", io), _ptr(w_router, "w_router", io), _ptr(router_bias, "router_bias", torch.float32, False),
        _ptr(w_gate, "w_gate", io), _ptr(w_up, "w_up", io), _ptr(w_down, "w_down", io),
        _ptr(ws_gate, "ws_gate", io, False), _ptr(ws_up, "ws_up", io, False), _ptr(ws_down, "ws_down", io, False),
        _ptr(y, "y", io), int(barrier), int(limit_us))
    _check(rc)


def moe_select_retained(dims: Dims, ws: torch.Tensor, dy, quota=None, retained_offsets=None, retained_rows=None,
                        scores=None, stream=None):
    io = _io_dtype(dims)
    rc = load().moe_select_retained(
        ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream), _ptr(dy, "dy", io),
        _ptr(quota, "quota", torch.int32, False), _ptr(retained_offsets, "retained_offsets", torch.int32, False),
        _ptr(retained_rows, "retained_rows", torch.int32, False), _ptr(scores, "scores", torch.float32, False))
    _check(rc)


def moe_bwd(dims: Dims, ws: torch.Tensor, dy, x, use_retained, dx, dw_router=None, dw_gate=None, dw_up=None,
            dw_down=None, dws_gate=None, dws_up=None, dws_down=None, stream=None):
    io = _io_dtype(dims)
    rc = load().moe_bwd(
        ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream), _ptr(dy, "dy", io),
        _ptr(x, "x", io), 1 if use_retained else 0, _ptr(dx, "dx", io),
        _ptr(dw_router, "dw_router", io, False), _ptr(dw_gate, "dw_gate", io, False), _ptr(dw_up, "dw_up", io, False),
        _ptr(dw_down, "dw_down", io, False), _ptr(dws_gate, "dws_gate", io, False),
        _ptr(dws_up, "dws_up", io, False), _ptr(dws_down, "dws_down", io, False))
    _check(rc)


def moe_route_noalloc(dims: Dims, x, w_router, router_bias, topk_idx, topk_w, expert_offsets, row_of_pair,
                      device_status=None, stream=None):
    """Routing stage of moe_fwd with no allocation and no workspace (fixed device scratch inside the library)."""
    io = _io_dtype(dims)
    rc = load().moe_route_noalloc(
        ctypes.byref(dims), _stream(stream), _ptr(x, "x", io), _ptr(w_router, "w_router", io),
        _ptr(router_bias, "router_bias", torch.float32, False), _ptr(topk_idx, "topk_idx", torch.int32),
        _ptr(topk_w, "topk_w", torch.float32), _ptr(expert_offsets, "expert_offsets", torch.int32),
        _ptr(row_of_pair, "row_of_pair", torch.int32), _ptr(device_status, "device_status", torch.int32, False))
    _check(rc)


def moe_plan_quota(dims: Dims, ws: torch.Tensor, rho_num: int, rho_den: int, quota, budget=None, stream=None):
    """Device-side retention quotas from the last forward's per-expert counts."""
    rc = load().moe_plan_quota(ctypes.byref(dims), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream),
                               int(rho_num), int(rho_den), _ptr(budget, "budget", torch.int32, False),
                               _ptr(quota, "quota", torch.int32))
    _check(rc)


def moe_selftest_wait(arrive: bool, limit_us: int, device_status, stream=None):
    """One bounded barrier wait on the GPU; device_status receives MOE_OK or MOE_ERR_TIMEOUT."""
    rc = load().moe_selftest_wait(_stream(stream), 1 if arrive else 0, int(limit_us),
                                  _ptr(device_status, "device_status", torch.int32))
    _check(rc)


def moe_read_status(ws: torch.Tensor, stream=None) -> int:
    """Device status word (MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_ARG); syncs the stream and clears it."""
    return load().moe_read_status(_ptr(ws, "ws", torch.uint8), _stream(stream))


def moe_workspace_entries(dims: Dims) -> dict:
    """{name: (byte offset, byte size)} of the workspace layout for these dims (diagnostic)."""
    out, i = {}, 0
    lib = load()
    while True:
        name, off, size = ctypes.c_char_p(), ctypes.c_size_t(), ctypes.c_size_t()
        rc = lib.moe_workspace_entry(ctypes.byref(dims), i, ctypes.byref(name), ctypes.byref(off), ctypes.byref(size))
        if rc == MOE_ERR_INVALID_ARG and i > 0:
            return out
        _check(rc)
        out[name.value.decode()] = (off.value, size.value)
        i += 1


def ws_view(ws: torch.Tensor, dims: Dims, name: str, dtype, shape) -> torch.Tensor:
    """A typed view of one workspace buffer (diagnostic; copies nothing)."""
    off, size = moe_workspace_entries(dims)[name]
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    assert nbytes <= size, (name, nbytes, size)
    return ws[off:off + nbytes].view(dtype).view(*shape)


def moe_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().moe_kernel_launches())


def moe_timing_enable(on: bool) -> None:
    _check(load().moe_timing_enable(1 if on else 0))


def moe_timing_read():
    """(ms[2], launches[2]) for families (grouped GEMMs, bandwidth kernels); resets the counters."""
    ms = (ctypes.c_double * 2)()
    n = (ctypes.c_int64 * 2)()
    _check(load().moe_timing_read(ms, n))
    return [ms[0], ms[1]], [n[0], n[1]]


def moe_last_error() -> str:
    return load().moe_last_error().decode(errors="replace")

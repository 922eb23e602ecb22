"""Python binding of the GB300 local MoE forward chain.

Thin ctypes layer over the C ABI in ``include/moe.h`` (``libmoe_gb300.so``,
built in-tree by ``_build.build``). The functions carry the C names and only
marshal arguments: PyTorch supplies device memory and the current stream;
every step of the chain runs in the library's CUDA kernels. There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
from collections import namedtuple
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libmoe_gb300.so"

MOE_F32, MOE_F16, MOE_BF16 = 0, 1, 2
_DTYPE = {torch.float32: MOE_F32, torch.float16: MOE_F16, torch.bfloat16: MOE_BF16}

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_DTYPE", 4: "MOE_ERR_TOP_K",
    5: "MOE_ERR_ALIGNMENT", 6: "MOE_ERR_WORKSPACE", 7: "MOE_ERR_UNSUPPORTED", 8: "MOE_ERR_CUDA",
    9: "MOE_ERR_DEVICE_CHECK",
}


class GroupRoutingOptions(ctypes.Structure):
    """moe_group_routing_options (GroupRoutingOptions of the grouped sigmoid
    routing): top_k, groups, selected_groups, group_top_two, renormalize, scale."""
    _fields_ = [("top_k", ctypes.c_int32), ("groups", ctypes.c_int32), ("selected_groups", ctypes.c_int32),
                ("group_top_two", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("scale", ctypes.c_float)]

    def __init__(self, top_k, groups, selected_groups, group_top_two=False, renormalize=True, scale=1.0):
        super().__init__(int(top_k), int(groups), int(selected_groups), int(bool(group_top_two)),
                         int(bool(renormalize)), float(scale))


class RouterWeightOptions(ctypes.Structure):
    """moe_router_weight_options (RouterWeightOptions of first-order training):
    scoring ("softmax" or "sigmoid"), renormalize, scale."""
    _fields_ = [("scoring", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("scale", ctypes.c_float)]

    def __init__(self, scoring="softmax", renormalize=True, scale=1.0):
        code = {"softmax": 0, "sigmoid": 1}[scoring] if isinstance(scoring, str) else int(scoring)
        super().__init__(code, int(bool(renormalize)), float(scale))


_INDEX = {torch.int32: 1, torch.int64: 2}
if hasattr(torch, "uint32"):
    _INDEX[torch.uint32] = 0


# Every entry point declared in include/moe.h: name -> (restype, argtypes).
_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_OPT = ctypes.POINTER(GroupRoutingOptions)
_ROPT = ctypes.POINTER(RouterWeightOptions)
_FP = ctypes.c_void_p
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_version": (ctypes.c_int, []),
    "moe_route": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I32, _I32, _P, _P, _P, _P]),
    "moe_dispatch_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "moe_dispatch": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, ctypes.c_int, _I64, _P, _P, _P, _P, _P,
                                    _P, _SZ, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, ctypes.c_int, _I64, _P, _P, _P, _P, _P,
                                            _P]),
    "moe_route_dispatch_workspace_size": (_SZ, [_I64, _I64]),
    "moe_route_dispatch": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I32, _I32, _P, _P, _P, _P, ctypes.c_int,
                                          _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_rows": (ctypes.c_int, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _P]),
    "moe_experts_create": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                          ctypes.POINTER(ctypes.c_void_p)]),
    "moe_experts_destroy": (None, [_P]),
    "moe_experts_forward_dispatched_workspace_size": (_SZ, [_P, _I64]),
    "moe_experts_forward_dispatched": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _SZ, _P]),
    "moe_experts_forward_combine_workspace_size": (_SZ, [_P, _I64, _I32]),
    "moe_experts_forward_combine": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int, _I64, _I32, _P, _P, _SZ,
                                                   _P]),
    "moe_experts_gate_up": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _SZ, _P]),
    "moe_experts_down": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _SZ, _P]),
    "moe_experts_gate_up_gather": (ctypes.c_int, [_P, _P, _I64, _P, _I32, _P, _I64, _P, _P, _SZ, _P]),
    "moe_combine": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, ctypes.c_int, _I64, _I32, _I64, _P, _P]),
    "moe_forward_workspace_size": (_SZ, [_P, _I64, _I32]),
    "moe_forward": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_host_workspace_size": (ctypes.c_size_t, [_P, _I64, _I32, ctypes.c_int]),
    "moe_forward_host": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_sigmoid_grouped": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _P, _OPT, _P, _P, _P, _P]),
    "moe_route_sigmoid_grouped_dispatch": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _P, _OPT, _P, _P, _P, _P,
                                                          ctypes.c_int, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_sigmoid_grouped": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _P, _OPT, _P, _P, _P, _P,
                                                   _SZ, _P]),
    "moe_router_weights": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _P, ctypes.c_int, _I32, _ROPT, _P, _P]),
    "moe_router_backward": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _P, ctypes.c_int, _I32, _ROPT, _P, _P,
                                           _P]),
    "moe_experts_forward_training_workspace_size": (_SZ, [_P]),
    "moe_experts_forward_training": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine_backward": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P, _I64, _I32, _I64, _P,
                                            _P, _P]),
    "moe_experts_backward_workspace_size": (_SZ, [_P, _I64]),
    "moe_experts_backward": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_backward": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, _I32, _I64, _P, _P]),
    "moe_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _I32]),
    "moe_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, _P]),
}

_lib = None


class MoeError(RuntimeError):
    """A nonzero moe_status from the library (the MoeError of the pages)."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{self.name}: {message}")


def load_library(path: str | Path | None = None):
    """Load libmoe_gb300.so (once) and declare every entry point. Raises if it
    is missing: there is no CPU or eager fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no fallback path")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise MoeError(status, load_library().moe_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev_tensor(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE:
        raise MoeError(3, f"unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def _workspace(nbytes: int, device, ws: torch.Tensor | None) -> torch.Tensor:
    if ws is not None:
        return ws
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def moe_route(logits: torch.Tensor, top_k: int, renormalize: bool, *, indices=None, weights=None,
              weights_fp32=False, stream=None):
    """RoutingPlan: returns (indices [T,k] uint32 as int32 view, weights [T,k] in
    the logits dtype[, FP32 weights before the cast])."""
    lib = load_library()
    _dev_tensor(logits, "logits")
    T, E = logits.shape
    dev = logits.device
    if indices is None:
        indices = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(T, top_k, dtype=logits.dtype, device=dev)
    w32 = torch.empty(T, top_k, dtype=torch.float32, device=dev) if weights_fp32 is True else (
        weights_fp32 if isinstance(weights_fp32, torch.Tensor) else None)
    _check(lib.moe_route(_ptr(logits), _dt(logits), T, E, top_k, int(bool(renormalize)), _ptr(indices),
                         _ptr(weights), _ptr(w32), _stream(stream)))
    return (indices, weights, w32) if w32 is not None else (indices, weights)


DispatchedTokens = namedtuple("DispatchedTokens", "counts offsets row_src inv x_dispatched")


def moe_dispatch(indices: torch.Tensor, num_experts: int, x: torch.Tensor | None = None,
                 workspace=None, stream=None) -> DispatchedTokens:
    """RoutingPlan::dispatch: per-expert counts/offsets, row_src, inv and (if x
    is given) x_dispatched [T*k, H]."""
    lib = load_library()
    _dev_tensor(indices, "indices")
    T, k = indices.shape
    dev = indices.device
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    row_src = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    xd = None
    H, xdt = 0, MOE_F32
    if x is not None:
        _dev_tensor(x, "x")
        H, xdt = x.shape[1], _dt(x)
        xd = torch.empty(T * k, H, dtype=x.dtype, device=dev)
    need = lib.moe_dispatch_workspace_size(T, num_experts, k)
    ws = _workspace(need, dev, workspace)
    _check(lib.moe_dispatch(_ptr(indices), T, num_experts, k, _ptr(x), xdt, H, _ptr(counts),
                            _ptr(offsets), _ptr(row_src), _ptr(inv), _ptr(xd), _ptr(ws),
                            ws.numel(), _stream(stream)))
    return DispatchedTokens(counts, offsets, row_src, inv, xd)


def moe_route_dispatch(logits: torch.Tensor, top_k: int, renormalize: bool, x: torch.Tensor | None = None,
                       *, weights_fp32=False, workspace=None, stream=None):
    """moe_route then moe_dispatch as one launch (the same outputs, bit for
    bit): returns (indices, weights[, FP32 weights], DispatchedTokens)."""
    lib = load_library()
    _dev_tensor(logits, "logits")
    T, E = logits.shape
    dev = logits.device
    indices = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    weights = torch.empty(T, top_k, dtype=logits.dtype, device=dev)
    w32 = torch.empty(T, top_k, dtype=torch.float32, device=dev) if weights_fp32 else None
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_src = torch.empty(T * top_k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * top_k, dtype=torch.int32, device=dev)
    xd = None
    H, xdt = 0, MOE_F32
    if x is not None:
        _dev_tensor(x, "x")
        H, xdt = x.shape[1], _dt(x)
        xd = torch.empty(T * top_k, H, dtype=x.dtype, device=dev)
    need = lib.moe_route_dispatch_workspace_size(T, E)
    ws = _workspace(need, dev, workspace)
    _check(lib.moe_route_dispatch(_ptr(logits), _dt(logits), T, E, top_k, int(bool(renormalize)), _ptr(indices),
                                  _ptr(weights), _ptr(w32), _ptr(x), xdt, H, _ptr(counts), _ptr(offsets),
                                  _ptr(row_src), _ptr(inv), _ptr(xd), _ptr(ws), ws.numel(), _stream(stream)))
    disp = DispatchedTokens(counts, offsets, row_src, inv, xd)
    return (indices, weights, w32, disp) if w32 is not None else (indices, weights, disp)


def moe_permute_rows(src: torch.Tensor, index: torch.Tensor, *, scatter: bool = False, out=None,
                     out_rows: int | None = None, stream=None) -> torch.Tensor:
    """Row moves by an int64 index on the device: gather out[r] = src[index[r]]
    (out has index.numel() rows), or with scatter out[index[r]] = src[r] (out
    has out_rows rows, default src's)."""
    lib = load_library()
    _dev_tensor(src, "src")
    _dev_tensor(index, "index")
    if index.dtype != torch.int64:
        raise MoeError(3, "index must be int64")
    rows = index.numel()
    row_shape = tuple(src.shape[1:])
    if out is None:
        n_out = (out_rows if out_rows is not None else src.shape[0]) if scatter else rows
        out = torch.empty((n_out,) + row_shape, dtype=src.dtype, device=src.device)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 1
    _check(lib.moe_permute_rows(_ptr(src), src.shape[0], _ptr(out), out.shape[0], _ptr(index), rows, row_bytes,
                                int(bool(scatter)), _stream(stream)))
    return out


def moe_dispatch_noalloc(indices: torch.Tensor, num_experts: int, x: torch.Tensor | None = None,
                         stream=None) -> DispatchedTokens:
    """moe_dispatch with the library's fixed 1 MiB scratch instead of a
    workspace, for callers that cannot allocate device memory when they
    dispatch (the output tensors here are still allocated by torch)."""
    lib = load_library()
    _dev_tensor(indices, "indices")
    T, k = indices.shape
    dev = indices.device
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    row_src = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    xd = None
    H, xdt = 0, MOE_F32
    if x is not None:
        _dev_tensor(x, "x")
        H, xdt = x.shape[1], _dt(x)
        xd = torch.empty(T * k, H, dtype=x.dtype, device=dev)
    _check(lib.moe_dispatch_noalloc(_ptr(indices), T, num_experts, k, _ptr(x), xdt, H, _ptr(counts),
                                    _ptr(offsets), _ptr(row_src), _ptr(inv), _ptr(xd), _stream(stream)))
    return DispatchedTokens(counts, offsets, row_src, inv, xd)


class Experts:
    """SwiGluExperts: a handle over gate/up [E,I,H] and down [E,H,I] (kept alive here)."""

    def __init__(self, gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor):
        lib = load_library()
        for name, t in (("gate", gate), ("up", up), ("down", down)):
            _dev_tensor(t, name)
        E, I, H = gate.shape
        self.gate, self.up, self.down = gate, up, down
        self.E, self.H, self.I = E, H, I
        self.dtype = gate.dtype
        handle = ctypes.c_void_p()
        _check(lib.moe_experts_create(_ptr(gate), _ptr(up), _ptr(down), _dt(gate), E, H, I,
                                      ctypes.byref(handle)))
        self.handle = handle

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.moe_experts_destroy(self.handle)
            self.handle = None


def moe_experts_create(gate, up, down) -> Experts:
    return Experts(gate, up, down)


def moe_experts_forward_dispatched(experts: Experts, x_dispatched: torch.Tensor,
                                   offsets: torch.Tensor, out=None, workspace=None, stream=None):
    """SwiGluExperts::forward_dispatched: y_dispatched [rows, H] in the experts' dtype."""
    lib = load_library()
    _dev_tensor(x_dispatched, "x_dispatched")
    rows = x_dispatched.shape[0]
    y = out if out is not None else torch.empty(rows, experts.H, dtype=experts.dtype,
                                                device=x_dispatched.device)
    need = lib.moe_experts_forward_dispatched_workspace_size(experts.handle, rows)
    ws = _workspace(need, x_dispatched.device, workspace)
    _check(lib.moe_experts_forward_dispatched(experts.handle, _ptr(x_dispatched), _ptr(offsets), rows,
                                              _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))
    return y


def moe_experts_forward_combine(experts: Experts, x_dispatched: torch.Tensor, offsets: torch.Tensor,
                                inv: torch.Tensor, weights: torch.Tensor, out=None, workspace=None, stream=None):
    """forward_dispatched and combine in one launch: out [T, H] = sum over
    slots j (in order) of w[t, j] * y[inv[t * top_k + j]] (inv from
    moe_dispatch, weights [T, top_k] from moe_route)."""
    lib = load_library()
    _dev_tensor(x_dispatched, "x_dispatched")
    T, top_k = weights.shape
    y = out if out is not None else torch.empty(T, experts.H, dtype=experts.dtype, device=x_dispatched.device)
    need = lib.moe_experts_forward_combine_workspace_size(experts.handle, T, top_k)
    ws = _workspace(need, x_dispatched.device, workspace)
    _check(lib.moe_experts_forward_combine(experts.handle, _ptr(x_dispatched), _ptr(offsets), _ptr(inv),
                                           _ptr(weights), _dt(weights), T, top_k, _ptr(y), _ptr(ws), ws.numel(),
                                           _stream(stream)))
    return y


STAGE_WORKSPACE_BYTES = 256


def moe_experts_gate_up(experts: Experts, x_dispatched: torch.Tensor, offsets: torch.Tensor, out=None,
                        workspace=None, stream=None):
    """First GEMM stage: h [rows, I] = SiLU(x W_gate^T) * (x W_up^T) per expert."""
    lib = load_library()
    _dev_tensor(x_dispatched, "x_dispatched")
    rows = x_dispatched.shape[0]
    h = out if out is not None else torch.empty(rows, experts.I, dtype=experts.dtype,
                                                device=x_dispatched.device)
    ws = _workspace(STAGE_WORKSPACE_BYTES, x_dispatched.device, workspace)
    _check(lib.moe_experts_gate_up(experts.handle, _ptr(x_dispatched), _ptr(offsets), rows, _ptr(h),
                                   _ptr(ws), ws.numel(), _stream(stream)))
    return h


def moe_experts_gate_up_gather(experts: Experts, x: torch.Tensor, row_src: torch.Tensor, top_k: int,
                               offsets: torch.Tensor, rows: int | None = None, out=None, workspace=None,
                               stream=None):
    """Gate/up stage reading dispatched row r from x[row_src[r] // top_k]:
    h [rows, I] without an x_dispatched copy (rows defaults to row_src's length)."""
    lib = load_library()
    _dev_tensor(x, "x")
    _dev_tensor(row_src, "row_src")
    T = x.shape[0]
    rows = row_src.shape[0] if rows is None else rows
    h = out if out is not None else torch.empty(rows, experts.I, dtype=experts.dtype, device=x.device)
    ws = _workspace(STAGE_WORKSPACE_BYTES, x.device, workspace)
    _check(lib.moe_experts_gate_up_gather(experts.handle, _ptr(x), T, _ptr(row_src), top_k, _ptr(offsets), rows,
                                          _ptr(h), _ptr(ws), ws.numel(), _stream(stream)))
    return h


def moe_experts_down(experts: Experts, h: torch.Tensor, offsets: torch.Tensor, out=None, workspace=None,
                     stream=None):
    """Second GEMM stage: y [rows, H] = h W_down^T per expert."""
    lib = load_library()
    _dev_tensor(h, "h")
    rows = h.shape[0]
    y = out if out is not None else torch.empty(rows, experts.H, dtype=experts.dtype, device=h.device)
    ws = _workspace(STAGE_WORKSPACE_BYTES, h.device, workspace)
    _check(lib.moe_experts_down(experts.handle, _ptr(h), _ptr(offsets), rows, _ptr(y), _ptr(ws), ws.numel(),
                                _stream(stream)))
    return y


def moe_combine(y_dispatched: torch.Tensor, inv: torch.Tensor, weights: torch.Tensor, out=None,
                stream=None):
    """DispatchedTokens::combine: out [T, H] in y's dtype."""
    lib = load_library()
    _dev_tensor(y_dispatched, "y_dispatched")
    T, k = weights.shape
    H = y_dispatched.shape[1]
    o = out if out is not None else torch.empty(T, H, dtype=y_dispatched.dtype, device=y_dispatched.device)
    _check(lib.moe_combine(_ptr(y_dispatched), _dt(y_dispatched), _ptr(inv), _ptr(weights), _dt(weights),
                           T, k, H, _ptr(o), _stream(stream)))
    return o


def moe_forward_workspace_size(experts: Experts, T: int, top_k: int) -> int:
    return int(load_library().moe_forward_workspace_size(experts.handle, T, top_k))


def moe_forward(experts: Experts, x: torch.Tensor, logits: torch.Tensor, top_k: int,
                renormalize: bool, *, out=None, indices=None, weights=None, workspace=None,
                stream=None):
    """SwiGluExperts::forward: the whole chain, out [T, H]."""
    lib = load_library()
    _dev_tensor(x, "x")
    _dev_tensor(logits, "logits")
    T = x.shape[0]
    o = out if out is not None else torch.empty(T, experts.H, dtype=experts.dtype, device=x.device)
    ws = _workspace(lib.moe_forward_workspace_size(experts.handle, T, top_k), x.device, workspace)
    _check(lib.moe_forward(experts.handle, _ptr(x), _ptr(logits), _dt(logits), T, top_k,
                           int(bool(renormalize)), _ptr(o), _ptr(indices), _ptr(weights), _ptr(ws),
                           ws.numel(), _stream(stream)))
    return o


def moe_forward_host(experts: Experts, x: torch.Tensor, logits: torch.Tensor, top_k: int, renormalize: bool, *,
                     out=None, indices=None, weights=None, workspace=None, stream=None):
    """moe_forward on host (CPU) tensors: x [T, H] and logits [T, E] are
    copied to the device, the chain runs and out [T, H] is copied back, all
    enqueued on the stream. Pin the host tensors (`pin_memory()`) for
    asynchronous copies; the result is in `out` once the stream has passed
    the call's work."""
    lib = load_library()
    for t, name in ((x, "x"), (logits, "logits")):
        if t.is_cuda or not t.is_contiguous():
            raise MoeError(2, f"{name} must be a contiguous host tensor")
    T = x.shape[0]
    o = out if out is not None else torch.empty(T, experts.H, dtype=experts.dtype).pin_memory()
    if o.is_cuda or not o.is_contiguous():
        raise MoeError(2, "out must be a contiguous host tensor")
    dev = torch.device("cuda", torch.cuda.current_device())
    ws = _workspace(lib.moe_forward_host_workspace_size(experts.handle, T, top_k, _dt(logits)), dev, workspace)
    _check(lib.moe_forward_host(experts.handle, _ptr(x), _ptr(logits), _dt(logits), T, top_k, int(bool(renormalize)),
                                _ptr(o), _ptr(indices), _ptr(weights), _ptr(ws), ws.numel(), _stream(stream)))
    return o


def _options(options) -> GroupRoutingOptions:
    if isinstance(options, GroupRoutingOptions):
        return options
    return GroupRoutingOptions(options.top_k, options.groups, options.selected_groups, options.group_top_two,
                               options.renormalize, options.scale)


def moe_route_sigmoid_grouped(logits: torch.Tensor, bias: torch.Tensor | None, options, *, indices=None,
                              weights=None, weights_fp32=False, stream=None):
    """route_sigmoid_grouped: (indices [T,k], weights [T,k] in the logits
    dtype[, FP32 weights before the cast]). `options` is a
    GroupRoutingOptions (or any object with the same fields); `bias` is an
    FP32 [E] device tensor or None."""
    lib = load_library()
    _dev_tensor(logits, "logits")
    if bias is not None:
        _dev_tensor(bias, "bias")
        if bias.dtype != torch.float32:
            raise MoeError(3, "bias must be float32")
    o = _options(options)
    T, E = logits.shape
    k = o.top_k
    dev = logits.device
    if indices is None:
        indices = torch.empty(T, k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(T, k, dtype=logits.dtype, device=dev)
    w32 = torch.empty(T, k, dtype=torch.float32, device=dev) if weights_fp32 is True else (
        weights_fp32 if isinstance(weights_fp32, torch.Tensor) else None)
    _check(lib.moe_route_sigmoid_grouped(_ptr(logits), _dt(logits), T, E, _ptr(bias), ctypes.byref(o),
                                         _ptr(indices), _ptr(weights), _ptr(w32), _stream(stream)))
    return (indices, weights, w32) if w32 is not None else (indices, weights)


def moe_route_sigmoid_grouped_dispatch(logits: torch.Tensor, bias: torch.Tensor | None, options,
                                       x: torch.Tensor | None = None, *, weights_fp32=False, workspace=None,
                                       stream=None):
    """moe_route_sigmoid_grouped then moe_dispatch as one launch (the same
    outputs, bit for bit): returns (indices, weights[, FP32 weights],
    DispatchedTokens)."""
    lib = load_library()
    _dev_tensor(logits, "logits")
    if bias is not None:
        _dev_tensor(bias, "bias")
        if bias.dtype != torch.float32:
            raise MoeError(3, "bias must be float32")
    o = _options(options)
    T, E = logits.shape
    k = o.top_k
    dev = logits.device
    indices = torch.empty(T, k, dtype=torch.int32, device=dev)
    weights = torch.empty(T, k, dtype=logits.dtype, device=dev)
    w32 = torch.empty(T, k, dtype=torch.float32, device=dev) if weights_fp32 else None
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_src = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    xd = None
    H, xdt = 0, MOE_F32
    if x is not None:
        _dev_tensor(x, "x")
        H, xdt = x.shape[1], _dt(x)
        xd = torch.empty(T * k, H, dtype=x.dtype, device=dev)
    ws = _workspace(lib.moe_route_dispatch_workspace_size(T, E), dev, workspace)
    _check(lib.moe_route_sigmoid_grouped_dispatch(_ptr(logits), _dt(logits), T, E, _ptr(bias), ctypes.byref(o),
                                                  _ptr(indices), _ptr(weights), _ptr(w32), _ptr(x), xdt, H,
                                                  _ptr(counts), _ptr(offsets), _ptr(row_src), _ptr(inv), _ptr(xd),
                                                  _ptr(ws), ws.numel(), _stream(stream)))
    disp = DispatchedTokens(counts, offsets, row_src, inv, xd)
    return (indices, weights, w32, disp) if w32 is not None else (indices, weights, disp)


def moe_forward_sigmoid_grouped(experts: Experts, x: torch.Tensor, logits: torch.Tensor,
                                bias: torch.Tensor | None, options, *, out=None, indices=None, weights=None,
                                workspace=None, stream=None):
    """SwiGluExperts::forward_sigmoid_grouped: the whole chain with grouped
    sigmoid routing, out [T, H]."""
    lib = load_library()
    _dev_tensor(x, "x")
    _dev_tensor(logits, "logits")
    if bias is not None:
        _dev_tensor(bias, "bias")
    o = _options(options)
    T = x.shape[0]
    res = out if out is not None else torch.empty(T, experts.H, dtype=experts.dtype, device=x.device)
    ws = _workspace(lib.moe_forward_workspace_size(experts.handle, T, o.top_k), x.device, workspace)
    _check(lib.moe_forward_sigmoid_grouped(experts.handle, _ptr(x), _ptr(logits), _dt(logits), T, _ptr(bias),
                                           ctypes.byref(o), _ptr(res), _ptr(indices), _ptr(weights), _ptr(ws),
                                           ws.numel(), _stream(stream)))
    return res


def _router_opts(options) -> RouterWeightOptions:
    if isinstance(options, RouterWeightOptions):
        return options
    return RouterWeightOptions(options.scoring, options.renormalize, options.scale)


def _index_type(indices: torch.Tensor) -> int:
    if indices.dtype not in _INDEX:
        raise MoeError(3, f"indices must be uint32, int32 or int64, not {indices.dtype}")
    return _INDEX[indices.dtype]


def moe_router_weights(logits: torch.Tensor, indices: torch.Tensor, options, *, out=None, stream=None):
    """selected_router_weights: FP32 [T, top_k] weights of a fixed selection."""
    lib = load_library()
    _dev_tensor(logits, "logits")
    _dev_tensor(indices, "indices")
    T, E = logits.shape
    k = indices.shape[1]
    o = _router_opts(options)
    w = out if out is not None else torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib.moe_router_weights(_ptr(logits), _dt(logits), T, E, _ptr(indices), _index_type(indices), k,
                                  ctypes.byref(o), _ptr(w), _stream(stream)))
    return w


def moe_router_backward(logits: torch.Tensor, indices: torch.Tensor, grad_weights: torch.Tensor, options, *,
                        out=None, stream=None):
    """selected_router_backward: dlogits [T, E] in the logits dtype."""
    lib = load_library()
    for name, t in (("logits", logits), ("indices", indices), ("grad_weights", grad_weights)):
        _dev_tensor(t, name)
    if grad_weights.dtype != torch.float32:
        raise MoeError(3, "grad_weights must be float32")
    T, E = logits.shape
    k = indices.shape[1]
    o = _router_opts(options)
    d = out if out is not None else torch.empty_like(logits)
    _check(lib.moe_router_backward(_ptr(logits), _dt(logits), T, E, _ptr(indices), _index_type(indices), k,
                                   ctypes.byref(o), _ptr(grad_weights), _ptr(d), _stream(stream)))
    return d


TrainingCache = namedtuple("TrainingCache", "x_dispatched offsets h g u")


def moe_experts_forward_training(experts: Experts, x_dispatched: torch.Tensor, offsets: torch.Tensor,
                                 workspace=None, stream=None):
    """forward_dispatched_training: (y_dispatched [rows, H], cache) where the
    cache holds what moe_experts_backward needs (h, g, u)."""
    lib = load_library()
    _dev_tensor(x_dispatched, "x_dispatched")
    rows = x_dispatched.shape[0]
    dev = x_dispatched.device
    y = torch.empty(rows, experts.H, dtype=experts.dtype, device=dev)
    h, g, u = (torch.empty(rows, experts.I, dtype=experts.dtype, device=dev) for _ in range(3))
    ws = _workspace(lib.moe_experts_forward_training_workspace_size(experts.handle), dev, workspace)
    _check(lib.moe_experts_forward_training(experts.handle, _ptr(x_dispatched), _ptr(offsets), rows, _ptr(h),
                                            _ptr(y), _ptr(g), _ptr(u), _ptr(ws), ws.numel(), _stream(stream)))
    return y, TrainingCache(x_dispatched, offsets, h, g, u)


ExpertGrads = namedtuple("ExpertGrads", "dx_dispatched dgate dup ddown")


def moe_experts_backward(experts: Experts, cache: TrainingCache, dexpert: torch.Tensor, workspace=None,
                         stream=None) -> ExpertGrads:
    """cache.backward(dexpert): dx_dispatched [rows, H] and FP32 dgate, dup
    [E, I, H] and ddown [E, H, I]."""
    lib = load_library()
    _dev_tensor(dexpert, "dexpert")
    rows = cache.x_dispatched.shape[0]
    dev = dexpert.device
    dx = torch.empty(rows, experts.H, dtype=experts.dtype, device=dev)
    dgate = torch.empty(experts.E, experts.I, experts.H, dtype=torch.float32, device=dev)
    dup = torch.empty_like(dgate)
    ddown = torch.empty(experts.E, experts.H, experts.I, dtype=torch.float32, device=dev)
    ws = _workspace(lib.moe_experts_backward_workspace_size(experts.handle, rows), dev, workspace)
    _check(lib.moe_experts_backward(experts.handle, _ptr(cache.x_dispatched), _ptr(cache.offsets), rows,
                                    _ptr(cache.h), _ptr(cache.g), _ptr(cache.u), _ptr(dexpert), _ptr(dx),
                                    _ptr(dgate), _ptr(dup), _ptr(ddown), _ptr(ws), ws.numel(), _stream(stream)))
    return ExpertGrads(dx, dgate, dup, ddown)


def moe_combine_backward(y_dispatched: torch.Tensor, inv: torch.Tensor, row_src: torch.Tensor,
                         weights: torch.Tensor, grad_out: torch.Tensor, stream=None):
    """combine_backward: (dexpert [rows, H] in y's dtype, dweights [T, top_k]
    FP32). inv and row_src are moe_dispatch's two maps."""
    lib = load_library()
    for name, t in (("y_dispatched", y_dispatched), ("inv", inv), ("row_src", row_src), ("weights", weights),
                    ("grad_out", grad_out)):
        _dev_tensor(t, name)
    T, k = weights.shape
    if inv.numel() != T * k or row_src.numel() != T * k:
        raise MoeError(2, "inv and row_src must hold T * top_k entries")
    H = y_dispatched.shape[1]
    dexp = torch.empty_like(y_dispatched)
    dw = torch.empty(T, k, dtype=torch.float32, device=y_dispatched.device)
    _check(lib.moe_combine_backward(_ptr(y_dispatched), _dt(y_dispatched), _ptr(inv), _ptr(row_src), _ptr(weights),
                                    _dt(weights), _ptr(grad_out), T, k, H, _ptr(dexp), _ptr(dw), _stream(stream)))
    return dexp, dw


def moe_dispatch_backward(dinput: torch.Tensor, inv: torch.Tensor, T: int, top_k: int, stream=None):
    """dispatch_backward: dx [T, H], each token's dispatched rows added in slot order."""
    lib = load_library()
    _dev_tensor(dinput, "dinput")
    _dev_tensor(inv, "inv")
    H = dinput.shape[1]
    dx = torch.empty(T, H, dtype=dinput.dtype, device=dinput.device)
    _check(lib.moe_dispatch_backward(_ptr(dinput), _dt(dinput), _ptr(inv), T, top_k, H, _ptr(dx), _stream(stream)))
    return dx


def moe_device_status(clear: bool = True) -> int:
    code = ctypes.c_uint32(0)
    _check(load_library().moe_device_status(ctypes.byref(code), int(clear)))
    return code.value


def moe_selftest_bounded_wait(limit_us: int, stream=None):
    _check(load_library().moe_selftest_bounded_wait(limit_us, _stream(stream)))

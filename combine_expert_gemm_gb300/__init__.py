"""Python binding of the routed-expert layer C ABI (``include/moe.h`` and
``include/moe_mxfp8.h``).

Argument marshalling only: every step of the layer runs in the sm_103a
kernels of ``_build/libmoe_gb300.so``.  Tensors are torch CUDA tensors (the
caller owns them); bf16 buffers are ``torch.bfloat16``, fp32 ``torch.float32``,
indices ``torch.int32``, all contiguous.  Calls enqueue on the current torch
CUDA stream (or ``stream=``) and never synchronise.

Importing this package fails loudly if the library has not been built
(``python combine_expert_gemm_gb300/build.py``); there is no fallback.
"""
import ctypes
import os

import torch

from .build import LIB

__all__ = ["Shape", "MoEError", "lib", "route", "dispatch", "expert_ffn", "combine",
           "combine_backward", "dispatch_backward", "read_device_error", "dispatch_checked",
           "combine_checked", "combine_backward_checked", "dispatch_backward_checked",
           "route_workspace_bytes", "route_logits", "expert_ffn_workspace_bytes", "capacity", "LayerBuffers",
           "layer_forward", "expert_ffn_backward", "expert_ffn_backward_workspace_bytes",
           "BackwardBuffers", "layer_backward", "MxWeights", "MxLayerBuffers", "mx_act_scale_bytes",
           "mx_quantize_weights", "dispatch_mxfp8", "expert_ffn_mxfp8", "combine_mxfp8",
           "layer_forward_mxfp8", "StreamedLayer"]

if not os.path.exists(LIB):
    raise ImportError(f"{LIB} is missing: build it with `python combine_expert_gemm_gb300/build.py` "
                      "(or __graft_entry__.build()); there is no CPU fallback")

_lib = ctypes.CDLL(LIB)


def lib():
    return _lib


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("N", ctypes.c_int32),
                ("K", ctypes.c_int32), ("h", ctypes.c_int32), ("cap", ctypes.c_int32)]

    def __repr__(self):
        return f"Shape(T={self.T}, d={self.d}, N={self.N}, K={self.K}, h={self.h}, cap={self.cap})"

    @property
    def R(self):
        """Rows of every capacity buffer, min(N*cap, T*K) (moe_buffer_rows)."""
        return min(self.N * self.cap, self.T * self.K)


_P = ctypes.c_void_p
_SP = ctypes.POINTER(Shape)
_SZ = ctypes.c_size_t
_SIG = {
    "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "moe_route_workspace_bytes": ([_SP], _SZ),
    "moe_route_logits_offset": ([_SP], _SZ),
    "moe_expert_ffn_workspace_bytes": ([_SP], _SZ),
    "moe_route": ([_SP] + [_P] * 9 + [_P, _SZ, _P], ctypes.c_int),
    "moe_dispatch": ([_SP, _P, _P, _P, _P], ctypes.c_int),
    "moe_expert_ffn": ([_SP] + [_P] * 10 + [_P, _SZ, _P], ctypes.c_int),
    "moe_combine": ([_SP, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_combine_backward": ([_SP, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_dispatch_backward": ([_SP, _P, _P, _P, _P], ctypes.c_int),
    "moe_dispatch_checked": ([_SP, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_combine_checked": ([_SP, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_combine_backward_checked": ([_SP] + [_P] * 6 + [_P, _P], ctypes.c_int),
    "moe_dispatch_backward_checked": ([_SP, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_read_device_error": ([_P, ctypes.POINTER(ctypes.c_int32), _P], ctypes.c_int),
    "moe_expert_ffn_backward_workspace_bytes": ([_SP], _SZ),
    "moe_expert_ffn_backward": ([_SP] + [_P] * 14 + [_P, _SZ, _P], ctypes.c_int),
    "moe_selftest_wait_timeout": ([_P, ctypes.c_uint64, _P], ctypes.c_int),
    "moe_router_backward_workspace_bytes": ([_SP], _SZ),
    "moe_router_backward": ([_SP] + [_P] * 9 + [_P, _SZ, _P], ctypes.c_int),
    "moe_buffer_rows": ([_SP], ctypes.c_int64),
    "moe_dispatch_router_backward": ([_SP] + [_P] * 8 + [_P], ctypes.c_int),
    "moe_router_weight_backward": ([_SP] + [_P] * 5 + [_P, _SZ, _P], ctypes.c_int),
    "moe_expert_ffn_gather_workspace_bytes": ([_SP], _SZ),
    "moe_expert_ffn_gather": ([_SP] + [_P] * 11 + [_P, _SZ, _P], ctypes.c_int),
    "moe_mx_act_scale_bytes": ([_SP, ctypes.c_int32], _SZ),
    "moe_mx_quantize_weights": ([ctypes.c_int32] * 3 + [_P] * 3 + [_P], ctypes.c_int),
    "moe_dispatch_mxfp8": ([_SP] + [_P] * 7 + [_P], ctypes.c_int),
    "moe_expert_ffn_mxfp8": ([_SP] + [_P] * 14 + [_P, _SZ, _P], ctypes.c_int),
    "moe_combine_mxfp8": ([_SP] + [_P] * 5 + [_P], ctypes.c_int),
}
for _name, (_args, _res) in _SIG.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIG)


class MoEError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = _lib.moe_status_string(code).decode()
        super().__init__(f"{where}: {msg} (status {code})")


def _check(code, where):
    if code != 0:
        raise MoEError(code, where)


def capacity(T, K, N, cf_num, cf_den=1):
    """ceil(cf * T * K / N) with cf = cf_num / cf_den, in integers."""
    return (cf_num * T * K + cf_den * N - 1) // (cf_den * N)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    # the kernels run on the current device: memory of another GPU would be
    # read through a pointer that is not this device's
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_bf16, _f32, _i32 = torch.bfloat16, torch.float32, torch.int32


def route_workspace_bytes(shape):
    return int(_lib.moe_route_workspace_bytes(ctypes.byref(shape)))


def route_logits(shape, ws):
    """The router logits [T, N] fp32 that the last moe_route call on the
    workspace ``ws`` (a uint8 CUDA tensor) left there: a view, not a copy."""
    off = int(_lib.moe_route_logits_offset(ctypes.byref(shape)))
    if off == 0:
        raise MoEError(1, "moe_route_logits_offset")
    n = shape.T * shape.N * 4
    return ws[off:off + n].view(torch.float32).view(shape.T, shape.N)


def expert_ffn_workspace_bytes(shape):
    return int(_lib.moe_expert_ffn_workspace_bytes(ctypes.byref(shape)))


def route(shape, x, w_router, bias, topk_idx, topk_gate, route_row, expert_count, expert_offset,
          expert_demand, ws, stream=None):
    _check(_lib.moe_route(ctypes.byref(shape), _ptr(x, _bf16, "x"), _ptr(w_router, _f32, "w_router"),
                          _ptr(bias, _f32, "bias"), _ptr(topk_idx, _i32, "topk_idx"),
                          _ptr(topk_gate, _f32, "topk_gate"), _ptr(route_row, _i32, "route_row"),
                          _ptr(expert_count, _i32, "expert_count"),
                          _ptr(expert_offset, _i32, "expert_offset"),
                          _ptr(expert_demand, _i32, "expert_demand"), _ptr(ws, None, "ws"),
                          ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def dispatch(shape, x, route_row, x_disp, stream=None):
    _check(_lib.moe_dispatch(ctypes.byref(shape), _ptr(x, _bf16, "x"),
                             _ptr(route_row, _i32, "route_row"), _ptr(x_disp, _bf16, "x_disp"),
                             _stream(stream)), "moe_dispatch")


def expert_ffn(shape, x_disp, expert_count, expert_offset, w_gate, w_up, w_down, h_act, g_save,
               u_save, y_disp, ws, stream=None):
    _check(_lib.moe_expert_ffn(ctypes.byref(shape), _ptr(x_disp, _bf16, "x_disp"),
                               _ptr(expert_count, _i32, "expert_count"),
                               _ptr(expert_offset, _i32, "expert_offset"),
                               _ptr(w_gate, _bf16, "w_gate"), _ptr(w_up, _bf16, "w_up"),
                               _ptr(w_down, _bf16, "w_down"), _ptr(h_act, _bf16, "h_act"),
                               _ptr(g_save, _bf16, "g_save"), _ptr(u_save, _bf16, "u_save"),
                               _ptr(y_disp, _bf16, "y_disp"), _ptr(ws, None, "ws"),
                               ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn")


def expert_ffn_gather_workspace_bytes(shape):
    return int(_lib.moe_expert_ffn_gather_workspace_bytes(ctypes.byref(shape)))


def expert_ffn_gather(shape, x, route_row, expert_count, expert_offset, w_gate, w_up, w_down, h_act,
                      g_save, u_save, y_disp, ws, stream=None):
    """Dispatch fused into the grouped SwiGLU experts: x rows are fetched by route (include/moe.h)."""
    _check(_lib.moe_expert_ffn_gather(ctypes.byref(shape), _ptr(x, _bf16, "x"),
                                      _ptr(route_row, _i32, "route_row"),
                                      _ptr(expert_count, _i32, "expert_count"),
                                      _ptr(expert_offset, _i32, "expert_offset"),
                                      _ptr(w_gate, _bf16, "w_gate"), _ptr(w_up, _bf16, "w_up"),
                                      _ptr(w_down, _bf16, "w_down"), _ptr(h_act, _bf16, "h_act"),
                                      _ptr(g_save, _bf16, "g_save"), _ptr(u_save, _bf16, "u_save"),
                                      _ptr(y_disp, _bf16, "y_disp"), _ptr(ws, None, "ws"),
                                      ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_gather")


def combine(shape, y_disp, route_row, topk_gate, y, stream=None):
    _check(_lib.moe_combine(ctypes.byref(shape), _ptr(y_disp, _bf16, "y_disp"),
                            _ptr(route_row, _i32, "route_row"), _ptr(topk_gate, _f32, "topk_gate"),
                            _ptr(y, _bf16, "y"), _stream(stream)), "moe_combine")


def combine_backward(shape, dy, y_disp, route_row, topk_gate, dy_disp, dgate, stream=None):
    _check(_lib.moe_combine_backward(ctypes.byref(shape), _ptr(dy, _bf16, "dy"),
                                     _ptr(y_disp, _bf16, "y_disp"),
                                     _ptr(route_row, _i32, "route_row"),
                                     _ptr(topk_gate, _f32, "topk_gate"),
                                     _ptr(dy_disp, _bf16, "dy_disp"), _ptr(dgate, _f32, "dgate"),
                                     _stream(stream)), "moe_combine_backward")


def dispatch_backward(shape, dx_disp, route_row, dx, stream=None):
    _check(_lib.moe_dispatch_backward(ctypes.byref(shape), _ptr(dx_disp, _bf16, "dx_disp"),
                                      _ptr(route_row, _i32, "route_row"), _ptr(dx, _f32, "dx"),
                                      _stream(stream)), "moe_dispatch_backward")


def _status_ptr(status_ws):
    if status_ws.dtype != torch.uint8 or status_ws.numel() < 256:
        raise ValueError("status_ws: a uint8 CUDA tensor of at least 256 bytes")
    return _ptr(status_ws, None, "status_ws")


def dispatch_checked(shape, x, route_row, x_disp, status_ws, stream=None):
    """moe_dispatch with every route row compared with the buffer rows on the
    device; a row past them is skipped and recorded in status_ws (include/moe.h)."""
    _check(_lib.moe_dispatch_checked(ctypes.byref(shape), _ptr(x, _bf16, "x"),
                                     _ptr(route_row, _i32, "route_row"),
                                     _ptr(x_disp, _bf16, "x_disp"), _status_ptr(status_ws),
                                     _stream(stream)), "moe_dispatch_checked")


def combine_checked(shape, y_disp, route_row, topk_gate, y, status_ws, stream=None):
    _check(_lib.moe_combine_checked(ctypes.byref(shape), _ptr(y_disp, _bf16, "y_disp"),
                                    _ptr(route_row, _i32, "route_row"),
                                    _ptr(topk_gate, _f32, "topk_gate"), _ptr(y, _bf16, "y"),
                                    _status_ptr(status_ws), _stream(stream)), "moe_combine_checked")


def combine_backward_checked(shape, dy, y_disp, route_row, topk_gate, dy_disp, dgate, status_ws,
                             stream=None):
    _check(_lib.moe_combine_backward_checked(
        ctypes.byref(shape), _ptr(dy, _bf16, "dy"), _ptr(y_disp, _bf16, "y_disp"),
        _ptr(route_row, _i32, "route_row"), _ptr(topk_gate, _f32, "topk_gate"),
        _ptr(dy_disp, _bf16, "dy_disp"), _ptr(dgate, _f32, "dgate"), _status_ptr(status_ws),
        _stream(stream)), "moe_combine_backward_checked")


def dispatch_backward_checked(shape, dx_disp, route_row, dx, status_ws, stream=None):
    _check(_lib.moe_dispatch_backward_checked(
        ctypes.byref(shape), _ptr(dx_disp, _bf16, "dx_disp"), _ptr(route_row, _i32, "route_row"),
        _ptr(dx, _f32, "dx"), _status_ptr(status_ws), _stream(stream)),
        "moe_dispatch_backward_checked")


def expert_ffn_backward_workspace_bytes(shape):
    return int(_lib.moe_expert_ffn_backward_workspace_bytes(ctypes.byref(shape)))


def expert_ffn_backward(shape, x_disp, expert_count, expert_offset, w_gate, w_up, w_down, g_save,
                        u_save, h_act, dy_disp, dx_disp, dw_gate, dw_up, dw_down, ws, stream=None):
    _check(_lib.moe_expert_ffn_backward(
        ctypes.byref(shape), _ptr(x_disp, _bf16, "x_disp"), _ptr(expert_count, _i32, "expert_count"),
        _ptr(expert_offset, _i32, "expert_offset"), _ptr(w_gate, _bf16, "w_gate"),
        _ptr(w_up, _bf16, "w_up"), _ptr(w_down, _bf16, "w_down"), _ptr(g_save, _bf16, "g_save"),
        _ptr(u_save, _bf16, "u_save"), _ptr(h_act, _bf16, "h_act"), _ptr(dy_disp, _bf16, "dy_disp"),
        _ptr(dx_disp, _bf16, "dx_disp"), _ptr(dw_gate, _f32, "dw_gate"), _ptr(dw_up, _f32, "dw_up"),
        _ptr(dw_down, _f32, "dw_down"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
        _stream(stream)), "moe_expert_ffn_backward")


def buffer_rows(shape):
    """Rows of every capacity buffer, min(N*cap, T*K); -1 for an invalid shape."""
    return int(_lib.moe_buffer_rows(ctypes.byref(shape)))


def router_backward_workspace_bytes(shape):
    return int(_lib.moe_router_backward_workspace_bytes(ctypes.byref(shape)))


def router_backward(shape, x, w_router, topk_idx, topk_gate, dgate, dlogit, dx, dw_router, dbias,
                    ws, stream=None):
    """dlogit, dx += router term, dw_router, dbias (may be None); see include/moe.h."""
    _check(_lib.moe_router_backward(
        ctypes.byref(shape), _ptr(x, _bf16, "x"), _ptr(w_router, _f32, "w_router"),
        _ptr(topk_idx, _i32, "topk_idx"), _ptr(topk_gate, _f32, "topk_gate"),
        _ptr(dgate, _f32, "dgate"), _ptr(dlogit, _f32, "dlogit"), _ptr(dx, _f32, "dx"),
        _ptr(dw_router, _f32, "dw_router"), _ptr(dbias, _f32, "dbias"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_router_backward")


def dispatch_router_backward(shape, dx_disp, route_row, w_router, topk_idx, topk_gate, dgate,
                             dlogit, dx, stream=None):
    """dx = dispatch backward + router term, and dlogit, in one pass (include/moe.h)."""
    _check(_lib.moe_dispatch_router_backward(
        ctypes.byref(shape), _ptr(dx_disp, _bf16, "dx_disp"), _ptr(route_row, _i32, "route_row"),
        _ptr(w_router, _f32, "w_router"), _ptr(topk_idx, _i32, "topk_idx"),
        _ptr(topk_gate, _f32, "topk_gate"), _ptr(dgate, _f32, "dgate"), _ptr(dlogit, _f32, "dlogit"),
        _ptr(dx, _f32, "dx"), _stream(stream)), "moe_dispatch_router_backward")


def router_weight_backward(shape, x, topk_idx, dlogit, dw_router, dbias, ws, stream=None):
    """dw_router and dbias (may be None) from dlogit (include/moe.h)."""
    _check(_lib.moe_router_weight_backward(
        ctypes.byref(shape), _ptr(x, _bf16, "x"), _ptr(topk_idx, _i32, "topk_idx"),
        _ptr(dlogit, _f32, "dlogit"), _ptr(dw_router, _f32, "dw_router"),
        _ptr(dbias, _f32, "dbias"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
        _stream(stream)), "moe_router_weight_backward")


def selftest_wait_timeout(ws, limit_ns, stream=None):
    """Runs the bounded-wait failure path once (see include/moe.h)."""
    _check(_lib.moe_selftest_wait_timeout(_ptr(ws, None, "ws"), int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def read_device_error(ws, stream=None):
    code = ctypes.c_int32(0)
    _check(_lib.moe_read_device_error(_ptr(ws, None, "ws"), ctypes.byref(code), _stream(stream)),
           "moe_read_device_error")
    return code.value


class LayerBuffers:
    """Device buffers of one layer instance, allocated once before the loop
    (capacity-shaped, so no allocation depends on the routing)."""

    def __init__(self, shape, device="cuda", save_for_backward=False):
        T, d, N, K, h, R = shape.T, shape.d, shape.N, shape.K, shape.h, shape.R
        e = dict(device=device)
        self.shape = shape
        self.topk_idx = torch.empty((T, K), dtype=_i32, **e)
        self.topk_gate = torch.empty((T, K), dtype=_f32, **e)
        self.route_row = torch.empty((T, K), dtype=_i32, **e)
        self.expert_count = torch.empty(N, dtype=_i32, **e)
        self.expert_offset = torch.empty(N + 1, dtype=_i32, **e)
        self.expert_demand = torch.empty(N, dtype=_i32, **e)
        self.route_ws = torch.zeros(max(route_workspace_bytes(shape), 256), dtype=torch.uint8, **e)
        self.ffn_ws = torch.zeros(max(expert_ffn_workspace_bytes(shape), 256), dtype=torch.uint8, **e)
        self.gather_ws = torch.zeros(max(expert_ffn_gather_workspace_bytes(shape), 256),
                                     dtype=torch.uint8, **e)
        self.x_disp = torch.empty((R, d), dtype=_bf16, **e)
        self.h_act = torch.empty((R, h), dtype=_bf16, **e)
        self.g_save = torch.empty((R, h), dtype=_bf16, **e) if save_for_backward else None
        self.u_save = torch.empty((R, h), dtype=_bf16, **e) if save_for_backward else None
        self.y_disp = torch.empty((R, d), dtype=_bf16, **e)
        self.y = torch.empty((T, d), dtype=_bf16, **e)

    def route_logits(self):
        """The router logits [T, N] fp32 of the last forward (a view into route_ws)."""
        return route_logits(self.shape, self.route_ws)


def layer_forward(buf, x, w_router, bias, w_gate, w_up, w_down, stream=None, fused_dispatch=False):
    """Route -> dispatch -> grouped SwiGLU experts -> combine into buf.y (4 C-ABI calls).
    fused_dispatch: the experts fetch x rows by route instead (3 calls, no x_disp;
    for a forward without backward)."""
    s = buf.shape
    route(s, x, w_router, bias, buf.topk_idx, buf.topk_gate, buf.route_row, buf.expert_count,
          buf.expert_offset, buf.expert_demand, buf.route_ws, stream)
    if fused_dispatch:
        expert_ffn_gather(s, x, buf.route_row, buf.expert_count, buf.expert_offset, w_gate, w_up,
                          w_down, buf.h_act, buf.g_save, buf.u_save, buf.y_disp, buf.gather_ws,
                          stream)
    else:
        dispatch(s, x, buf.route_row, buf.x_disp, stream)
        expert_ffn(s, buf.x_disp, buf.expert_count, buf.expert_offset, w_gate, w_up, w_down,
                   buf.h_act, buf.g_save, buf.u_save, buf.y_disp, buf.ffn_ws, stream)
    combine(s, buf.y_disp, buf.route_row, buf.topk_gate, buf.y, stream)
    return buf.y


class BackwardBuffers:
    """Device buffers of one layer's backward (allocated once before the loop)."""

    def __init__(self, shape, device="cuda"):
        T, d, N, K, h, R = shape.T, shape.d, shape.N, shape.K, shape.h, shape.R
        e = dict(device=device)
        self.shape = shape
        self.dy_disp = torch.empty((R, d), dtype=_bf16, **e)
        self.dgate = torch.empty((T, K), dtype=_f32, **e)
        self.dx_disp = torch.empty((R, d), dtype=_bf16, **e)
        self.dx = torch.empty((T, d), dtype=_f32, **e)
        self.dw_gate = torch.empty((N, h, d), dtype=_f32, **e)
        self.dw_up = torch.empty((N, h, d), dtype=_f32, **e)
        self.dw_down = torch.empty((N, d, h), dtype=_f32, **e)
        self.ws = torch.zeros(max(expert_ffn_backward_workspace_bytes(shape), 256),
                              dtype=torch.uint8, **e)
        self.dlogit = torch.empty((T, K), dtype=_f32, **e)
        self.dw_router = torch.empty((N, d), dtype=_f32, **e)
        self.dbias = torch.empty(N, dtype=_f32, **e)
        self.router_ws = torch.zeros(max(router_backward_workspace_bytes(shape), 256),
                                     dtype=torch.uint8, **e)


def layer_backward(fwd, bwd, dy, w_gate, w_up, w_down, stream=None, x=None, w_router=None,
                   with_bias=False):
    """Combine backward -> grouped expert backward -> dispatch backward (3 C-ABI
    calls) for the forward whose buffers are `fwd` (saved with
    save_for_backward=True).  Fills bwd.dgate, bwd.dx, bwd.dw_*.  Given the
    forward's x and w_router, the dispatch backward also adds the router term
    to bwd.dx (one pass) and a fourth call fills bwd.dlogit, bwd.dw_router (and
    bwd.dbias)."""
    s = fwd.shape
    combine_backward(s, dy, fwd.y_disp, fwd.route_row, fwd.topk_gate, bwd.dy_disp, bwd.dgate,
                     stream)
    expert_ffn_backward(s, fwd.x_disp, fwd.expert_count, fwd.expert_offset, w_gate, w_up, w_down,
                        fwd.g_save, fwd.u_save, fwd.h_act, bwd.dy_disp, bwd.dx_disp, bwd.dw_gate,
                        bwd.dw_up, bwd.dw_down, bwd.ws, stream)
    if w_router is None:
        dispatch_backward(s, bwd.dx_disp, fwd.route_row, bwd.dx, stream)
    else:
        dispatch_router_backward(s, bwd.dx_disp, fwd.route_row, w_router, fwd.topk_idx,
                                 fwd.topk_gate, bwd.dgate, bwd.dlogit, bwd.dx, stream)
        router_weight_backward(s, x, fwd.topk_idx, bwd.dlogit, bwd.dw_router,
                               bwd.dbias if with_bias else None, bwd.router_ws, stream)
    return bwd


# ------------------------------------------------------------------- MXFP8 --
# include/moe_mxfp8.h: E4M3 codes and E8M0 scale bytes are torch.uint8.

_u8 = torch.uint8


def mx_act_scale_bytes(shape, k):
    """Bytes of the scale chunks of a capacity buffer with k columns (k = d or h)."""
    return int(_lib.moe_mx_act_scale_bytes(ctypes.byref(shape), int(k)))


def mx_quantize_weights(w, q, sf, stream=None):
    """w [E, rows, k] bf16 -> q [E, rows, k] E4M3 codes and sf (E*rows*k/8 bytes: the
    scale chunks, each stored four times; see include/moe_mxfp8.h)."""
    E, rows, k = w.shape
    _check(_lib.moe_mx_quantize_weights(E, rows, k, _ptr(w, _bf16, "w"), _ptr(q, _u8, "q"),
                                        _ptr(sf, _u8, "sf"), _stream(stream)),
           "moe_mx_quantize_weights")


def dispatch_mxfp8(shape, x, route_row, topk_idx, expert_count, expert_offset, x_q, x_sf,
                   stream=None):
    _check(_lib.moe_dispatch_mxfp8(ctypes.byref(shape), _ptr(x, _bf16, "x"),
                                   _ptr(route_row, _i32, "route_row"),
                                   _ptr(topk_idx, _i32, "topk_idx"),
                                   _ptr(expert_count, _i32, "expert_count"),
                                   _ptr(expert_offset, _i32, "expert_offset"),
                                   _ptr(x_q, _u8, "x_q"), _ptr(x_sf, _u8, "x_sf"),
                                   _stream(stream)), "moe_dispatch_mxfp8")


def expert_ffn_mxfp8(shape, x_q, x_sf, expert_count, expert_offset, w, h_q, h_sf, y_q, y_scale, ws,
                     stream=None):
    """w: an MxWeights.  Fills h_q/h_sf (SwiGLU output) and y_q/y_scale."""
    _check(_lib.moe_expert_ffn_mxfp8(
        ctypes.byref(shape), _ptr(x_q, _u8, "x_q"), _ptr(x_sf, _u8, "x_sf"),
        _ptr(expert_count, _i32, "expert_count"), _ptr(expert_offset, _i32, "expert_offset"),
        _ptr(w.gate_q, _u8, "w_gate_q"), _ptr(w.gate_sf, _u8, "w_gate_sf"),
        _ptr(w.up_q, _u8, "w_up_q"), _ptr(w.up_sf, _u8, "w_up_sf"),
        _ptr(w.down_q, _u8, "w_down_q"), _ptr(w.down_sf, _u8, "w_down_sf"),
        _ptr(h_q, _u8, "h_q"), _ptr(h_sf, _u8, "h_sf"), _ptr(y_q, _u8, "y_q"),
        _ptr(y_scale, _u8, "y_scale"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
        _stream(stream)), "moe_expert_ffn_mxfp8")


def combine_mxfp8(shape, y_q, y_scale, route_row, topk_gate, y, stream=None):
    _check(_lib.moe_combine_mxfp8(ctypes.byref(shape), _ptr(y_q, _u8, "y_q"),
                                  _ptr(y_scale, _u8, "y_scale"), _ptr(route_row, _i32, "route_row"),
                                  _ptr(topk_gate, _f32, "topk_gate"), _ptr(y, _bf16, "y"),
                                  _stream(stream)), "moe_combine_mxfp8")


class MxWeights:
    """Expert weights in MXFP8, quantized once from bf16 [N,h,d], [N,h,d],
    [N,d,h] along each product's reduction dimension."""

    def __init__(self, w_gate, w_up, w_down, stream=None):
        def q(w):
            E, rows, k = w.shape
            codes = torch.empty((E, rows, k), dtype=_u8, device=w.device)
            sf = torch.empty(E * rows * k // 8, dtype=_u8, device=w.device)
            mx_quantize_weights(w, codes, sf, stream)
            return codes, sf
        self.gate_q, self.gate_sf = q(w_gate)
        self.up_q, self.up_sf = q(w_up)
        self.down_q, self.down_sf = q(w_down)


class MxLayerBuffers(LayerBuffers):
    """LayerBuffers plus the quantized payloads of the MXFP8 path."""

    def __init__(self, shape, device="cuda"):
        super().__init__(shape, device)
        d, h, R = shape.d, shape.h, shape.R
        e = dict(device=device, dtype=_u8)
        self.x_q = torch.empty((R, d), **e)
        self.x_sf = torch.zeros(max(mx_act_scale_bytes(shape, d), 16), **e)
        self.h_q = torch.empty((R, h), **e)
        self.h_sf = torch.zeros(max(mx_act_scale_bytes(shape, h), 16), **e)
        self.y_q = torch.empty((R, d), **e)
        self.y_scale = torch.empty((R, d // 32), **e)


def layer_forward_mxfp8(buf, x, w_router, bias, w, stream=None):
    """Route -> quantizing dispatch -> MXFP8 experts -> dequantizing combine
    into buf.y (4 C-ABI calls); w is an MxWeights."""
    s = buf.shape
    route(s, x, w_router, bias, buf.topk_idx, buf.topk_gate, buf.route_row, buf.expert_count,
          buf.expert_offset, buf.expert_demand, buf.route_ws, stream)
    dispatch_mxfp8(s, x, buf.route_row, buf.topk_idx, buf.expert_count, buf.expert_offset,
                   buf.x_q, buf.x_sf, stream)
    expert_ffn_mxfp8(s, buf.x_q, buf.x_sf, buf.expert_count, buf.expert_offset, w, buf.h_q,
                     buf.h_sf, buf.y_q, buf.y_scale, buf.ffn_ws, stream)
    combine_mxfp8(s, buf.y_q, buf.y_scale, buf.route_row, buf.topk_gate, buf.y, stream)
    return buf.y


class StreamedLayer:
    """A stream of token batches through the layer, with the host copies of
    one batch overlapping the device work of its neighbours.

    Each submit(x_host, y_host[, dy_host, dx_host]) enqueues, for one batch:
    the input copy from pinned host memory to the device (stream h2d), the
    layer forward -- and the backward when dy_host is given -- (stream
    compute), and the output copy back to pinned host memory (stream d2h).
    Two sets of device buffers alternate, so batch i's copies run while
    batch i - 1 or i + 1 computes; events order each set's reuse (an input
    copy waits for the layer that last read that set's input, a layer waits
    for the output copy that last read that set's outputs).  submit returns
    at once; synchronize() waits for every submitted batch.  The host
    buffers of a batch must stay untouched until then.
    """

    def __init__(self, shape, w_router, bias, w_gate, w_up, w_down, device="cuda",
                 backward=False):
        self.shape = shape
        self.w = (w_router, bias, w_gate, w_up, w_down)
        self.backward = backward
        dev = torch.device(device)
        T, d = shape.T, shape.d
        self.fwd = [LayerBuffers(shape, dev, save_for_backward=backward) for _ in range(2)]
        self.bwd = [BackwardBuffers(shape, dev) for _ in range(2)] if backward else None
        self.x = [torch.empty((T, d), dtype=_bf16, device=dev) for _ in range(2)]
        self.dy = [torch.empty((T, d), dtype=_bf16, device=dev) for _ in range(2)] if backward else None
        self.h2d, self.compute, self.d2h = (torch.cuda.Stream(dev) for _ in range(3))
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.copied, self.layer_done, self.read_done = ev(), ev(), ev()
        self.i = 0

    def submit(self, x_host, y_host, dy_host=None, dx_host=None):
        j = self.i % 2
        wr, bias, wg, wu, wd = self.w
        self.h2d.wait_event(self.layer_done[j])
        with torch.cuda.stream(self.h2d):
            self.x[j].copy_(x_host, non_blocking=True)
            if self.backward:
                self.dy[j].copy_(dy_host, non_blocking=True)
            self.copied[j].record(self.h2d)
        self.compute.wait_event(self.copied[j])
        self.compute.wait_event(self.read_done[j])
        fb = self.fwd[j]
        layer_forward(fb, self.x[j], wr, bias, wg, wu, wd, stream=self.compute)
        if self.backward:
            layer_backward(fb, self.bwd[j], self.dy[j], wg, wu, wd, stream=self.compute,
                           x=self.x[j], w_router=wr, with_bias=bias is not None)
        self.layer_done[j].record(self.compute)
        self.d2h.wait_event(self.layer_done[j])
        with torch.cuda.stream(self.d2h):
            y_host.copy_(fb.y, non_blocking=True)
            if self.backward:
                dx_host.copy_(self.bwd[j].dx, non_blocking=True)
            self.read_done[j].record(self.d2h)
        self.i += 1

    def synchronize(self):
        self.d2h.synchronize()

    def status(self):
        """Device status words of every workspace (0 = no device error)."""
        codes = [read_device_error(b.route_ws) for b in self.fwd]
        codes += [read_device_error(b.ffn_ws) for b in self.fwd]
        if self.backward:
            codes += [read_device_error(b.ws) for b in self.bwd]
        return max(codes)

"""ORACLE -- test infrastructure, not part of the product.

numpy front end of the plain C oracle (``moe_oracle.c``): a slow,
single-threaded CPU statement of the routed-expert layer.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It never imports the CUDA package and the CUDA package never imports it.

bf16 tensors are numpy ``uint16`` bit patterns; fp32 tensors ``float32``;
indices ``int32``.  Every function follows the passage cited in the C source.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_oracle())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def _declare(L):
    sig = {
        "oracle_bf16_from_f64": [_I64, _P, _P],
        "oracle_bf16_from_f32": [_I64, _P, _P],
        "oracle_router_logits": [_I, _I, _I, _P, _P, _P, _P],
        "oracle_topk_gates": [_I, _I, _I, _P, _P, _P],
        "oracle_route_slots": [_I, _I, _I, _I, _P, _P, _P, _P, _P],
        "oracle_dispatch": [_I, _I, _I, _P, _P, _P],
        "oracle_ffn_fwd_f64": [_I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P],
        "oracle_ffn_bwd_f64": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P],
        "oracle_expert_ffn_rows": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
        "oracle_expert_ffn": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
        "oracle_combine": [_I, _I, _I, _P, _P, _P, _P],
        "oracle_combine_bwd": [_I, _I, _I, _P, _P, _P, _P, _P, _P],
        "oracle_dispatch_bwd": [_I, _I, _I, _P, _P, _P],
        "oracle_expert_ffn_bwd": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _P],
        "oracle_router_bwd": [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P],
        "oracle_mx_quantize_f64": [_I64, _I, _P, _P, _P],
        "oracle_mx_quantize_bf16": [_I64, _I, _P, _P, _P],
        "oracle_mx_dequantize": [_I64, _I, _P, _P, _P],
        "oracle_expert_ffn_mx": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _P, _P],
        "oracle_combine_mx": [_I, _I, _I, _P, _P, _P, _P, _P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = None


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------- helpers --

def bf16_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_from_f64(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_from_f64(v.size, _p(v), _p(out))
    return out


def bf16_from_f32(v):
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_from_f32(v.size, _p(v), _p(out))
    return out


# ------------------------------------------------------------------ routing --

def router_logits(x, w_r, bias=None):
    x = _c(x, np.uint16)
    w_r = _c(w_r, np.float32)
    T, d = x.shape
    N = w_r.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, N), dtype=np.float32)
    lib().oracle_router_logits(T, d, N, _p(x), _p(w_r), _p(b), _p(out))
    return out


def topk_gates(logits, K):
    logits = _c(logits, np.float32)
    T, N = logits.shape
    idx = np.empty((T, K), dtype=np.int32)
    gate = np.empty((T, K), dtype=np.float32)
    lib().oracle_topk_gates(T, N, K, _p(logits), _p(idx), _p(gate))
    return idx, gate


def route_slots(idx, N, cap):
    idx = _c(idx, np.int32)
    T, K = idx.shape
    row = np.empty((T, K), dtype=np.int32)
    count = np.empty(N, dtype=np.int32)
    offset = np.empty(N + 1, dtype=np.int32)
    demand = np.empty(N, dtype=np.int32)
    lib().oracle_route_slots(T, N, K, cap, _p(idx), _p(row), _p(count), _p(offset), _p(demand))
    return row, count, offset, demand


def route(x, w_r, bias, K, cap):
    """R0-R3: logits, top-K indices and gates, route map, counts, offsets, demand."""
    logits = router_logits(x, w_r, bias)
    idx, gate = topk_gates(logits, K)
    row, count, offset, demand = route_slots(idx, w_r.shape[0], cap)
    return dict(logits=logits, topk_idx=idx, topk_gate=gate, route_row=row,
                expert_count=count, expert_offset=offset, expert_demand=demand)


# ----------------------------------------------------------------- movement --

def dispatch(x, route_row, R, fill=0):
    x = _c(x, np.uint16)
    route_row = _c(route_row, np.int32)
    T, d = x.shape
    K = route_row.shape[1]
    out = np.full((R, d), fill, dtype=np.uint16)
    lib().oracle_dispatch(T, d, K, _p(x), _p(route_row), _p(out))
    return out


def combine(y_disp, route_row, gate):
    y_disp = _c(y_disp, np.uint16)
    route_row = _c(route_row, np.int32)
    gate = _c(gate, np.float32)
    T, K = route_row.shape
    d = y_disp.shape[1]
    out = np.empty((T, d), dtype=np.uint16)
    lib().oracle_combine(T, d, K, _p(y_disp), _p(route_row), _p(gate), _p(out))
    return out


def combine_bwd(dy, y_disp, route_row, gate, fill=0):
    dy = _c(dy, np.uint16)
    y_disp = _c(y_disp, np.uint16)
    route_row = _c(route_row, np.int32)
    gate = _c(gate, np.float32)
    T, d = dy.shape
    K = route_row.shape[1]
    dy_disp = np.full(y_disp.shape, fill, dtype=np.uint16)
    dgate = np.empty((T, K), dtype=np.float32)
    lib().oracle_combine_bwd(T, d, K, _p(dy), _p(y_disp), _p(route_row), _p(gate),
                             _p(dy_disp), _p(dgate))
    return dy_disp, dgate


def dispatch_bwd(dx_disp, route_row, T):
    dx_disp = _c(dx_disp, np.uint16)
    route_row = _c(route_row, np.int32)
    K = route_row.shape[1]
    d = dx_disp.shape[1]
    out = np.empty((T, d), dtype=np.float32)
    lib().oracle_dispatch_bwd(T, d, K, _p(dx_disp), _p(route_row), _p(out))
    return out


# ------------------------------------------------------------------ experts --

def ffn_fwd_f64(x, wg, wu, wd, round_a=False):
    """fp64 SwiGLU expert on rows x: returns g, u, a, y (all float64)."""
    x = _c(x, np.float64); wg = _c(wg, np.float64); wu = _c(wu, np.float64); wd = _c(wd, np.float64)
    n, d = x.shape
    h = wg.shape[0]
    g = np.empty((n, h)); u = np.empty((n, h)); a = np.empty((n, h)); y = np.empty((n, d))
    lib().oracle_ffn_fwd_f64(n, d, h, _p(x), _p(wg), _p(wu), _p(wd), int(round_a),
                             _p(g), _p(u), _p(a), _p(y))
    return g, u, a, y


def ffn_bwd_f64(x, g, u, a, dy, wg, wu, wd, round_dgu=False):
    """fp64 backward of the SwiGLU expert: returns dx, dwg, dwu, dwd.

    round_dgu rounds dG and dU to bf16 before the products that consume them,
    as the grouped backward does (they are bf16 payloads there)."""
    arrs = [_c(v, np.float64) for v in (x, g, u, a, dy, wg, wu, wd)]
    x, g, u, a, dy, wg, wu, wd = arrs
    n, d = x.shape
    h = wg.shape[0]
    dx = np.empty((n, d)); dwg = np.zeros((h, d)); dwu = np.zeros((h, d)); dwd = np.zeros((d, h))
    lib().oracle_ffn_bwd_f64(n, d, h, _p(x), _p(g), _p(u), _p(a), _p(dy), _p(wg), _p(wu), _p(wd),
                             int(round_dgu), _p(dx), _p(dwg), _p(dwu), _p(dwd))
    return dx, dwg, dwu, dwd


def expert_ffn(x_disp, count, offset, wg, wu, wd, save=False, fill=0):
    """Grouped SwiGLU experts over the valid rows; returns h_act, g_save, u_save, y_disp.

    Tail rows (past offset[N]) keep ``fill``.  g_save / u_save are None unless save.
    """
    x_disp = _c(x_disp, np.uint16); count = _c(count, np.int32); offset = _c(offset, np.int32)
    wg = _c(wg, np.uint16); wu = _c(wu, np.uint16); wd = _c(wd, np.uint16)
    R, d = x_disp.shape
    N, h, _ = wg.shape
    h_act = np.full((R, h), fill, dtype=np.uint16)
    y = np.full((R, d), fill, dtype=np.uint16)
    gs = np.full((R, h), fill, dtype=np.uint16) if save else None
    us = np.full((R, h), fill, dtype=np.uint16) if save else None
    lib().oracle_expert_ffn(N, d, h, _p(count), _p(offset), _p(x_disp), _p(wg), _p(wu), _p(wd),
                            _p(h_act), _p(gs), _p(us), _p(y))
    return h_act, gs, us, y


def expert_ffn_rows(rows, experts, x_disp, wg, wu, wd, save=False):
    """The same, for a list of (row, expert) pairs; outputs are compact [len(rows), .]."""
    rows = _c(rows, np.int32); experts = _c(experts, np.int32)
    x_disp = _c(x_disp, np.uint16)
    wg = _c(wg, np.uint16); wu = _c(wu, np.uint16); wd = _c(wd, np.uint16)
    n = rows.size
    d = x_disp.shape[1]
    h = wg.shape[1]
    h_out = np.empty((n, h), dtype=np.uint16)
    y_out = np.empty((n, d), dtype=np.uint16)
    g_out = np.empty((n, h), dtype=np.uint16) if save else None
    u_out = np.empty((n, h), dtype=np.uint16) if save else None
    lib().oracle_expert_ffn_rows(d, h, n, _p(rows), _p(experts), _p(x_disp), _p(wg), _p(wu),
                                 _p(wd), _p(h_out), _p(g_out), _p(u_out), _p(y_out))
    return h_out, g_out, u_out, y_out


def expert_ffn_bwd(count, offset, x_disp, g_save, u_save, h_act, dy_disp, wg, wu, wd, fill=0):
    """Grouped expert backward; returns dx_disp (bf16, tail = fill), dwg, dwu, dwd (fp32)."""
    count = _c(count, np.int32); offset = _c(offset, np.int32)
    x_disp, g_save, u_save, h_act, dy_disp, wg, wu, wd = (
        _c(v, np.uint16) for v in (x_disp, g_save, u_save, h_act, dy_disp, wg, wu, wd))
    R, d = x_disp.shape
    N, h, _ = wg.shape
    dx = np.full((R, d), fill, dtype=np.uint16)
    dwg = np.empty((N, h, d), dtype=np.float32)
    dwu = np.empty((N, h, d), dtype=np.float32)
    dwd = np.empty((N, d, h), dtype=np.float32)
    lib().oracle_expert_ffn_bwd(N, d, h, _p(count), _p(offset), _p(x_disp), _p(g_save),
                                _p(u_save), _p(h_act), _p(dy_disp), _p(wg), _p(wu), _p(wd),
                                _p(dx), _p(dwg), _p(dwu), _p(dwd))
    return dx, dwg, dwu, dwd


def router_bwd(x, w_r, idx, gate, dgate, dx=None, with_bias=True):
    """Router backward for a fixed top-K selection: returns dlogit [T,K],
    dx (the given dx plus the router's share; zeros if None), dW_r [N,d] and
    dbias [N] (None unless with_bias)."""
    x = _c(x, np.uint16); w_r = _c(w_r, np.float32)
    idx = _c(idx, np.int32); gate = _c(gate, np.float32); dgate = _c(dgate, np.float32)
    T, d = x.shape
    N = w_r.shape[0]
    K = idx.shape[1]
    dx = np.zeros((T, d), np.float32) if dx is None else np.array(dx, dtype=np.float32, copy=True)
    dlogit = np.empty((T, K), np.float32)
    dw = np.empty((N, d), np.float32)
    dbias = np.empty(N, np.float32) if with_bias else None
    lib().oracle_router_bwd(T, d, N, K, _p(x), _p(w_r), _p(idx), _p(gate), _p(dgate),
                            _p(dlogit), _p(dx), _p(dw), _p(dbias))
    return dlogit, dx, dw, dbias


# ------------------------------------------------------------- whole layer --

def layer_forward(x, w_r, bias, wg, wu, wd, K, cap, save=False):
    """Route -> dispatch -> grouped SwiGLU experts -> combine, all on the CPU."""
    r = route(x, w_r, bias, K, cap)
    N = w_r.shape[0]
    R = min(N * cap, x.shape[0] * K)
    x_disp = dispatch(x, r["route_row"], R)
    h_act, gs, us, y_disp = expert_ffn(x_disp, r["expert_count"], r["expert_offset"],
                                       wg, wu, wd, save=save)
    y = combine(y_disp, r["route_row"], r["topk_gate"])
    r.update(x_disp=x_disp, h_act=h_act, g_save=gs, u_save=us, y_disp=y_disp, y=y)
    return r


# ------------------------------------------------------------------- MXFP8 --

def mx_quantize(v):
    """MXFP8 of the rows of v (last dimension a multiple of 32): returns codes
    (uint8, same shape) and E8M0 scale bytes (uint8, last dimension / 32).
    uint16 input is read as bf16 bit patterns, anything else as float64."""
    v = np.asarray(v)
    k = v.shape[-1]
    rows = int(np.prod(v.shape[:-1], dtype=np.int64))
    q = np.empty(v.shape, dtype=np.uint8)
    sc = np.empty(v.shape[:-1] + (k // 32,), dtype=np.uint8)
    if v.dtype == np.uint16:
        v = _c(v, np.uint16)
        lib().oracle_mx_quantize_bf16(rows, k, _p(v), _p(q), _p(sc))
    else:
        v = _c(v, np.float64)
        lib().oracle_mx_quantize_f64(rows, k, _p(v), _p(q), _p(sc))
    return q, sc


def mx_dequantize(q, sc):
    """float64 values of MXFP8 codes q with scale bytes sc (one per 32 along the last dimension)."""
    q = _c(q, np.uint8); sc = _c(sc, np.uint8)
    k = q.shape[-1]
    rows = int(np.prod(q.shape[:-1], dtype=np.int64))
    out = np.empty(q.shape, dtype=np.float64)
    lib().oracle_mx_dequantize(rows, k, _p(q), _p(sc), _p(out))
    return out


def expert_ffn_mx(xq, xs, count, offset, wg, wu, wd, fill=0):
    """Grouped MXFP8 SwiGLU experts.  wg, wu, wd are (codes, scales) pairs of
    shapes [N,h,d]/[N,h,d/32] and [N,d,h]/[N,d,h/32].  Returns hq, hs, yq, ys
    (row-major scale rows); rows outside the experts' intervals keep ``fill``."""
    xq = _c(xq, np.uint8); xs = _c(xs, np.uint8)
    count = _c(count, np.int32); offset = _c(offset, np.int32)
    (wgq, wgs), (wuq, wus), (wdq, wds) = [(_c(a, np.uint8), _c(b, np.uint8)) for a, b in (wg, wu, wd)]
    R, d = xq.shape
    N, h, _ = wgq.shape
    hq = np.full((R, h), fill, np.uint8); hs = np.full((R, h // 32), fill, np.uint8)
    yq = np.full((R, d), fill, np.uint8); ys = np.full((R, d // 32), fill, np.uint8)
    lib().oracle_expert_ffn_mx(N, d, h, _p(count), _p(offset), _p(xq), _p(xs), _p(wgq), _p(wgs),
                               _p(wuq), _p(wus), _p(wdq), _p(wds), _p(hq), _p(hs), _p(yq), _p(ys))
    return hq, hs, yq, ys


def combine_mx(yq, ys, route_row, gate):
    """Gate-weighted sum of dequantized expert rows into token order (bf16 result)."""
    yq = _c(yq, np.uint8); ys = _c(ys, np.uint8)
    route_row = _c(route_row, np.int32); gate = _c(gate, np.float32)
    T, K = route_row.shape
    d = yq.shape[1]
    y = np.empty((T, d), dtype=np.uint16)
    lib().oracle_combine_mx(T, d, K, _p(yq), _p(ys), _p(route_row), _p(gate), _p(y))
    return y


def layer_forward_mx(x, w_r, bias, wg, wu, wd, K, cap):
    """The MXFP8 layer: route as in bf16; token rows quantized as they are
    dispatched; MXFP8 experts; quantized outputs combined.  Weights are bf16
    and quantized here along each product's reduction dimension."""
    r = route(x, w_r, bias, K, cap)
    N = w_r.shape[0]
    R = min(N * cap, x.shape[0] * K)
    xq_tok, xs_tok = mx_quantize(x)
    xq = np.zeros((R, x.shape[1]), np.uint8); xs = np.zeros((R, x.shape[1] // 32), np.uint8)
    rr = r["route_row"]
    for t, k in zip(*np.nonzero(rr >= 0)):
        xq[rr[t, k]] = xq_tok[t]; xs[rr[t, k]] = xs_tok[t]
    wq = [mx_quantize(w) for w in (wg, wu, wd)]
    hq, hs, yq, ys = expert_ffn_mx(xq, xs, r["expert_count"], r["expert_offset"], *wq)
    y = combine_mx(yq, ys, rr, r["topk_gate"])
    r.update(xq=xq, xs=xs, w_mx=wq, hq=hq, hs=hs, yq=yq, ys=ys, y=y)
    return r

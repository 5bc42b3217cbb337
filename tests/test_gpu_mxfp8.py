"""MXFP8 path on the GPU versus the CPU oracle, through the C ABI
(include/moe_mxfp8.h).

Bit-exact: weight quantization, the quantizing dispatch (codes and scale
bytes of every accepted route row; other rows untouched) and the dequantizing
combine, given identical inputs: each decision there is made on exactly
known values (bf16 inputs, or E4M3 x 2^k products).

Within a bound: the experts' quantized outputs H and Y.  The GPU accumulates
G, U and Y in fp32 on the tensor cores and the oracle in fp64, so a value
that lies within fp32 error of a rounding boundary (or of a power of two that
moves the block's shared exponent) can take the neighbouring code.  Each
such disagreement costs at most two code steps of the block's top binade,
2^(E + 6) for shared exponent E (one step, plus the step change when the
exponent moves by one near the saturation point), and disagreements are
rare: at least 99% of codes and scale bytes must be equal.  The layer output
inherits a bound of sum_k gate_k * 2^(E_k + 6) plus bf16 rounding.

Scale chunks (the GEMM operands' layout) are compared by gathering the bytes
of each valid row at the positions the header defines.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import MoEConfig

from _gpu_util import DEV, bf, f32, i32

pytestmark = pytest.mark.gpu

U8 = torch.uint8
FILL = 0xA5

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    "ragged": MoEConfig("mx_ragged", T=1000, d=256, N=16, K=4, h=384, cf_num=5, cf_den=4, seed=31),
    "zipf_ragged_cols": MoEConfig("mx_zipf", T=777, d=384, N=32, K=8, h=128, cf_num=1, cf_den=1,
                                  seed=32, zipf_s=1.2),
    "deep_experts": MoEConfig("mx_deep", T=2000, d=1152, N=8, K=2, h=256, cf_num=5, cf_den=4,
                              seed=33),
    "dense_N1": MoEConfig("mx_N1", T=300, d=128, N=1, K=1, h=128, cf_num=1, cf_den=1, seed=34),
    "many_experts": MoEConfig("mx_N200", T=600, d=128, N=200, K=6, h=128, cf_num=2, cf_den=1,
                              seed=35),
    "cap0": MoEConfig("mx_cap0", T=100, d=128, N=8, K=2, h=128, cf_num=0, cf_den=1, seed=36),
}


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _shape(moe, cfg):
    return moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def _np(t):
    return t.cpu().numpy()


# ----------------------------------------------------------- chunk layout --

def _chunk_pos(blk, rin, k):
    """Byte offsets [n, k/32] of the scales of rows (block128, row-in-block)."""
    kb = np.arange(k // 32)[None, :]
    blk = np.asarray(blk, np.int64)[:, None]
    rin = np.asarray(rin, np.int64)[:, None]
    return (blk * (k // 128) + kb // 4) * 512 + (rin % 32) * 16 + (rin // 32) * 4 + kb % 4


def _act_rows(count, offset):
    """Valid packed rows with their chunk block and row within the block."""
    pad = np.concatenate([[0], np.cumsum((np.asarray(count) + 127) // 128)])
    rows, blk, rin = [], [], []
    for e, c in enumerate(count):
        s = np.arange(c)
        rows.append(offset[e] + s)
        blk.append(pad[e] + s // 128)
        rin.append(s % 128)
    cat = lambda v: np.concatenate(v).astype(np.int64) if v else np.zeros(0, np.int64)
    return cat(rows), cat(blk), cat(rin)


def _to_chunks(scale_rows, blk, rin, k, nbytes):
    out = np.full(nbytes, FILL, np.uint8)
    if len(blk):
        out[_chunk_pos(blk, rin, k)] = scale_rows
    return out


def _weight_chunks(scales):
    """Row-major weight scales [E, rows, k/32] -> chunk bytes, every 512-byte
    chunk stored four times in a row (the weights' layout)."""
    E, rows, nb = scales.shape
    flat = scales.reshape(E * rows, nb)
    r = np.arange(E * rows)
    once = _to_chunks(flat, r // 128, r % 128, nb * 32, E * rows * nb).reshape(-1, 512)
    return np.repeat(once[:, None, :], 4, axis=1).reshape(-1)


# ---------------------------------------------------------------- bounds --

def _assert_mx_close(gq, gs, oq, os_, what, min_equal=0.99):
    """GPU (codes, scale rows) against the oracle's: every dequantized value
    within 2^(E+6) of the oracle's, and >= min_equal of codes and scales equal."""
    assert gq.shape == oq.shape and gs.shape == os_.shape, what
    if oq.size == 0:
        return
    gd = oracle.mx_dequantize(gq, gs)
    od = oracle.mx_dequantize(oq, os_)
    assert np.all(np.isfinite(gd)), f"{what}: non-finite"
    E = (os_.astype(np.int64) - 127).repeat(32, axis=-1)
    err = np.abs(gd - od)
    bad = err > np.exp2(E + 6)
    assert not bad.any(), f"{what}: {int(bad.sum())} values off by more than two code steps"
    eq_q = float((gq == oq).mean())
    eq_s = float((gs == os_).mean())
    assert eq_q >= min_equal and eq_s >= min_equal, f"{what}: codes {eq_q:.4f}, scales {eq_s:.4f} equal"


# ----------------------------------------------------------------- inputs --

def _oracle_route(cfg):
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    bias = synth.gen_bias(cfg)
    return x, wr, bias, oracle.route(x, wr, bias, cfg.K, cfg.cap)


def _scaled_weights(cfg):
    """Expert weights with a different power-of-two range per 32-block, so a
    block read with a neighbour's scale shows."""
    wg, wu, wd = synth.gen_expert_weights(cfg)
    rng = np.random.default_rng(cfg.seed + 1000)
    out = []
    for w in (wg, wu, wd):
        f = oracle.bf16_to_f32(w).astype(np.float64)
        nb = w.shape[-1] // 32
        sc = np.exp2(rng.integers(-4, 5, w.shape[:-1] + (nb,))).repeat(32, axis=-1)
        out.append(oracle.bf16_from_f64(f * sc))
    return out


def _route_tensors(ref):
    return (i32(ref["route_row"]), i32(ref["topk_idx"]), i32(ref["expert_count"]),
            i32(ref["expert_offset"]))


# ------------------------------------------------------------------ tests --

def test_quantize_weights_bit_exact(moe):
    rng = np.random.default_rng(7)
    E, rows, k = 3, 256, 384
    v = rng.standard_normal((E, rows, k)) * np.exp2(rng.integers(-30, 30, (E, rows, k // 32))).repeat(32, -1)
    v[0, 5, 32:64] = 0.0                      # an all-zero block
    v[1, 7, :32] = -0.0                       # negative zeros
    v[2, 9, 64:96] = 3e38                     # near the top of bf16
    v[2, 10, 96:128] *= 1e-38                 # bf16 subnormals
    w = oracle.bf16_from_f64(v)
    oq, os_ = oracle.mx_quantize(w)
    q = torch.full((E, rows, k), FILL, dtype=U8, device=DEV)
    sf = torch.full((E * rows * k // 8,), FILL, dtype=U8, device=DEV)
    moe.mx_quantize_weights(bf(w), q, sf)
    torch.cuda.synchronize()
    assert np.array_equal(_np(q), oq)
    assert np.array_equal(_np(sf), _weight_chunks(os_))


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_mxfp8_bit_exact(moe, name):
    cfg = CASES[name]
    x, wr, bias, ref = _oracle_route(cfg)
    s = _shape(moe, cfg)
    R = s.R
    xq = torch.full((max(R, 1), cfg.d), FILL, dtype=U8, device=DEV)
    nsf = max(moe.mx_act_scale_bytes(s, cfg.d), 16)
    xsf = torch.full((nsf,), FILL, dtype=U8, device=DEV)
    rr, ti, cnt, off = _route_tensors(ref)
    moe.dispatch_mxfp8(s, bf(x), rr, ti, cnt, off, xq, xsf)
    torch.cuda.synchronize()
    tq, ts = oracle.mx_quantize(x)
    rows, blk, rin = _act_rows(ref["expert_count"], ref["expert_offset"])
    gq = _np(xq)
    want_q = np.full_like(gq, FILL)
    want_sf = np.full(nsf, FILL, np.uint8)
    tok = np.full(max(R, 1), -1)
    for t, k in zip(*np.nonzero(ref["route_row"] >= 0)):
        tok[ref["route_row"][t, k]] = t
    if rows.size:
        want_q[rows] = tq[tok[rows]]
        want_sf[_chunk_pos(blk, rin, cfg.d)] = ts[tok[rows]]
    assert np.array_equal(gq, want_q), name
    assert np.array_equal(_np(xsf), want_sf), name


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf_ragged_cols", "cap0"])
def test_combine_mxfp8_bit_exact(moe, name):
    cfg = CASES[name]
    _, _, _, ref = _oracle_route(cfg)
    s = _shape(moe, cfg)
    R = max(s.R, 1)
    rng = np.random.default_rng(cfg.seed)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    yq = rng.choice(codes, (R, cfg.d)).astype(np.uint8)
    ys = rng.integers(110, 140, (R, cfg.d // 32)).astype(np.uint8)
    want = oracle.combine_mx(yq, ys, ref["route_row"], ref["topk_gate"])
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=DEV)
    moe.combine_mxfp8(s, _u8(yq), _u8(ys), i32(ref["route_row"]), f32(ref["topk_gate"]), y)
    torch.cuda.synchronize()
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want), name


def _run_ffn_mx(moe, cfg, ref, xq_rows, xs_rows, wq):
    """GPU experts on oracle-quantized inputs (scale rows moved into chunks)."""
    s = _shape(moe, cfg)
    R = max(s.R, 1)
    rows, blk, rin = _act_rows(ref["expert_count"], ref["expert_offset"])
    nsx = max(moe.mx_act_scale_bytes(s, cfg.d), 16)
    nsh = max(moe.mx_act_scale_bytes(s, cfg.h), 16)
    xsf = _to_chunks(xs_rows[rows], blk, rin, cfg.d, nsx)

    class W:
        pass
    w = W()
    (w.gate_q, gs), (w.up_q, us), (w.down_q, ds) = [(_u8(q), s_) for q, s_ in wq]
    w.gate_sf, w.up_sf, w.down_sf = (_u8(_weight_chunks(v)) for v in (gs, us, ds))
    hq = torch.full((R, cfg.h), FILL, dtype=U8, device=DEV)
    hsf = torch.full((nsh,), FILL, dtype=U8, device=DEV)
    yq = torch.full((R, cfg.d), FILL, dtype=U8, device=DEV)
    ys = torch.full((R, cfg.d // 32), FILL, dtype=U8, device=DEV)
    ws = torch.zeros(256, dtype=U8, device=DEV)
    moe.expert_ffn_mxfp8(s, _u8(xq_rows), _u8(xsf), i32(ref["expert_count"]),
                         i32(ref["expert_offset"]), w, hq, hsf, yq, ys, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws) == 0
    return rows, blk, rin, _np(hq), _np(hsf), _np(yq), _np(ys)


@pytest.mark.parametrize("name", list(CASES))
def test_expert_ffn_mxfp8(moe, name):
    cfg = CASES[name]
    x, wr, bias, ref = _oracle_route(cfg)
    R = max(min(cfg.N * cfg.cap, cfg.T * cfg.K), 1)
    wq = [oracle.mx_quantize(w) for w in _scaled_weights(cfg)]
    tq, ts = oracle.mx_quantize(x)
    xq = np.zeros((R, cfg.d), np.uint8)
    xs = np.zeros((R, cfg.d // 32), np.uint8)
    rr = ref["route_row"]
    for t, k in zip(*np.nonzero(rr >= 0)):
        xq[rr[t, k]] = tq[t]
        xs[rr[t, k]] = ts[t]
    ohq, ohs, oyq, oys = oracle.expert_ffn_mx(xq, xs, ref["expert_count"], ref["expert_offset"], *wq)
    rows, blk, rin, hq, hsf, yq, ys = _run_ffn_mx(moe, cfg, ref, xq, xs, wq)
    if rows.size == 0:
        assert np.all(hq == FILL) and np.all(yq == FILL)
        return
    ghs = hsf[_chunk_pos(blk, rin, cfg.h)]
    _assert_mx_close(hq[rows], ghs, ohq[rows], ohs[rows], f"{name}: H")
    _assert_mx_close(yq[rows], ys[rows], oyq[rows], oys[rows], f"{name}: Y")
    tail = np.setdiff1d(np.arange(R), rows)
    assert np.all(hq[tail] == FILL) and np.all(yq[tail] == FILL) and np.all(ys[tail] == FILL)


def _layer_bound(ref_mx, rr, gate):
    """Per output element: sum_k gate_k 2^(E_k + 6) over the token's accepted
    routes (E_k the oracle's shared exponent of that Y block)."""
    T, K = rr.shape
    d = ref_mx["yq"].shape[1]
    E = (ref_mx["ys"].astype(np.int64) - 127).repeat(32, axis=1)
    b = np.zeros((T, d))
    for k in range(K):
        ok = rr[:, k] >= 0
        b[ok] += np.abs(gate[ok, k])[:, None] * np.exp2(E[rr[ok, k]] + 6)
    return b


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf_ragged_cols", "deep_experts", "cap0"])
def test_layer_forward_mxfp8(moe, name):
    cfg = CASES[name]
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    bias = synth.gen_bias(cfg)
    wg, wu, wd = _scaled_weights(cfg)
    ref = oracle.layer_forward_mx(x, wr, bias, wg, wu, wd, cfg.K, cfg.cap)
    s = _shape(moe, cfg)
    buf = moe.MxLayerBuffers(s, DEV)
    w = moe.MxWeights(bf(wg), bf(wu), bf(wd))
    moe.layer_forward_mxfp8(buf, bf(x), f32(wr), None if bias is None else f32(bias), w)
    torch.cuda.synchronize()
    assert moe.read_device_error(buf.route_ws) == 0 and moe.read_device_error(buf.ffn_ws) == 0
    assert np.array_equal(_np(buf.route_row), ref["route_row"])
    got = oracle.bf16_to_f32(buf.y.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    want = oracle.bf16_to_f32(ref["y"]).astype(np.float64)
    bound = _layer_bound(ref, ref["route_row"], ref["topk_gate"]) + 2.0 ** -7 * np.abs(want)
    err = np.abs(got - want)
    assert np.all(err <= bound), f"{name}: {int((err > bound).sum())} outside the bound"
    if want.size and np.any(want):
        rel = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(want ** 2))
        assert rel < 1e-2, f"{name}: rms difference {rel:.3e}"


def test_full_size_sampled_rows(moe):
    """The OLMoE-1B-7B-shaped workload (T 8192, d 2048, 64 experts, top-8,
    h 1024) end to end on the GPU; 48 sampled packed rows recomputed by the
    oracle from the GPU's own quantized inputs' oracle counterparts."""
    cfg = synth.CONFIGS["olmoe"]
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    bias = synth.gen_bias(cfg)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    s = _shape(moe, cfg)
    buf = moe.MxLayerBuffers(s, DEV)
    w = moe.MxWeights(bf(wg), bf(wu), bf(wd))
    moe.layer_forward_mxfp8(buf, bf(x), f32(wr), None if bias is None else f32(bias), w)
    torch.cuda.synchronize()
    assert moe.read_device_error(buf.ffn_ws) == 0
    rr = _np(buf.route_row)
    cnt = _np(buf.expert_count)
    off = _np(buf.expert_offset)
    rng = np.random.default_rng(9)
    routes = np.argwhere(rr >= 0)
    pick = routes[rng.choice(len(routes), 48, replace=False)]
    pick = pick[np.argsort(rr[pick[:, 0], pick[:, 1]])]
    prow = rr[pick[:, 0], pick[:, 1]]
    pexp = np.searchsorted(off, prow, side="right") - 1
    # the oracle on the sampled rows alone: a packed problem of 48 rows
    tq, ts = oracle.mx_quantize(x[pick[:, 0]])
    sub_cnt = np.bincount(pexp, minlength=cfg.N).astype(np.int32)
    sub_off = np.concatenate([[0], np.cumsum(sub_cnt)]).astype(np.int32)
    wq = [oracle.mx_quantize(v) for v in (wg, wu, wd)]
    ohq, ohs, oyq, oys = oracle.expert_ffn_mx(tq, ts, sub_cnt, sub_off, *wq)
    gq = _np(buf.x_q)[prow]
    assert np.array_equal(gq, tq)
    slot = prow - off[pexp]
    pad = np.concatenate([[0], np.cumsum((cnt + 127) // 128)])
    blk = pad[pexp] + slot // 128
    ghs = _np(buf.h_sf)[_chunk_pos(blk, slot % 128, cfg.h)]
    _assert_mx_close(_np(buf.h_q)[prow], ghs, ohq, ohs, "olmoe: H", min_equal=0.98)
    _assert_mx_close(_np(buf.y_q)[prow], _np(buf.y_scale)[prow], oyq, oys, "olmoe: Y",
                     min_equal=0.98)


def test_mxfp8_graph_capture_and_determinism(moe):
    """The MXFP8 forward enqueues without host synchronisation, so it captures
    into a CUDA graph; replays, eager runs and the quantized intermediates
    are bitwise identical run to run."""
    cfg = CASES["ragged"]
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    wg, wu, wd = _scaled_weights(cfg)
    s = _shape(moe, cfg)
    w = moe.MxWeights(bf(wg), bf(wu), bf(wd))
    args = [bf(x), f32(wr), None, w]
    b1 = moe.MxLayerBuffers(s, DEV)
    b2 = moe.MxLayerBuffers(s, DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        moe.layer_forward_mxfp8(b1, *args)  # warm-up: one-time kernel attribute setup
        torch.cuda.synchronize()
        y_eager = b1.y.clone()
        hq_eager = b1.h_q.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.layer_forward_mxfp8(b2, *args)
        for _ in range(2):
            b2.y.zero_()
            g.replay()
    torch.cuda.synchronize()
    A = int(b1.expert_offset[-1])
    assert torch.equal(b2.y.view(torch.int16), y_eager.view(torch.int16))
    assert torch.equal(b2.h_q[:A], hq_eager[:A])
    moe.layer_forward_mxfp8(b1, *args)
    torch.cuda.synchronize()
    assert torch.equal(b1.y.view(torch.int16), y_eager.view(torch.int16))
    assert moe.read_device_error(b1.ffn_ws) == 0 and moe.read_device_error(b2.ffn_ws) == 0

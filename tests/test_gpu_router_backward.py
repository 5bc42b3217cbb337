"""GPU router backward (dlogit, dx += router term, dW_r, dbias) versus the CPU
oracle, through the C ABI.

The oracle sums in fp64; the GPU in fp32 in a fixed order.  Each output is
checked against a bound derived from that arithmetic: with
s_k = g_k (|dg_k| + sum_k' g_k' |dg_k'|) >= |dlogit_k| the scale of a route,
  dlogit: |err| <= 1e-5 s_k
  dx:     |err| <= 1e-5 (|dx_in| + sum_k s_k |W_r[e_k, j]|)
  dW_r:   |err| <= 3e-5 sum over routes of s_k |x[t, j]|
(fp32 chains of at most ~300 terms: 300 * 2^-24 < 2e-5, plus the dlogit
error), dbias likewise.  Inputs: the oracle's own routing of seeded tokens,
dgate drawn N(0, 1) and zero on dropped routes (as the combine backward
writes it), dx_in drawn N(0, 1).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import MoEConfig

from _gpu_util import DEV, bf, f32, i32

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    "ragged": MoEConfig("ragged", T=1000, d=256, N=16, K=4, h=64, cf_num=5, cf_den=4, seed=41),
    "zipf_bias": MoEConfig("zipf_bias", T=777, d=136, N=32, K=8, h=64, cf_num=1, cf_den=1,
                           seed=42, zipf_s=1.2),
    "K1": MoEConfig("K1", T=300, d=128, N=8, K=1, h=64, cf_num=1, cf_den=1, seed=43),
    "N1024_K16": MoEConfig("N1024_K16", T=300, d=64, N=1024, K=16, h=64, cf_num=1, cf_den=1,
                           seed=44),
    "N200": MoEConfig("N200", T=600, d=200, N=200, K=6, h=64, cf_num=2, cf_den=1, seed=45),
    # more sub-chunks than chunks: each CTA strides over several sub-chunks
    "many_chunks": MoEConfig("many_chunks", T=9000, d=64, N=16, K=2, h=64, cf_num=1, cf_den=1,
                             seed=46),
    "cap0": MoEConfig("cap0", T=100, d=64, N=8, K=2, h=64, cf_num=0, cf_den=1, seed=47),
    "T0": MoEConfig("T0", T=0, d=64, N=8, K=2, h=64, cf_num=1, cf_den=1, seed=48),
}


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _inputs(cfg):
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    bias = synth.gen_bias(cfg)
    if cfg.T:
        r = oracle.route(x, wr, bias, cfg.K, cfg.cap)
        idx, gate, row = r["topk_idx"], r["topk_gate"], r["route_row"]
    else:
        idx = np.zeros((0, cfg.K), np.int32)
        gate = np.zeros((0, cfg.K), np.float32)
        row = idx
    dg = synth.normal_f32(synth.stream_key(cfg.seed, "dgate"), (cfg.T, cfg.K))
    dg = np.where(row >= 0, dg, 0).astype(np.float32)
    dx0 = synth.normal_f32(synth.stream_key(cfg.seed, "dx_in"), (cfg.T, cfg.d))
    return x, wr, idx, gate, dg, dx0


def _run(moe, cfg, x, wr, idx, gate, dg, dx0, with_bias):
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    dlogit = torch.full((cfg.T, cfg.K), float("nan"), device=DEV)
    dx = f32(dx0)
    dw = torch.full((cfg.N, cfg.d), float("nan"), device=DEV)
    db = torch.full((cfg.N,), float("nan"), device=DEV) if with_bias else None
    ws = torch.zeros(max(moe.router_backward_workspace_bytes(s), 256), dtype=torch.uint8,
                     device=DEV)
    moe.router_backward(s, bf(x), f32(wr), i32(idx), f32(gate), f32(dg), dlogit, dx, dw, db, ws)
    torch.cuda.synchronize()
    return (dlogit.cpu().numpy(), dx.cpu().numpy(), dw.cpu().numpy(),
            None if db is None else db.cpu().numpy())


def _scales(cfg, x, wr, idx, gate, dg, dx0):
    g = gate.astype(np.float64)
    adg = np.abs(dg.astype(np.float64))
    sk = g * (adg + (g * adg).sum(1, keepdims=True))          # [T, K]
    dense = np.zeros((cfg.T, cfg.N))
    np.add.at(dense, (np.repeat(np.arange(cfg.T), cfg.K), idx.reshape(-1)), sk.reshape(-1))
    ax = np.abs(oracle.bf16_to_f32(x).astype(np.float64))
    s_dw = dense.T @ ax                                       # [N, d]
    s_db = dense.sum(0)
    s_dx = np.abs(dx0.astype(np.float64)) + dense @ np.abs(wr.astype(np.float64))
    return sk, s_dx, s_dw, s_db


def _check(got, want, scale, factor, what):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    bad = err > factor * scale + 1e-30
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{got.size} outside; "
                           f"max err/scale {np.max(err / (scale + 1e-30)):.3e}")


@pytest.mark.parametrize("name", list(CASES))
def test_router_backward_small(moe, name):
    cfg = CASES[name]
    x, wr, idx, gate, dg, dx0 = _inputs(cfg)
    with_bias = cfg.zipf_s is not None or name == "tiny"
    dl, dx, dw, db = _run(moe, cfg, x, wr, idx, gate, dg, dx0, with_bias)
    rdl, rdx, rdw, rdb = oracle.router_bwd(x, wr, idx, gate, dg, dx=dx0, with_bias=with_bias)
    sk, s_dx, s_dw, s_db = _scales(cfg, x, wr, idx, gate, dg, dx0)
    _check(dl, rdl, sk, 1e-5, f"{name} dlogit")
    _check(dx, rdx, s_dx, 1e-5, f"{name} dx")
    _check(dw, rdw, s_dw, 3e-5, f"{name} dw_router")
    if with_bias:
        _check(db, rdb, s_db, 3e-5, f"{name} dbias")
    if cfg.K == 1 or cfg.cap == 0 or cfg.T == 0:
        # one gate (always 1) or all dgate zero: no gradient at all
        assert np.all(dl == 0) and np.all(dw == 0) and np.array_equal(dx, dx0)
    unused = np.setdiff1d(np.arange(cfg.N), idx.reshape(-1))
    assert np.all(dw[unused] == 0)


def test_router_backward_full_size_and_deterministic(moe):
    """Training workload shapes (T=8192, d=2048, N=64, K=8): every output
    against the oracle, then a second call gives identical bits."""
    cfg = synth.CONFIGS["train"]
    x, wr, idx, gate, dg, dx0 = _inputs(cfg)
    dl, dx, dw, db = _run(moe, cfg, x, wr, idx, gate, dg, dx0, True)
    rdl, rdx, rdw, rdb = oracle.router_bwd(x, wr, idx, gate, dg, dx=dx0)
    sk, s_dx, s_dw, s_db = _scales(cfg, x, wr, idx, gate, dg, dx0)
    _check(dl, rdl, sk, 1e-5, "dlogit")
    _check(dx, rdx, s_dx, 1e-5, "dx")
    _check(dw, rdw, s_dw, 3e-5, "dw_router")
    _check(db, rdb, s_db, 3e-5, "dbias")
    dl2, dx2, dw2, db2 = _run(moe, cfg, x, wr, idx, gate, dg, dx0, True)
    for a, b in ((dl, dl2), (dx, dx2), (dw, dw2), (db, db2)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_layer_backward_with_router_term(moe):
    """The chained training step with the router backward appended: dW_r and
    the router's share of dx from the GPU's own dgate agree with the oracle."""
    cfg = synth.CONFIGS["tiny"].with_(T=1500, seed=49)
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    dy = synth.gen_dy(cfg)
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    fwd = moe.LayerBuffers(s, DEV, save_for_backward=True)
    W = [bf(wg), bf(wu), bf(wd)]
    xg, wrg = bf(x), f32(wr)
    moe.layer_forward(fwd, xg, wrg, None, *W)
    b0 = moe.BackwardBuffers(s, DEV)
    moe.layer_backward(fwd, b0, bf(dy), *W)
    torch.cuda.synchronize()
    dx_no_router = b0.dx.cpu().numpy().copy()
    b1 = moe.BackwardBuffers(s, DEV)
    moe.layer_backward(fwd, b1, bf(dy), *W, x=xg, w_router=wrg, with_bias=True)
    torch.cuda.synchronize()
    idx = fwd.topk_idx.cpu().numpy()
    gate = fwd.topk_gate.cpu().numpy()
    dg = b1.dgate.cpu().numpy()
    rdl, rdx, rdw, rdb = oracle.router_bwd(x, wr, idx, gate, dg, dx=dx_no_router)
    sk, s_dx, s_dw, s_db = _scales(cfg, x, wr, idx, gate, dg, dx_no_router)
    _check(b1.dlogit.cpu().numpy(), rdl, sk, 1e-5, "dlogit")
    _check(b1.dx.cpu().numpy(), rdx, s_dx, 1e-5, "dx")
    _check(b1.dw_router.cpu().numpy(), rdw, s_dw, 3e-5, "dw_router")
    _check(b1.dbias.cpu().numpy(), rdb, s_db, 3e-5, "dbias")


@pytest.mark.parametrize("name", ["tiny", "zipf_bias", "N1024_K16", "many_chunks", "cap0", "train"])
def test_fused_dispatch_router_backward_equals_two_step(moe, name):
    """moe_dispatch_router_backward + moe_router_weight_backward give the same
    bits as moe_dispatch_backward + moe_router_backward, and agree with the
    oracle's dispatch backward followed by its router backward."""
    cfg = synth.CONFIGS["train"] if name == "train" else CASES[name]
    x, wr, idx, gate, dg, _ = _inputs(cfg)
    r = oracle.route(x, wr, synth.gen_bias(cfg), cfg.K, cfg.cap)
    row = r["route_row"]
    dxd = synth.gen_bf16(cfg.seed, (cfg.R, cfg.d), "dx_disp")
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    ws = torch.zeros(max(moe.router_backward_workspace_bytes(s), 256), dtype=torch.uint8,
                     device=DEV)
    g_x, g_wr, g_idx, g_gate, g_dg = bf(x), f32(wr), i32(idx), f32(gate), f32(dg)
    g_row, g_dxd = i32(row), bf(dxd)

    def outs():
        return (torch.full((cfg.T, cfg.K), float("nan"), device=DEV),
                torch.full((cfg.T, cfg.d), float("nan"), device=DEV),
                torch.full((cfg.N, cfg.d), float("nan"), device=DEV),
                torch.full((cfg.N,), float("nan"), device=DEV))

    dl_a, dx_a, dw_a, db_a = outs()
    moe.dispatch_backward(s, g_dxd, g_row, dx_a)
    moe.router_backward(s, g_x, g_wr, g_idx, g_gate, g_dg, dl_a, dx_a, dw_a, db_a, ws)
    dl_b, dx_b, dw_b, db_b = outs()
    moe.dispatch_router_backward(s, g_dxd, g_row, g_wr, g_idx, g_gate, g_dg, dl_b, dx_b)
    moe.router_weight_backward(s, g_x, g_idx, dl_b, dw_b, db_b, ws)
    torch.cuda.synchronize()
    for a, b, what in ((dl_a, dl_b, "dlogit"), (dx_a, dx_b, "dx"), (dw_a, dw_b, "dw_router"),
                       (db_a, db_b, "dbias")):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), what
    dx0 = oracle.dispatch_bwd(dxd, row, cfg.T)
    rdl, rdx, rdw, rdb = oracle.router_bwd(x, wr, idx, gate, dg, dx=dx0)
    sk, s_dx, s_dw, s_db = _scales(cfg, x, wr, idx, gate, dg, dx0)
    # the dispatch part is an fp32 sum of up to K bf16 values (the oracle's
    # is the same chain): its rounding is covered by K ulp of |dx0|'s terms
    s_dx = s_dx + cfg.K * np.abs(dx0)
    _check(dl_b.cpu().numpy(), rdl, sk, 1e-5, f"{name} dlogit")
    _check(dx_b.cpu().numpy(), rdx, s_dx, 1e-5, f"{name} dx")
    _check(dw_b.cpu().numpy(), rdw, s_dw, 3e-5, f"{name} dw_router")
    _check(db_b.cpu().numpy(), rdb, s_db, 3e-5, f"{name} dbias")

"""GPU backward of the layer versus the CPU oracle, through the C ABI.

moe_expert_ffn_backward on small cases (every output compared), on the
full-size training workload (sampled rows and one expert's whole weight
gradient), and the chained training step (forward, combine backward, expert
backward, dispatch backward) on sampled tokens whose gradients the oracle
computes one by one.  Unwritten tail rows hold NaN throughout: a weight
gradient that read one would not be finite.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import MoEConfig

from _gpu_util import DEV, as64, assert_close_bf16, bf, bits, f32, i32

pytestmark = pytest.mark.gpu

NAN = 0x7FC1
SMALL = {
    "tiny": synth.CONFIGS["tiny"],
    "ragged": MoEConfig("ragged", T=1000, d=256, N=16, K=4, h=192, cf_num=5, cf_den=4, seed=11),
    "zipf_drops": MoEConfig("zipf_drops", T=777, d=128, N=32, K=8, h=128, cf_num=1, cf_den=1,
                            seed=12, zipf_s=1.2),
    "wide_ragged": MoEConfig("wide_ragged", T=513, d=320, N=4, K=2, h=256, cf_num=3, cf_den=2,
                             seed=13, router_std=0.01),
    "dense_N1": MoEConfig("dense_N1", T=300, d=128, N=1, K=1, h=128, cf_num=1, cf_den=1, seed=14),
    "N200": MoEConfig("N200", T=600, d=192, N=200, K=6, h=64, cf_num=2, cf_den=1, seed=18),
    "cap0": MoEConfig("cap0", T=100, d=64, N=8, K=2, h=64, cf_num=0, cf_den=1, seed=16),
}


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    return m


def _poisoned(a, A):
    out = np.array(a, dtype=np.uint16, copy=True)
    out[A:] = NAN
    return out


def assert_close_f32(got, want, what, rel=2e-2, abs_=1e-2):
    g = np.asarray(got, dtype=np.float64)
    w = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    err = np.abs(g - w)
    assert np.all(err <= abs_ + rel * np.abs(w)), f"{what}: max err {err.max():.3e}"
    rms = float(np.sqrt(np.mean(w ** 2))) if w.size else 0.0
    bad = err > rel * np.abs(w) + abs_ * rms
    assert not bad.any(), f"{what}: {int(bad.sum())}/{w.size} outside; max err {err.max():.3e}"


def _run_bwd(moe, cfg, xd, cnt, off, wg, wu, wd, gs, us, ha, dyd):
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    dx = torch.full((cfg.R, cfg.d), NAN, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    dwg = torch.full((cfg.N, cfg.h, cfg.d), float("nan"), dtype=torch.float32, device=DEV)
    dwu = torch.full_like(dwg, float("nan"))
    dwd = torch.full((cfg.N, cfg.d, cfg.h), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(moe.expert_ffn_backward_workspace_bytes(s), dtype=torch.uint8, device=DEV)
    moe.expert_ffn_backward(s, bf(xd), i32(cnt), i32(off), bf(wg), bf(wu), bf(wd), bf(gs), bf(us),
                            bf(ha), bf(dyd), dx, dwg, dwu, dwd, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws) == 0
    return bits(dx), dwg.cpu().numpy(), dwu.cpu().numpy(), dwd.cpu().numpy()


@pytest.mark.parametrize("name", list(SMALL))
def test_expert_backward_small(moe, name):
    cfg = SMALL[name]
    x = synth.gen_x(cfg)
    wr, bias = synth.gen_router(cfg), synth.gen_bias(cfg)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    ref = oracle.layer_forward(x, wr, bias, wg, wu, wd, cfg.K, cfg.cap, save=True)
    cnt, off = ref["expert_count"], ref["expert_offset"]
    A = int(off[-1])
    dyd = synth.gen_bf16(cfg.seed, (cfg.R, cfg.d), "dy_disp", 0.1)
    ins = [_poisoned(ref[k], A) for k in ("x_disp", "g_save", "u_save", "h_act")]
    dyd = _poisoned(dyd, A)
    dx, dwg, dwu, dwd = _run_bwd(moe, cfg, ins[0], cnt, off, wg, wu, wd, ins[1], ins[2], ins[3], dyd)
    rdx, rdwg, rdwu, rdwd = oracle.expert_ffn_bwd(cnt, off, ins[0], ins[1], ins[2], ins[3], dyd,
                                                  wg, wu, wd, fill=NAN)
    assert np.all(dx[A:] == NAN)
    if A:
        assert_close_bf16(dx[:A], rdx[:A], f"{name} dx_disp")
    assert_close_f32(dwg, rdwg, f"{name} dw_gate")
    assert_close_f32(dwu, rdwu, f"{name} dw_up")
    assert_close_f32(dwd, rdwd, f"{name} dw_down")
    empty = cnt == 0
    if empty.any():
        assert np.all(dwg[empty] == 0) and np.all(dwd[empty] == 0)


def test_expert_backward_full_size(moe):
    """Training workload shapes with synthetic saved activations: 48 sampled
    rows of dx_disp and the whole weight gradient of one expert."""
    cfg = synth.CONFIGS["train"]
    x = synth.gen_x(cfg)
    r = oracle.route(x, synth.gen_router(cfg), None, cfg.K, cfg.cap)
    cnt, off = r["expert_count"], r["expert_offset"]
    A = int(off[-1])
    wg, wu, wd = synth.gen_expert_weights(cfg)
    sd = cfg.seed + 100
    xd = _poisoned(oracle.dispatch(x, r["route_row"], cfg.R), A)
    gs = _poisoned(synth.gen_bf16(sd, (cfg.R, cfg.h), "g_save", 0.9), A)
    us = _poisoned(synth.gen_bf16(sd, (cfg.R, cfg.h), "u_save", 0.9), A)
    ha = _poisoned(synth.gen_bf16(sd, (cfg.R, cfg.h), "h_act", 0.3), A)
    dyd = _poisoned(synth.gen_bf16(sd, (cfg.R, cfg.d), "dy_disp", 0.1), A)
    dx, dwg, dwu, dwd = _run_bwd(moe, cfg, xd, cnt, off, wg, wu, wd, gs, us, ha, dyd)
    assert np.all(np.isfinite(dwg)) and np.all(np.isfinite(dwu)) and np.all(np.isfinite(dwd))
    f = oracle.bf16_to_f32
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(A, size=48, replace=False))
    for rrow in rows:
        e = int(np.searchsorted(off, rrow, side="right") - 1)
        sl = slice(rrow, rrow + 1)
        rdx, _, _, _ = oracle.ffn_bwd_f64(f(xd[sl]), f(gs[sl]), f(us[sl]), f(ha[sl]), f(dyd[sl]),
                                          f(wg[e]), f(wu[e]), f(wd[e]), round_dgu=True)
        assert_close_bf16(dx[sl], oracle.bf16_from_f64(rdx), f"dx_disp row {rrow}")
    e = int(np.argmax(cnt))
    sl = slice(int(off[e]), int(off[e] + cnt[e]))
    rdx, rdwg, rdwu, rdwd = oracle.ffn_bwd_f64(f(xd[sl]), f(gs[sl]), f(us[sl]), f(ha[sl]),
                                               f(dyd[sl]), f(wg[e]), f(wu[e]), f(wd[e]), round_dgu=True)
    assert_close_f32(dwg[e], rdwg, "dw_gate[e]")
    assert_close_f32(dwu[e], rdwu, "dw_up[e]")
    assert_close_f32(dwd[e], rdwd, "dw_down[e]")
    assert_close_bf16(dx[sl], oracle.bf16_from_f64(rdx), "dx_disp rows of e")

    # the same call six more times on device-resident inputs: every output bit
    # for bit the first run's (the weight gradients bound each tile's last
    # k-block through map copies rewritten on the device, tile after tile)
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    ins = [bf(a) for a in (xd, wg, wu, wd, gs, us, ha, dyd)]
    cnt_d, off_d = i32(cnt), i32(off)
    ws = torch.zeros(moe.expert_ffn_backward_workspace_bytes(s), dtype=torch.uint8, device=DEV)
    first = None
    for _ in range(6):
        dxr = torch.full((cfg.R, cfg.d), NAN, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        outs = [torch.full((cfg.N, cfg.h, cfg.d), float("nan"), dtype=torch.float32, device=DEV)
                for _ in range(2)]
        outs.append(torch.full((cfg.N, cfg.d, cfg.h), float("nan"), dtype=torch.float32,
                               device=DEV))
        moe.expert_ffn_backward(s, ins[0], cnt_d, off_d, ins[1], ins[2], ins[3], ins[4], ins[5],
                                ins[6], ins[7], dxr, outs[0], outs[1], outs[2], ws)
        got = [dxr.view(torch.int16)[:A]] + outs
        if first is None:
            first = got
            assert np.array_equal(got[0].cpu().numpy().view(np.uint16), dx[:A])
        else:
            assert all(torch.equal(a, b) for a, b in zip(got, first))
    torch.cuda.synchronize()
    assert moe.read_device_error(ws) == 0


def test_training_step_chain_full_size(moe):
    """Forward with saving, then combine backward, expert backward and dispatch
    backward on the GPU; dgate and dx of 12 sampled tokens against the oracle,
    which recomputes each of their routes row by row."""
    cfg = synth.CONFIGS["train"]
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    dy = synth.gen_dy(cfg)
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    fwd = moe.LayerBuffers(s, DEV, save_for_backward=True)
    bwd = moe.BackwardBuffers(s, DEV)
    W = [bf(wg), bf(wu), bf(wd)]
    moe.layer_forward(fwd, bf(x), f32(wr), None, *W)
    moe.layer_backward(fwd, bwd, bf(dy), *W)
    torch.cuda.synchronize()
    assert moe.read_device_error(bwd.ws) == 0
    r = oracle.route(x, wr, None, cfg.K, cfg.cap)
    np.testing.assert_array_equal(fwd.route_row.cpu().numpy(), r["route_row"])
    row, idx, gate = r["route_row"], r["topk_idx"], r["topk_gate"]
    f = oracle.bf16_to_f32
    rng = np.random.default_rng(9)
    toks = rng.choice(cfg.T, size=12, replace=False)
    got_dg = bwd.dgate.cpu().numpy()
    got_dx = bwd.dx.cpu().numpy()
    for t in toks:
        dx_t = np.zeros(cfg.d, np.float32)
        dg_ref = np.zeros(cfg.K, np.float32)
        for k in range(cfg.K):
            if row[t, k] < 0:
                continue
            e = int(idx[t, k])
            h_o, g_o, u_o, y_o = oracle.expert_ffn_rows(np.array([0], np.int32),
                                                        np.array([e], np.int32), x[t:t + 1],
                                                        wg, wu, wd, save=True)
            dyd_r, dg_r = oracle.combine_bwd(dy[t:t + 1], y_o, np.array([[0]], np.int32),
                                             gate[t:t + 1, k:k + 1])
            dg_ref[k] = dg_r[0, 0]
            rdx, _, _, _ = oracle.ffn_bwd_f64(f(x[t:t + 1]), f(g_o), f(u_o), f(h_o), f(dyd_r),
                                              f(wg[e]), f(wu[e]), f(wd[e]), round_dgu=True)
            dx_t = dx_t + f(oracle.bf16_from_f64(rdx))[0]
        assert_close_f32(got_dg[t], dg_ref, f"dgate token {t}", rel=2e-2, abs_=1e-2)
        assert_close_f32(got_dx[t], dx_t, f"dx token {t}")

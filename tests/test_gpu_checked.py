"""Checked row movements (moe_dispatch_checked, moe_combine_checked,
moe_combine_backward_checked, moe_dispatch_backward_checked).

A route map built on the host with rows past the capacity buffers (R and
beyond) is passed to the checked calls: each out-of-range route is skipped,
so nothing is read or written through it, and the status word records
MOE_ERR_DEVICE_ROUTE_RANGE.  The outputs equal the oracle's for the same map
with those entries set to -1 (a dropped route, Section 05, 5.4).  On a valid
map the checked calls give the release calls' bits and leave the status 0.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import MoEConfig

from _gpu_util import DEV, bf, bits, f32, i32

pytestmark = pytest.mark.gpu

SENT = 0x7FC1
ROUTE_RANGE = 7


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    return m


def _case(K):
    cfg = MoEConfig("checked", T=1500, d=264, N=24, K=K, h=64, cf_num=1, cf_den=1, seed=51 + K)
    idx = synth.gen_topk_idx(cfg.seed, cfg.T, cfg.N, cfg.K)
    row, count, offset, demand = oracle.route_slots(idx, cfg.N, cfg.cap)
    gate = synth.gen_gates(cfg.seed, cfg.T, cfg.K)
    x = synth.gen_bf16(cfg.seed, (cfg.T, cfg.d), "x")
    yd = synth.gen_bf16(cfg.seed, (cfg.R, cfg.d), "y_disp")
    dy = synth.gen_bf16(cfg.seed, (cfg.T, cfg.d), "dy")
    return cfg, row, gate, x, yd, dy


def _run(moe, cfg, row, gate, x, yd, dy, checked):
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    out = dict(x_disp=torch.full((cfg.R, cfg.d), SENT, dtype=torch.int16, device=DEV).view(torch.bfloat16),
               y=torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=DEV),
               dy_disp=torch.full((cfg.R, cfg.d), SENT, dtype=torch.int16, device=DEV).view(torch.bfloat16),
               dgate=torch.empty((cfg.T, cfg.K), dtype=torch.float32, device=DEV),
               dx=torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=DEV))
    r, g = i32(row), f32(gate)
    if checked:
        moe.dispatch_checked(s, bf(x), r, out["x_disp"], ws)
        moe.combine_checked(s, bf(yd), r, g, out["y"], ws)
        moe.combine_backward_checked(s, bf(dy), bf(yd), r, g, out["dy_disp"], out["dgate"], ws)
        moe.dispatch_backward_checked(s, bf(yd), r, out["dx"], ws)
    else:
        moe.dispatch(s, bf(x), r, out["x_disp"])
        moe.combine(s, bf(yd), r, g, out["y"])
        moe.combine_backward(s, bf(dy), bf(yd), r, g, out["dy_disp"], out["dgate"])
        moe.dispatch_backward(s, bf(yd), r, out["dx"])
    torch.cuda.synchronize()
    status = moe.read_device_error(ws)
    return {k: (bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()) for k, v in out.items()}, status


@pytest.mark.parametrize("K", [4, 12])
def test_checked_calls_equal_release_calls_on_a_valid_map(moe, K):
    cfg, row, gate, x, yd, dy = _case(K)
    assert (row < 0).any()
    rel, st0 = _run(moe, cfg, row, gate, x, yd, dy, checked=False)
    chk, st1 = _run(moe, cfg, row, gate, x, yd, dy, checked=True)
    assert st1 == 0
    for k in rel:
        np.testing.assert_array_equal(chk[k], rel[k], err_msg=k)


@pytest.mark.parametrize("K", [4, 12])
def test_checked_calls_skip_rows_past_the_buffers(moe, K):
    cfg, row, gate, x, yd, dy = _case(K)
    R = cfg.R
    bad = row.copy()
    rng = np.random.default_rng(K)
    picks = rng.choice(cfg.T * cfg.K, size=6, replace=False)
    flat = bad.reshape(-1)
    flat[picks[0]] = R
    flat[picks[1]] = R + 1
    flat[picks[2]] = R + 100000
    flat[picks[3]] = 2 ** 30
    flat[picks[4]] = 2 ** 31 - 1
    flat[picks[5]] = -7  # any negative row is a dropped route, not an error
    got, status = _run(moe, cfg, bad, gate, x, yd, dy, checked=True)
    assert status == ROUTE_RANGE
    fixed = np.where(bad >= R, -1, bad).astype(np.int32)
    np.testing.assert_array_equal(got["x_disp"], oracle.dispatch(x, fixed, R, fill=SENT))
    np.testing.assert_array_equal(got["y"], oracle.combine(yd, fixed, gate))
    ref_dyd, ref_dg = oracle.combine_bwd(dy, yd, fixed, gate, fill=SENT)
    np.testing.assert_array_equal(got["dy_disp"], ref_dyd)
    assert np.all(got["dgate"][fixed < 0] == 0)
    w = ref_dg.astype(np.float64)
    rms = np.sqrt(np.mean(w ** 2))
    assert np.all(np.abs(got["dgate"].astype(np.float64) - w) <= 1e-4 * np.abs(w) + 1e-5 * rms)
    np.testing.assert_array_equal(got["dx"], oracle.dispatch_bwd(yd, fixed, cfg.T))
    # the word was read and cleared: a valid map afterwards leaves it 0
    _, status = _run(moe, cfg, row, gate, x, yd, dy, checked=True)
    assert status == 0

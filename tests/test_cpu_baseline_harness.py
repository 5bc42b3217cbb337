"""The benchmark's CPU baseline splits the oracle's work over host threads.
The split must not change what is computed: on small workloads the threaded
harness gives the oracle's own results (bit for bit; the router-weight
gradient, summed from per-thread partials, within fp32 rounding)."""
import numpy as np
import pytest

import bench
import oracle
import synth
from synth import MoEConfig


def _plain(cfg, inp, tokens):
    sub = cfg.with_(T=tokens)
    x = inp["x"][:tokens]
    wg, wu, wd = inp["w"]
    out = oracle.layer_forward(x, inp["wr"], inp["bias"], wg, wu, wd, cfg.K, sub.cap,
                               save=cfg.backward)
    if cfg.backward:
        dyd, dg = oracle.combine_bwd(inp["dy"][:tokens], out["y_disp"], out["route_row"],
                                     out["topk_gate"])
        dxd, dwg, dwu, dwd = oracle.expert_ffn_bwd(out["expert_count"], out["expert_offset"],
                                                   out["x_disp"], out["g_save"], out["u_save"],
                                                   out["h_act"], dyd, wg, wu, wd)
        dx = oracle.dispatch_bwd(dxd, out["route_row"], tokens)
        dl, dx, dwr, _ = oracle.router_bwd(x, inp["wr"], out["topk_idx"], out["topk_gate"], dg,
                                           dx=dx, with_bias=inp["bias"] is not None)
        out.update(dgate=dg, dy_disp=dyd, dx_disp=dxd, dw_gate=dwg, dw_up=dwu, dw_down=dwd,
                   dlogit=dl, dx=dx, dw_router=dwr)
    return out


@pytest.mark.parametrize("cfg,tokens,threads", [
    (synth.CONFIGS["tiny"], 200, 3),
    (MoEConfig("zipf_small", T=300, d=128, N=16, K=4, h=64, cf_num=1, cf_den=1, seed=41,
               zipf_s=1.2), 300, 4),
    (MoEConfig("train_small", T=96, d=64, N=8, K=2, h=64, cf_num=5, cf_den=4, seed=42,
               backward=True), 96, 5),
])
def test_threaded_oracle_equals_the_oracle(cfg, tokens, threads):
    inp = bench._oracle_inputs(cfg)
    want = _plain(cfg, inp, tokens)
    A = int(want["expert_offset"][-1])
    for t in (1, threads):
        got = bench.oracle_layer(cfg, inp, tokens, t)
        for k in ("logits", "topk_idx", "topk_gate", "route_row", "expert_count", "expert_offset",
                  "y"):
            np.testing.assert_array_equal(got[k], want[k], err_msg=f"{k}, {t} threads")
        for k in ("x_disp", "h_act", "y_disp"):
            np.testing.assert_array_equal(got[k][:A], want[k][:A], err_msg=f"{k}, {t} threads")
        if cfg.backward:
            for k in ("dgate", "dlogit", "dx", "dw_gate", "dw_up", "dw_down"):
                np.testing.assert_array_equal(got[k], want[k], err_msg=f"{k}, {t} threads")
            for k in ("dy_disp", "dx_disp"):
                np.testing.assert_array_equal(got[k][:A], want[k][:A], err_msg=k)
            np.testing.assert_allclose(got["dw_router"], want["dw_router"], rtol=1e-5, atol=1e-6)


def test_expert_ranges_cover_every_expert_once():
    count = np.array([0, 5, 0, 0, 9, 1, 1, 30, 0, 2], np.int32)
    for parts in (1, 2, 3, 7, 20):
        r = bench._expert_ranges(count, parts)
        assert r[0][0] == 0 and r[-1][1] == len(count)
        assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
        assert len(r) <= parts

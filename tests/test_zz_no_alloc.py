"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc, for example a plugin that its host
framework hands only input and output buffers, or a latency-critical loop
where an allocation that may synchronise the device is not allowed.  For them
moe_route_noalloc keeps its scratch in a fixed array inside the library.  This
test calls it through the C ABI twice in a row, on different inputs and
shapes (so stale scratch from the first call would show up in the second),
and checks each result against moe_route on the same inputs.  It also checks
that shapes whose scratch would not fit are refused before any work.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import synth
from synth import MoEConfig

from _gpu_util import DEV, bf, f32

pytestmark = pytest.mark.gpu

CASES = [
    MoEConfig("noalloc_a", T=1000, d=256, N=16, K=4, h=64, cf_num=5, cf_den=4, seed=31),
    MoEConfig("noalloc_b", T=8192, d=2048, N=64, K=8, h=64, cf_num=1, cf_den=1, seed=32,
              zipf_s=1.2),
]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    f = m.lib().moe_route_noalloc
    f.argtypes = [ctypes.POINTER(m.Shape)] + [ctypes.c_void_p] * 10
    f.restype = ctypes.c_int
    return m


def _outputs(cfg):
    e = dict(device=DEV)
    return dict(topk_idx=torch.empty((cfg.T, cfg.K), dtype=torch.int32, **e),
                topk_gate=torch.empty((cfg.T, cfg.K), dtype=torch.float32, **e),
                route_row=torch.empty((cfg.T, cfg.K), dtype=torch.int32, **e),
                expert_count=torch.empty(cfg.N, dtype=torch.int32, **e),
                expert_offset=torch.empty(cfg.N + 1, dtype=torch.int32, **e),
                expert_demand=torch.empty(cfg.N, dtype=torch.int32, **e))


def test_route_noalloc_matches_route_on_two_calls_in_a_row(moe):
    results = []
    for cfg in CASES:
        x = bf(synth.gen_x(cfg))
        wr = f32(synth.gen_router(cfg))
        b = synth.gen_bias(cfg)
        bias = None if b is None else f32(b)
        s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
        mine = _outputs(cfg)
        o = mine
        stream = torch.cuda.current_stream().cuda_stream
        rc = moe.lib().moe_route_noalloc(
            ctypes.byref(s), x.data_ptr(), wr.data_ptr(), None if bias is None else bias.data_ptr(),
            o["topk_idx"].data_ptr(), o["topk_gate"].data_ptr(), o["route_row"].data_ptr(),
            o["expert_count"].data_ptr(), o["expert_offset"].data_ptr(),
            o["expert_demand"].data_ptr(), stream)
        assert rc == 0, moe.lib().moe_status_string(rc)
        ref = _outputs(cfg)
        ws = torch.zeros(moe.route_workspace_bytes(s), dtype=torch.uint8, device=DEV)
        moe.route(s, x, wr, bias, ref["topk_idx"], ref["topk_gate"], ref["route_row"],
                  ref["expert_count"], ref["expert_offset"], ref["expert_demand"], ws)
        torch.cuda.synchronize()
        results.append((mine, ref))
    # the same kernels on the same inputs: every output is bit-identical
    for cfg, (mine, ref) in zip(CASES, results):
        for k in ("topk_idx", "topk_gate", "route_row", "expert_count", "expert_offset",
                  "expert_demand"):
            assert torch.equal(mine[k], ref[k]), (cfg.name, k)
    assert int(results[1][0]["expert_offset"][-1]) < CASES[1].T * CASES[1].K  # drops happened


def test_route_noalloc_refuses_shapes_past_its_scratch(moe):
    """A shape whose logits alone (70000 x 1024 fp32, 273 MiB) exceed the
    64 MiB array is refused before anything is enqueued.  Every buffer the
    caller passes is a real device tensor of the shape's size."""
    cfg = MoEConfig("noalloc_big", T=70000, d=64, N=1024, K=2, h=64, cf_num=1, cf_den=1, seed=33)
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    assert moe.route_workspace_bytes(s) > (64 << 20)
    x = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros((cfg.N, cfg.d), dtype=torch.float32, device=DEV)
    o = _outputs(cfg)
    torch.cuda.synchronize()
    rc = moe.lib().moe_route_noalloc(
        ctypes.byref(s), x.data_ptr(), wr.data_ptr(), None, o["topk_idx"].data_ptr(),
        o["topk_gate"].data_ptr(), o["route_row"].data_ptr(), o["expert_count"].data_ptr(),
        o["expert_offset"].data_ptr(), o["expert_demand"].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 5  # MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()

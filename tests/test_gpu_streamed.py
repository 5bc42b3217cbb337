"""StreamedLayer: batches whose host copies overlap the neighbouring batches'
layer work give, batch for batch, exactly the results of the plain
single-stream calls (a reuse race between the two alternating buffer sets
would show as a wrong batch)."""
import numpy as np
import pytest
import torch

import synth

from _gpu_util import DEV, bf, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("backward", [False, True])
def test_streamed_batches_match_plain_calls(moe, backward):
    cfg = synth.CONFIGS["tiny"]
    s = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    wr = f32(synth.gen_router(cfg))
    wg, wu, wd = (bf(a) for a in synth.gen_expert_weights(cfg))
    nb = 6
    xs = [synth.gen_x(cfg.with_(seed=100 + i)) for i in range(nb)]
    dys = [synth.gen_dy(cfg.with_(seed=200 + i)) for i in range(nb)]
    pin = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_host = [pin(a) for a in xs]
    dy_host = [pin(a) for a in dys] if backward else [None] * nb
    y_host = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    dx_host = ([torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory() for _ in range(nb)]
               if backward else [None] * nb)
    sl = moe.StreamedLayer(s, wr, None, wg, wu, wd, DEV, backward=backward)
    for i in range(nb):
        sl.submit(x_host[i], y_host[i], dy_host[i], dx_host[i])
    sl.synchronize()
    assert sl.status() == 0
    fb = moe.LayerBuffers(s, DEV, save_for_backward=backward)
    bb = moe.BackwardBuffers(s, DEV) if backward else None
    for i in range(nb):
        x = bf(xs[i])
        moe.layer_forward(fb, x, wr, None, wg, wu, wd)
        if backward:
            moe.layer_backward(fb, bb, bf(dys[i]), wg, wu, wd, x=x, w_router=wr)
        torch.cuda.synchronize()
        assert torch.equal(y_host[i].view(torch.int16), fb.y.cpu().view(torch.int16)), i
        if backward:
            assert torch.equal(dx_host[i], bb.dx.cpu()), i

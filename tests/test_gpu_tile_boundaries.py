"""Grouped expert GEMMs at every tile boundary.

The forward kernel computes an expert's rows in 256-row tiles; a last tile
with at most 128 valid rows runs with the operands exchanged (weights as the
256-row operand, the tile's tokens rounded up to 32 as the other), a longer
last tile as an ordinary 256-row tile.  Here the expert counts sit on both
sides of each boundary (0, 1, 31..33, 127..129, 255..257, 383..385, 512) and
h, d are not multiples of the 128 / 256 output columns of a tile, so every
kind of tile and every column tail runs.  moe_expert_ffn is called directly
on seeded packed rows and compared with the oracle on every valid row; the
tail rows stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from _gpu_util import DEV, assert_close_bf16, bf, bits, i32

pytestmark = pytest.mark.gpu

SENT = 0x7FC1
COUNTS = [0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 383, 384, 385, 512, 7]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    return m


@pytest.mark.parametrize("d,h,save", [(192, 320, True), (320, 192, False), (128, 64, True)])
def test_expert_ffn_at_tile_boundaries(moe, d, h, save):
    N = len(COUNTS)
    count = np.array(COUNTS, np.int32)
    offset = np.concatenate([[0], np.cumsum(count)]).astype(np.int32)
    A = int(offset[-1])
    R = A + 40  # a tail of rows past the packed prefix, read by the last tiles
    T, K = R, 1  # R = min(N * cap, T * K) = T
    cap = int(count.max())
    seed = 61 + d + h
    x_disp = synth.gen_bf16(seed, (R, d), "x_disp")
    x_disp[A:] = SENT  # NaN tail: must not reach any stored row
    wg = synth.gen_bf16(seed, (N, h, d), "w_gate", std=0.02)
    wu = synth.gen_bf16(seed, (N, h, d), "w_up", std=0.02)
    wd = synth.gen_bf16(seed, (N, d, h), "w_down", std=0.02)
    ref_h, ref_g, ref_u, ref_y = oracle.expert_ffn(x_disp, count, offset, wg, wu, wd, save=save,
                                                   fill=SENT)
    s = moe.Shape(T, d, N, K, h, cap)
    assert s.R == R
    rows = R
    xd = torch.full((rows, d), SENT, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    xd[:R] = bf(x_disp)
    out = {k: torch.full((rows, w), SENT, dtype=torch.int16, device=DEV).view(torch.bfloat16)
           for k, w in (("h", h), ("y", d), ("g", h), ("u", h))}
    ws = torch.zeros(moe.expert_ffn_workspace_bytes(s), dtype=torch.uint8, device=DEV)
    moe.expert_ffn(s, xd, i32(count), i32(offset), bf(wg), bf(wu), bf(wd), out["h"],
                   out["g"] if save else None, out["u"] if save else None, out["y"], ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws) == 0
    for k, ref in (("h", ref_h), ("y", ref_y)) + ((("g", ref_g), ("u", ref_u)) if save else ()):
        got = bits(out[k])
        assert_close_bf16(got[:A], ref[:A], f"{k} d={d} h={h}")
        assert np.all(got[A:] == SENT), f"{k}: a row past the packed prefix was written"

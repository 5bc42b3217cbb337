"""Helpers shared by the GPU tests: host <-> device conversion of the bf16 bit
patterns that the oracle and the input generator use, and the tolerance
check of floating-point outputs."""
import numpy as np
import torch

DEV = torch.device("cuda:0")

# Expert outputs: rel 2e-2 / abs 1e-2 (bf16 payloads, fp32 accumulation).
REL_TOL = 2e-2
ABS_TOL = 1e-2


def bf(a, dev=DEV):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def f32(a, dev=DEV):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def i32(a, dev=DEV):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def bits(t):
    """bf16 tensor -> uint16 numpy bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def as64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(
        np.float64)


def assert_close_bf16(got_bits, want_bits, what, rel=REL_TOL, abs_=ABS_TOL):
    """Elementwise |got - want| <= abs + rel |want| (the stated tolerance), and
    the same with the absolute term scaled to the data (|want| RMS), so that
    small-magnitude outputs are not waved through by the absolute term."""
    g = as64(got_bits)
    w = as64(want_bits)
    assert g.shape == w.shape, what
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - w)
    assert np.all(err <= abs_ + rel * np.abs(w)), f"{what}: max err {err.max():.3e}"
    rms = float(np.sqrt(np.mean(w ** 2))) if w.size else 0.0
    bad = err > rel * np.abs(w) + abs_ * rms
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {w.size} outside rel {rel} + "
                           f"{abs_} x rms ({rms:.3e}); max err {err.max():.3e}")

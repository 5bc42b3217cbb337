"""Pins of the oracle's MXFP8 functions (quantizer, dequantizer, MXFP8 experts,
combine of quantized outputs) against facts fixed outside the oracle: the E4M3
code table of the OCP MX specification, round-to-nearest-even ties worked out
by hand, the shared-exponent rule on hand-picked blocks, the rounding error
bound of a 3-bit mantissa, exact arithmetic on inputs the format represents
exactly, and the bf16 combine that a quantized combine must reduce to.
"""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_mx_e4m3_codes.txt")


def _golden_codes():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()[:2]
        if val == "nan":
            v = math.nan
        elif val == "-0":
            v = -0.0
        elif "*" in val:
            a, b = val.split("*")
            v = float(a) * 2.0 ** int(b.split("^")[1])
        elif "^" in val:
            v = 2.0 ** int(val.split("^")[1])
        else:
            v = float(val)
        out.append((int(code, 16), v))
    return out


def _block(values, amax=448.0):
    """A 32-wide block holding `values` after one element of magnitude amax
    (which fixes the block's shared exponent)."""
    b = np.zeros(32)
    b[0] = amax
    b[1:1 + len(values)] = values
    return b


def test_e4m3_code_table():
    """Codes of the specification's table decode to its values (scale byte 127 = 2^0)."""
    for code, v in _golden_codes():
        got = oracle.mx_dequantize(np.array([[code] + [0] * 31], np.uint8),
                                   np.array([[127]], np.uint8))[0, 0]
        if math.isnan(v):
            assert math.isnan(got), hex(code)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(code), got, v)


def test_every_finite_code_quantizes_to_itself():
    """In a block whose largest element is 448 (shared exponent 0) each finite
    E4M3 value is stored as its own code, signs and both zeros included."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.mx_dequantize(codes[:, None].repeat(32, axis=1),
                                np.full((codes.size, 1), 127, np.uint8))[:, 0]
    for c, v in zip(codes, vals):
        q, s = oracle.mx_quantize(_block([v])[None, :])
        assert s[0, 0] == 127
        assert q[0, 1] == c, (hex(c), v, hex(q[0, 1]))


def test_ties_go_to_the_even_code():
    """Midpoints between neighbouring codes round to the code whose mantissa
    LSB is 0; a hair either side rounds to the nearer code.  Worked by hand:
    1 + 1/16 lies between 1.0 (0x38) and 1.125 (0x39) -> 0x38;
    1 + 3/16 between 0x39 and 1.25 (0x3A) -> 0x3A; 7.5 * 2^-9 between the
    largest subnormal 0x07 and the smallest normal 0x08 -> 0x08;
    2^-10 between 0 and the smallest subnormal -> 0 (code 0x00); 432 between
    416 (0x7D) and 448 (0x7E) -> 0x7E; 400 between 384 (0x7C) and 0x7D -> 0x7C."""
    cases = [(1 + 1 / 16, 0x38), (1 + 3 / 16, 0x3A), (7.5 * 2 ** -9, 0x08), (2 ** -10, 0x00),
             (1 + 1 / 16 + 1e-9, 0x39), (1 + 3 / 16 - 1e-9, 0x39), (2 ** -10 + 1e-12, 0x01),
             (-(1 + 1 / 16), 0xB8), (432.0, 0x7E), (432.0 - 1e-9, 0x7D), (400.0, 0x7C)]
    for v, want in cases:
        q, s = oracle.mx_quantize(_block([v])[None, :])
        assert s[0, 0] == 127 and q[0, 1] == want, (v, hex(q[0, 1]), hex(want))


def test_shared_exponent_rule():
    """E = floor(log2 max|v|) - 8, stored as E + 127, clamped to [-127, 127];
    an all-zero block gets byte 0.  Hand cases: max 1.0 -> E = -8 (byte 119)
    and 1.0 is stored as 256 = 0x78; max 448 and 449 and 511.9 -> E = 0;
    512 -> E = 1; 2^-140 -> clamped to -127; 2^130 -> E = 122."""
    cases = [(1.0, 119), (448.0, 127), (449.0, 127), (511.9, 127), (512.0, 128),
             (-512.0, 128), (2.0 ** -140, 0), (2.0 ** 130, 249), (0.0, 0)]
    for amax, byte in cases:
        b = np.zeros(32)
        b[5] = amax
        b[9] = amax / 3
        q, s = oracle.mx_quantize(b[None, :])
        assert s[0, 0] == byte, (amax, s[0, 0], byte)
    q, s = oracle.mx_quantize(np.array([[1.0] + [0.5] * 31]))
    assert q[0, 0] == 0x78 and q[0, 1] == 0x70  # 256 and 128


def test_saturation_past_448():
    """Scaled magnitudes past the largest normal store 448 (not NaN): block
    max 1000 -> E = 1; 1000 / 2 = 500 -> 448 (0x7E); 460 / 2 = 230 -> 224
    (0x76); 470 / 2 = 235 -> 240 (0x77)."""
    q, s = oracle.mx_quantize(np.array([[1000.0, 460.0, 470.0, -1000.0] + [0.0] * 28]))
    assert s[0, 0] == 128
    assert list(q[0, :4]) == [0x7E, 0x76, 0x77, 0xFE]


def test_rounding_error_bound():
    """For every element: the stored value is within half a unit in the last
    place of a 3-bit mantissa (2^(floor(log2|v|) - 4)) in the block's normal
    range, within 2^(E - 10) in its subnormal range, and exactly +-448 * 2^E
    when saturated; the block maximum lands in [256, 448] * 2^E."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 128)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    v[:, 7] *= 1e-4  # elements deep in the subnormal range of their block
    q, s = oracle.mx_quantize(v)
    dq = oracle.mx_dequantize(q, s)
    E = (s.astype(np.int64) - 127).repeat(32, axis=1).astype(np.float64)
    a = np.abs(v)
    scaled = a / np.exp2(E)
    sat = scaled > 448
    normal = (scaled >= 2.0 ** -6) & ~sat
    sub = scaled < 2.0 ** -6
    err = np.abs(dq - v)
    with np.errstate(divide="ignore"):
        ulp_half = np.exp2(np.floor(np.log2(a)) - 4)
    assert np.all(err[normal] <= ulp_half[normal])
    assert np.all(err[sub] <= np.exp2(E[sub] - 10))
    assert np.all(np.abs(dq[sat]) == 448 * np.exp2(E[sat]))
    blk_max = np.abs(dq).reshape(64, 4, 32).max(axis=2)
    Eb = (s.astype(np.int64) - 127).astype(np.float64)
    assert np.all(blk_max >= 256 * np.exp2(Eb)) and np.all(blk_max <= 448 * np.exp2(Eb))
    assert np.all(np.sign(dq[dq != 0]) == np.sign(v[dq != 0]))


def _exact_mx(rng, shape, lo, hi):
    """Values the format holds exactly: 4-significant-bit numbers m * 2^e with
    m in [1, 1.75] (so no element of a block scales past 448) or zero, each
    32-block with its own power-of-two range, so that a block read with its
    neighbour's scale is visibly wrong."""
    m = rng.integers(8, 15, shape) / 8.0 * rng.choice([-1.0, 1.0], shape)
    m[rng.random(shape) < 0.1] = 0.0
    blocks = rng.integers(lo, hi, shape[:-1] + (shape[-1] // 32,))
    return m * np.exp2(np.repeat(blocks, 32, axis=-1) + rng.integers(-3, 1, shape))


def test_mxfp8_experts_on_exact_inputs():
    """With inputs the format represents exactly, the MXFP8 experts equal the
    plain definition evaluated with library matmuls: G = X Wg^T, U = X Wu^T
    (exact in fp64 for these few-bit values), H = silu(G) * U quantized along
    h, Y = deq(H) Wd^T (exact) quantized along d.  Catches a transposed weight,
    a block read with another block's scale, gate and up exchanged, and rows
    written outside the experts' intervals."""
    rng = np.random.default_rng(11)
    N, d, h = 3, 96, 64
    count = np.array([5, 0, 7], np.int32)
    offset = np.array([0, 5, 5, 12], np.int32)
    R = 16
    x = _exact_mx(rng, (R, d), -3, 3)
    wg = _exact_mx(rng, (N, h, d), -8, -4)
    wu = _exact_mx(rng, (N, h, d), -8, -4)
    wd = _exact_mx(rng, (N, d, h), -8, -4)
    xq, xs = oracle.mx_quantize(x)
    assert np.array_equal(oracle.mx_dequantize(xq, xs), x)
    wq = [oracle.mx_quantize(w) for w in (wg, wu, wd)]
    for w, (q, s) in zip((wg, wu, wd), wq):
        assert np.array_equal(oracle.mx_dequantize(q, s), w)
    hq, hs, yq, ys = oracle.expert_ffn_mx(xq, xs, count, offset, *wq, fill=0xA5)
    for e in range(N):
        for i in range(count[e]):
            r = offset[e] + i
            g = wg[e] @ x[r]
            u = wu[e] @ x[r]
            a = g / (1.0 + np.exp(-g)) * u
            aq, as_ = oracle.mx_quantize(a[None, :])
            assert np.array_equal(hq[r], aq[0]) and np.array_equal(hs[r], as_[0])
            y = wd[e] @ oracle.mx_dequantize(aq, as_)[0]
            y_q, y_s = oracle.mx_quantize(y[None, :])
            assert np.array_equal(yq[r], y_q[0]) and np.array_equal(ys[r], y_s[0])
    assert np.all(hq[12:] == 0xA5) and np.all(yq[12:] == 0xA5)
    # the swapped-role SwiGLU differs on these inputs
    g = wg[0] @ x[0]; u = wu[0] @ x[0]
    swapped, _ = oracle.mx_quantize((u / (1.0 + np.exp(-u)) * g)[None, :])
    assert not np.array_equal(swapped[0], hq[0])


def test_combine_of_quantized_rows_is_the_bf16_combine_of_their_values():
    """Dequantized E4M3 values are exact in bf16, so the quantized combine
    must equal, bit for bit, the bf16 combine (pinned on its own) fed with
    those values; with one route and gate 1 it is the dequantized row."""
    rng = np.random.default_rng(5)
    T, K, R, d = 9, 3, 20, 64
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    yq = rng.choice(codes, (R, d)).astype(np.uint8)
    ys = rng.integers(120, 135, (R, d // 32)).astype(np.uint8)
    rr = rng.integers(-1, R, (T, K)).astype(np.int32)
    gate = rng.random((T, K)).astype(np.float32)
    y_bf16 = oracle.bf16_from_f64(oracle.mx_dequantize(yq, ys))
    assert np.array_equal(oracle.bf16_to_f32(y_bf16), oracle.mx_dequantize(yq, ys).astype(np.float32))
    assert np.array_equal(oracle.combine_mx(yq, ys, rr, gate), oracle.combine(y_bf16, rr, gate))
    one = oracle.combine_mx(yq, ys, np.arange(4, dtype=np.int32)[:, None], np.ones((4, 1), np.float32))
    # the sum starts from +0, so a -0 element comes out as +0: compare values
    assert np.array_equal(oracle.bf16_to_f32(one), oracle.bf16_to_f32(y_bf16[:4]))


def test_layer_forward_mx_close_to_bf16_layer():
    """The MXFP8 layer stays within MXFP8's error of the bf16 layer on the
    same inputs (it quantizes activations three times and weights once)."""
    rng = np.random.default_rng(2)
    T, d, N, K, h, cap = 24, 64, 4, 2, 64, 12
    x = oracle.bf16_from_f64(rng.standard_normal((T, d)))
    w_r = (rng.standard_normal((N, d)) * 0.2).astype(np.float32)
    wg = oracle.bf16_from_f64(rng.standard_normal((N, h, d)) * 0.15)
    wu = oracle.bf16_from_f64(rng.standard_normal((N, h, d)) * 0.15)
    wd = oracle.bf16_from_f64(rng.standard_normal((N, d, h)) * 0.15)
    ref = oracle.layer_forward(x, w_r, None, wg, wu, wd, K, cap)
    mx = oracle.layer_forward_mx(x, w_r, None, wg, wu, wd, K, cap)
    assert np.array_equal(ref["route_row"], mx["route_row"])
    a = oracle.bf16_to_f32(ref["y"]).astype(np.float64)
    b = oracle.bf16_to_f32(mx["y"]).astype(np.float64)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 0.12, rel

"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it cannot agree with by
construction: the worked example printed in the report, brute force on tiny
inputs, closed forms, invariants the pages state, special cases that reduce to
a textbook routine, adjoint identities and finite differences.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fig15_16_worked_example.txt")


def load_worked_example():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p = line.split()
            rows.append(dict(tok=p[0], src=int(p[1]), idx=[int(p[2]), int(p[3])],
                             w=[float(p[4]), float(p[5])], rank=[int(p[6]), int(p[7])],
                             row=[int(p[8]), int(p[9])]))
    return rows


# ------------------------------------------------------------ worked example --

def test_worked_example_router_output():
    """Figure 15: logits ln(w) for the two chosen experts reproduce the printed
    indices (in printed order, larger weight first) and weights."""
    ex = load_worked_example()
    logits = np.full((len(ex), 4), -30.0, dtype=np.float32)
    for t, r in enumerate(ex):
        for k in range(2):
            logits[t, r["idx"][k]] = math.log(r["w"][k])
    idx, gate = oracle.topk_gates(logits, 2)
    assert idx.tolist() == [r["idx"] for r in ex]
    np.testing.assert_allclose(gate, np.array([r["w"] for r in ex]), rtol=1e-6)


def test_worked_example_route_map_two_sources():
    """Figure 16: each source rank applies the capacity decision to its own 5
    tokens (cap 4), then accepted routes are packed per destination expert in
    token order.  Composing the oracle's per-source decisions that way
    reproduces every printed (rank, row) pair, including the E->1 drop."""
    ex = load_worked_example()
    N, K, cap = 4, 2, 4
    assert cap == math.ceil(1.25 * 5 * 2 / 4)
    per_src = {}
    for s in (0, 1):
        toks = [r for r in ex if r["src"] == s]
        idx = np.array([r["idx"] for r in toks], dtype=np.int32)
        row, count, offset, demand = oracle.route_slots(idx, N, cap)
        per_src[s] = (toks, idx, row, count, offset)
    expert_rank = {0: 0, 1: 0, 2: 1, 3: 1}
    total = per_src[0][3] + per_src[1][3]
    for s in (0, 1):
        toks, idx, row, count, offset = per_src[s]
        for t, r in enumerate(toks):
            for k in range(K):
                e = int(idx[t, k])
                if row[t, k] < 0:
                    assert (r["rank"][k], r["row"][k]) == (-1, -1), (r["tok"], k)
                    continue
                slot = int(row[t, k]) - int(offset[e])
                first = min(x for x in expert_rank if expert_rank[x] == expert_rank[e])
                base = int(sum(total[first:e]))
                before = int(per_src[0][3][e]) if s == 1 else 0
                assert expert_rank[e] == r["rank"][k]
                assert base + before + slot == r["row"][k], (r["tok"], k)
    # rank 0 holds the page's 12 rows
    assert int(total[0] + total[1]) == 12


def test_worked_example_single_buffer_no_drop():
    """One buffer for all 10 tokens with room for everything (cap 8): expert 0
    keeps the printed rows 0..4, expert 1 the printed rows of A-D; the three
    routes the page places after the dropped E->1 move up by one; experts 2,3
    keep their printed rows shifted by the offset of expert 2."""
    ex = load_worked_example()
    idx = np.array([r["idx"] for r in ex], dtype=np.int32)
    row, count, offset, demand = oracle.route_slots(idx, 4, 8)
    assert count.tolist() == [5, 8, 4, 3] and offset.tolist() == [0, 5, 13, 17, 20]
    for t, r in enumerate(ex):
        for k in range(2):
            e = r["idx"][k]
            if r["tok"] == "E" and e == 1:
                assert row[t, k] == 9
                continue
            want = r["row"][k]
            if e == 1 and r["tok"] in "GIJ":
                want += 1
            if e >= 2:
                want += 13
            assert row[t, k] == want, (r["tok"], k)


# ------------------------------------------------------------------ routing --

def _brute_topk(logits, K):
    T, N = logits.shape
    idx = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        key = np.where(np.isnan(logits[t]), -np.inf, logits[t]).astype(np.float64)
        order = sorted(range(N), key=lambda e: (-key[e], e))
        idx[t] = order[:K]
    return idx


@pytest.mark.parametrize("T,N,K,levels", [(64, 8, 2, None), (200, 16, 4, 3), (50, 64, 8, 2),
                                          (33, 5, 5, None)])
def test_topk_matches_full_sort(T, N, K, levels):
    """Top-K by selection equals the first K of a full sort by (logit desc,
    index asc), including many exact ties."""
    rng = np.random.default_rng(T * N + K)
    logits = rng.standard_normal((T, N)).astype(np.float32)
    if levels:
        logits = np.round(logits * levels / 3).astype(np.float32)
    logits[0, 0] = np.nan
    idx, gate = oracle.topk_gates(logits, K)
    np.testing.assert_array_equal(idx, _brute_topk(logits, K))


def test_gates_closed_forms():
    """Gates: equal to a full softmax over all N renormalised over the chosen K
    (fp64); sum to one; K = 1 gives 1; K = 2 gives the logistic of the gap."""
    rng = np.random.default_rng(7)
    T, N, K = 300, 32, 4
    logits = (rng.standard_normal((T, N)) * 3).astype(np.float32)
    idx, gate = oracle.topk_gates(logits, K)
    z = logits.astype(np.float64)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gate, sel / sel.sum(axis=1, keepdims=True), rtol=2e-7, atol=1e-30)
    np.testing.assert_allclose(gate.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(gate, axis=1) <= 0)
    _, g1 = oracle.topk_gates(logits, 1)
    assert np.all(g1 == 1.0)
    i2, g2 = oracle.topk_gates(logits, 2)
    gap = np.take_along_axis(z, i2.astype(np.int64), 1)
    np.testing.assert_allclose(g2[:, 0], 1 / (1 + np.exp(gap[:, 1] - gap[:, 0])), rtol=1e-6)


def test_gates_degenerate_logits():
    """All-equal logits (including all -inf) select experts 0..K-1 with equal
    gates; a single +inf logit takes the whole weight."""
    L = np.full((3, 6), -np.inf, dtype=np.float32)
    L[1] = 2.5
    L[2] = 0.0
    L[2, 4] = np.inf
    idx, gate = oracle.topk_gates(L, 3)
    assert idx[0].tolist() == [0, 1, 2] and idx[1].tolist() == [0, 1, 2]
    np.testing.assert_allclose(gate[:2], 1 / 3, rtol=1e-7)
    assert idx[2, 0] == 4 and gate[2].tolist() == [1.0, 0.0, 0.0]


def test_logits_exact_on_integers_and_error_bound():
    """Small-integer inputs make every product and partial sum exact, so the
    fp32 chain equals the integer dot product; for random inputs the chain is
    within the standard forward-error bound d*u*sum|x w| of the exact value."""
    rng = np.random.default_rng(3)
    T, d, N = 20, 96, 12
    xi = rng.integers(-8, 9, size=(T, d)).astype(np.float32)
    wi = rng.integers(-8, 9, size=(N, d)).astype(np.float32)
    bias = rng.integers(-4, 5, size=N).astype(np.float32)
    got = oracle.router_logits(synth.f32_to_bf16_bits(xi), wi, bias)
    want = xi.astype(np.int64) @ wi.astype(np.int64).T + bias.astype(np.int64)
    np.testing.assert_array_equal(got, want.astype(np.float32))

    x = synth.normal_bf16(11, (T, 512))
    w = synth.normal_f32(12, (N, 512), 0.02)
    got = oracle.router_logits(x, w).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    exact = np.array([[math.fsum(xf[t] * w[e].astype(np.float64)) for e in range(N)]
                      for t in range(T)])
    bound = 512 * 2.0 ** -24 * (np.abs(xf) @ np.abs(w.astype(np.float64)).T)
    assert np.all(np.abs(got - exact) <= bound)

    # d = 2000: within the recursive-summation bound d u sum|x w| (each fused
    # multiply-add rounds once, so d roundings in all)
    x = synth.normal_bf16(13, (T, 2000))
    w = synth.normal_f32(14, (N, 2000), 0.02)
    got = oracle.router_logits(x, w).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    exact = np.array([[math.fsum(xf[t] * w[e].astype(np.float64)) for e in range(N)]
                      for t in range(T)])
    bound = 2000 * 2.0 ** -24 * (np.abs(xf) @ np.abs(w.astype(np.float64)).T)
    assert np.all(np.abs(got - exact) <= bound)


def test_logits_left_to_right_order():
    """The logit is the dot product summed left to right from 0 (j = 0 first).
    With the product 2^24 first and 1023 unit products after it, every +1 meets
    2^24, lies exactly halfway between two fp32 neighbours and rounds back to
    the even 2^24, so the sum stays 2^24; a sum cut into blocks (say of 512)
    would keep the later blocks' ones exactly and end above 2^24.  The same
    products in the reverse order sum exactly to 1023 before meeting 2^24,
    giving 2^24 + 1023, which rounds to 2^24 + 1024."""
    d = 1024
    x = np.ones((2, d), np.float32)
    w = np.ones((1, d), np.float32)
    x[0, 0] = 4096.0
    w[0, 0] = 4096.0
    x[1, d - 1] = 4096.0  # token 1: the large product comes last ...
    w2 = np.ones((1, d), np.float32)
    w2[0, d - 1] = 4096.0
    got = oracle.router_logits(synth.f32_to_bf16_bits(x[:1]), w)
    assert got[0, 0] == np.float32(2.0 ** 24)
    got = oracle.router_logits(synth.f32_to_bf16_bits(x[1:]), w2)
    assert got[0, 0] == np.float32(2.0 ** 24 + 1024)


def test_logits_fused_multiply_add():
    """Each step is one fused multiply-add (a single rounding of x*w + acc):
    x = 1 + 2^-7 (exact in bf16) times w = 1 + 2^-23 is 1 + 2^-7 + 2^-23 +
    2^-30, whose fp32 rounding drops 2^-30.  Adding -(1 + 2^-7 + 2^-23) as the
    second product (x = -1, w = 1 + 2^-7 + 2^-23) therefore leaves the exact
    2^-30 after a fused step, where a separately rounded product would leave 0.
    The chain runs the small product first so that the large one is the fused
    step: acc = fma(x1, w1, fma(x0, w0, 0)) = fma(x1, w1, rn(x0 w0))."""
    x = synth.f32_to_bf16_bits(np.array([[-1.0, 1.0 + 2.0 ** -7]], np.float32))
    w = np.array([[1.0 + 2.0 ** -7 + 2.0 ** -23, 1.0 + 2.0 ** -23]], np.float32)
    got = oracle.router_logits(x, w)
    assert got[0, 0] == np.float32(2.0 ** -30)


def _brute_slots(idx, N, cap):
    T, K = idx.shape
    demand = np.bincount(idx.ravel(), minlength=N)
    count = np.minimum(demand, cap)
    offset = np.concatenate([[0], np.cumsum(count)])
    row = np.empty_like(idx)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            s = int(np.sum(idx[:t] == e))   # earlier tokens that chose e
            row[t, k] = offset[e] + s if s < cap else -1
    return row, count, offset, demand


@pytest.mark.parametrize("T,N,K,cap", [(40, 4, 2, 100), (40, 4, 2, 7), (120, 16, 4, 12),
                                       (64, 8, 8, 30), (10, 3, 1, 0), (0, 4, 2, 5)])
def test_slots_brute_force(T, N, K, cap):
    """Slots by an O(T^2) count of earlier tokens per expert."""
    idx = synth.gen_topk_idx(T + N, T, N, K) if T else np.zeros((0, K), np.int32)
    got = oracle.route_slots(idx, N, cap)
    want = _brute_slots(idx, N, cap)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def _check_invariants(idx, row, count, offset, demand, cap):
    T, K = idx.shape
    N = count.size
    assert np.all(count <= cap) and np.all(count == np.minimum(demand, cap))
    assert offset[0] == 0 and offset[-1] == count.sum() <= T * K
    kept = row >= 0
    # every kept route has its own row, inside its expert's interval
    assert len(set(row[kept].tolist())) == int(kept.sum()) == int(offset[-1])
    e = idx[kept]
    assert np.all(row[kept] >= offset[e]) and np.all(row[kept] < offset[e] + count[e])
    # token-stable: rows of one expert increase with the token index
    for ex in range(N):
        r = row[(idx == ex) & kept]
        assert np.all(np.diff(r) > 0)
    # drops are exactly the routes past capacity
    assert int((~kept).sum()) == int((demand - count).sum())


@pytest.mark.parametrize("name", ["tiny", "fine_zipf_small"])
def test_route_invariants(name):
    if name == "tiny":
        cfg = synth.CONFIGS["tiny"]
    else:
        cfg = synth.CONFIGS["fine_zipf"].with_(T=512, d=256)
    x = synth.gen_x(cfg)
    r = oracle.route(x, synth.gen_router(cfg), synth.gen_bias(cfg), cfg.K, cfg.cap)
    _check_invariants(r["topk_idx"], r["route_row"], r["expert_count"], r["expert_offset"],
                      r["expert_demand"], cfg.cap)
    if name != "tiny":
        assert (r["expert_demand"] > cfg.cap).any()   # the Zipf offsets force drops


# ----------------------------------------------------------------- movement --

def _route_case(seed, T, N, K, cap):
    idx = synth.gen_topk_idx(seed, T, N, K)
    row, count, offset, demand = oracle.route_slots(idx, N, cap)
    return idx, row, count, offset


def test_dispatch_places_each_kept_route_once():
    T, N, K, cap, d = 90, 6, 3, 40, 24
    idx, row, count, offset = _route_case(5, T, N, K, cap)
    x = synth.gen_bf16(5, (T, d), "x")
    xd = oracle.dispatch(x, row, N * cap, fill=0xFFFF)
    for t in range(T):
        for k in range(K):
            if row[t, k] >= 0:
                assert np.array_equal(xd[row[t, k]], x[t])
    assert np.all(xd[offset[-1]:] == 0xFFFF)   # tail untouched


@pytest.mark.parametrize("cap", [100, 9])
def test_identity_experts_combine_of_dispatch(cap):
    """With y_disp = x_disp (identity experts), combine(dispatch(x)) is the sum
    of the kept gates times x (within one bf16 rounding); without drops it is x."""
    T, N, K, d = 120, 8, 2, 40
    rng = np.random.default_rng(cap)
    logits = rng.standard_normal((T, N)).astype(np.float32)
    idx, gate = oracle.topk_gates(logits, K)
    row, count, offset, demand = oracle.route_slots(idx, N, cap)
    x = synth.gen_bf16(9, (T, d), "x")
    y = oracle.combine(oracle.dispatch(x, row, N * cap), row, gate)
    kept_g = np.where(row >= 0, gate, 0).astype(np.float64).sum(axis=1)
    want = kept_g[:, None] * oracle.bf16_to_f32(x).astype(np.float64)
    got = oracle.bf16_to_f32(y).astype(np.float64)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)
    if cap == 100:
        assert (row >= 0).all()
        np.testing.assert_allclose(got, oracle.bf16_to_f32(x), rtol=2 ** -8)
    else:
        assert (row < 0).any()


def test_combine_reads_no_tail_and_zero_for_dropped():
    """Unwritten tail rows (poisoned with NaN) never reach the output; a token
    whose routes are all dropped combines to exactly zero."""
    T, N, K, d, cap = 64, 4, 2, 16, 10
    idx, row, count, offset = _route_case(2, T, N, K, cap)
    gate = synth.gen_gates(2, T, K)
    yd = np.full((N * cap, d), 0x7FC0, dtype=np.uint16)   # NaN everywhere
    yd[: offset[-1]] = synth.gen_bf16(3, (int(offset[-1]), d), "y")
    y = oracle.combine(yd, row, gate)
    assert np.all(np.isfinite(oracle.bf16_to_f32(y)))
    dead = np.all(row < 0, axis=1)
    assert dead.any() and np.all(y[dead] == 0)


def test_adjoint_identities():
    """Table 8: backward movements are the adjoints of the forward ones:
    <dispatch(x), u> = <x, dispatch_bwd(u)> and <combine(v), w> = <v, combine_bwd(w)>,
    over the valid rows (fp64 inner products of the exact values)."""
    T, N, K, d, cap = 80, 5, 3, 16, 30
    idx, row, count, offset = _route_case(8, T, N, K, cap)
    gate = synth.gen_gates(8, T, K)
    A = int(offset[-1])
    R = N * cap
    x = synth.gen_bf16(1, (T, d), "x")
    u = synth.gen_bf16(1, (R, d), "u")
    f = lambda b: oracle.bf16_to_f32(b).astype(np.float64)
    lhs = np.sum(f(oracle.dispatch(x, row, R))[:A] * f(u)[:A])
    rhs = np.sum(f(x) * oracle.dispatch_bwd(u, row, T).astype(np.float64))
    assert abs(lhs - rhs) <= 1e-5 * (np.sum(np.abs(f(x))) + 1)
    # combine adjoint: compare with an fp64 restatement free of the bf16 output rounding
    v = synth.gen_bf16(2, (R, d), "v")
    w = synth.gen_bf16(3, (T, d), "w")
    dv, dg = oracle.combine_bwd(w, v, row, gate)
    lhs = np.sum(f(oracle.combine(v, row, gate)) * f(w))
    rhs = np.sum(f(v)[:A] * f(dv)[:A])
    scale = np.sum(np.abs(f(v)[:A])) * 4
    assert abs(lhs - rhs) <= 1e-2 * scale / np.sqrt(A * d)


def test_router_weight_gradient_finite_difference():
    """dgate = d<combine(v), dy>/dgate, checked by central differences in fp64."""
    T, N, K, d, cap = 12, 4, 2, 8, 12
    idx, row, count, offset = _route_case(4, T, N, K, cap)
    gate = synth.gen_gates(4, T, K)
    v = synth.gen_bf16(4, (N * cap, d), "v")
    dy = synth.gen_bf16(5, (T, d), "dy")
    _, dg = oracle.combine_bwd(dy, v, row, gate)
    f = lambda b: oracle.bf16_to_f32(b).astype(np.float64)

    def L(gv):
        out = np.zeros((T, d))
        for t in range(T):
            for k in range(K):
                if row[t, k] >= 0:
                    out[t] += gv[t, k] * f(v)[row[t, k]]
        return np.sum(out * f(dy))

    g64 = gate.astype(np.float64)
    for t, k in [(0, 0), (3, 1), (11, 0)]:
        e = np.zeros_like(g64)
        e[t, k] = 1e-6
        fd = (L(g64 + e) - L(g64 - e)) / 2e-6
        assert abs(fd - dg[t, k]) <= 1e-4 * (1 + abs(fd))


# ------------------------------------------------------------------ experts --

def _silu(z):
    return z / (1 + np.exp(-z))


def test_ffn_dense_special_case_is_textbook_swiglu():
    """One expert taking every token (N=1, K=1, no drops) is a dense bias-free
    SwiGLU MLP: Y = (silu(X Wg^T) * (X Wu^T)) Wd^T, evaluated with numpy matmul."""
    rng = np.random.default_rng(0)
    n, d, h = 17, 24, 40
    x = rng.standard_normal((n, d))
    wg, wu = rng.standard_normal((h, d)) * 0.2, rng.standard_normal((h, d)) * 0.2
    wd = rng.standard_normal((d, h)) * 0.2
    g, u, a, y = oracle.ffn_fwd_f64(x, wg, wu, wd)
    np.testing.assert_allclose(y, (_silu(x @ wg.T) * (x @ wu.T)) @ wd.T, rtol=1e-12, atol=1e-12)


def test_ffn_permutation_weights_closed_form():
    """Permutation weights make every reduction a single term, so each output is
    a closed form of one input: catches transposed operands and index slips."""
    rng = np.random.default_rng(1)
    d, h = 6, 6
    pg, pu, pd = rng.permutation(h), rng.permutation(h), rng.permutation(d)
    wg = np.zeros((h, d)); wg[np.arange(h), pg] = 1.5
    wu = np.zeros((h, d)); wu[np.arange(h), pu] = -0.5
    wd = np.zeros((d, h)); wd[np.arange(d), pd] = 2.0
    x = rng.standard_normal((4, d))
    _, _, _, y = oracle.ffn_fwd_f64(x, wg, wu, wd)
    for r in range(4):
        for o in range(d):
            i = pd[o]
            z = 1.5 * x[r, pg[i]]
            want = 2.0 * (z / (1 + math.exp(-z))) * (-0.5 * x[r, pu[i]])
            assert abs(y[r, o] - want) <= 1e-14


def test_silu_values():
    """Identity weights reduce the expert to y_i = silu(x_i) * x_i; compare with
    the logistic function evaluated by hand."""
    xs = [0.0, 1.0, -1.0, 30.0, -30.0, 0.5]
    x = np.array([xs])
    I = np.eye(len(xs))
    _, _, a, y = oracle.ffn_fwd_f64(x, I, I, I)
    want = [v * v / (1 + math.exp(-v)) for v in xs]
    np.testing.assert_allclose(y[0], want, rtol=1e-14, atol=0)
    assert want[1] == 1 / (1 + math.exp(-1)) and y[0, 0] == 0.0


def test_ffn_backward_finite_difference():
    """The fp64 expert backward equals central differences of the fp64 forward
    for L = <y, dy> with respect to x and all three weights."""
    rng = np.random.default_rng(2)
    n, d, h = 5, 7, 9
    x = rng.standard_normal((n, d))
    wg, wu, wd = (rng.standard_normal((h, d)) * 0.4, rng.standard_normal((h, d)) * 0.4,
                  rng.standard_normal((d, h)) * 0.4)
    dy = rng.standard_normal((n, d))
    g, u, a, y = oracle.ffn_fwd_f64(x, wg, wu, wd)
    dx, dwg, dwu, dwd = oracle.ffn_bwd_f64(x, g, u, a, dy, wg, wu, wd)

    def L(x_, wg_, wu_, wd_):
        return float(np.sum(oracle.ffn_fwd_f64(x_, wg_, wu_, wd_)[3] * dy))

    eps = 1e-6
    for name, arr, grad in [("x", x, dx), ("wg", wg, dwg), ("wu", wu, dwu), ("wd", wd, dwd)]:
        for pos in [(0, 0), (arr.shape[0] - 1, arr.shape[1] - 1), (1, 2)]:
            args = {"x": x, "wg": wg, "wu": wu, "wd": wd}
            p, m = {k: v.copy() for k, v in args.items()}, {k: v.copy() for k, v in args.items()}
            p[name][pos] += eps
            m[name][pos] -= eps
            fd = (L(p["x"], p["wg"], p["wu"], p["wd"]) - L(m["x"], m["wg"], m["wu"], m["wd"])) / (2 * eps)
            assert abs(fd - grad[pos]) <= 1e-6 * (1 + abs(fd)), (name, pos)


def test_grouped_ffn_equals_per_token_direct_evaluation():
    """The pipeline's y (route -> dispatch -> grouped experts -> combine) equals
    the per-token direct sum over the kept routes of g_k * FFN_{e_k}(x_t) in
    fp64, which uses no route map, slots or packing; dropped routes add zero."""
    cfg = synth.CONFIGS["tiny"].with_(T=96, d=32, h=48, N=6, K=2, cf_num=3, cf_den=4)
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg) * 20
    wg, wu, wd = (synth.normal_bf16(s, shp, 0.2) for s, shp in
                  [(1, (cfg.N, cfg.h, cfg.d)), (2, (cfg.N, cfg.h, cfg.d)), (3, (cfg.N, cfg.d, cfg.h))])
    out = oracle.layer_forward(x, wr, None, wg, wu, wd, cfg.K, cfg.cap)
    f = oracle.bf16_to_f32
    xf = f(x).astype(np.float64)
    assert (out["route_row"] < 0).any()
    direct = np.zeros((cfg.T, cfg.d))
    for t in range(cfg.T):
        for k in range(cfg.K):
            if out["route_row"][t, k] < 0:
                continue
            e = out["topk_idx"][t, k]
            _, _, _, y = oracle.ffn_fwd_f64(xf[t:t + 1], f(wg[e]), f(wu[e]), f(wd[e]))
            direct[t] += out["topk_gate"][t, k] * y[0]
    got = f(out["y"]).astype(np.float64)
    rms = np.sqrt(np.mean(direct ** 2))
    assert np.all(np.abs(got - direct) <= 2e-2 * np.abs(direct) + 1e-2 * rms)


def test_expert_additivity():
    """AWS Neuron EP page, "Why a Single All-Reduce/Reduce-Scatter Works":
    summing the outputs of disjoint expert groups (others' weights zeroed, so
    their FFN is exactly 0) gives the full output."""
    cfg = synth.CONFIGS["tiny"].with_(T=64, d=32, h=32, N=4, K=2)
    x = synth.gen_x(cfg)
    wr = synth.gen_router(cfg)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    full = oracle.layer_forward(x, wr, None, wg, wu, wd, cfg.K, cfg.cap)
    f = oracle.bf16_to_f32
    acc = np.zeros((cfg.T, cfg.d))
    mag = np.zeros((cfg.T, cfg.d))
    for grp in ([0, 1], [2, 3]):
        mask = np.zeros(cfg.N, bool); mask[grp] = True
        z = lambda w: np.where(mask[:, None, None], w, 0).astype(np.uint16)
        part = oracle.layer_forward(x, wr, None, z(wg), z(wu), z(wd), cfg.K, cfg.cap)
        acc += f(part["y"]).astype(np.float64)
        mag += np.abs(f(part["y"]).astype(np.float64))
    ref = f(full["y"]).astype(np.float64)
    # each bf16 output carries at most half an ulp (2^-9 relative) of rounding
    assert np.all(np.abs(acc - ref) <= 2 ** -8 * (mag + np.abs(ref)))


def test_grouped_ffn_rows_and_tails():
    """expert_ffn touches only rows [offset[e], offset[e]+count[e]); the
    row-list variant gives the same rows; saved G/U are the pre-activations."""
    cfg = synth.CONFIGS["tiny"].with_(T=40, d=16, h=24, N=4, K=2, cf_num=1, cf_den=2)
    x = synth.gen_x(cfg)
    r = oracle.route(x, synth.gen_router(cfg), None, cfg.K, cfg.cap)
    wg, wu, wd = synth.gen_expert_weights(cfg)
    xd = oracle.dispatch(x, r["route_row"], cfg.R, fill=0x7FC0)
    h, gs, us, y = oracle.expert_ffn(xd, r["expert_count"], r["expert_offset"], wg, wu, wd,
                                     save=True, fill=0x1234)
    A = int(r["expert_offset"][-1])
    assert np.all(h[A:] == 0x1234) and np.all(y[A:] == 0x1234)
    assert np.all(np.isfinite(oracle.bf16_to_f32(y[:A])))
    rows = np.arange(A, dtype=np.int32)
    ex = np.searchsorted(r["expert_offset"], rows, side="right").astype(np.int32) - 1
    h2, g2, u2, y2 = oracle.expert_ffn_rows(rows, ex, xd, wg, wu, wd, save=True)
    assert np.array_equal(h2, h[:A]) and np.array_equal(y2, y[:A]) and np.array_equal(g2, gs[:A])
    f = oracle.bf16_to_f32
    for i in [0, A // 2, A - 1]:
        e = ex[i]
        g, u, a, yy = oracle.ffn_fwd_f64(f(xd[i:i + 1]), f(wg[e]), f(wu[e]), f(wd[e]))
        assert np.array_equal(gs[i], oracle.bf16_from_f64(g[0]))
        assert np.array_equal(us[i], oracle.bf16_from_f64(u[0]))


# ------------------------------------------------------------------- bf16 --

def test_bf16_rounding():
    """Round-to-nearest-even at the bf16 grid: ties go to the even neighbour;
    fp64 values that are fp32-exact round like the independent fp32 rounding
    of the input generator; overflow goes to inf; subnormals are kept."""
    one = 1.0
    cases = {one + 2 ** -8: 0x3F80, one + 3 * 2 ** -8: 0x3F82, one + 2 ** -8 + 2 ** -30: 0x3F81,
             -one - 2 ** -8: 0xBF80, 2.0 ** 130: 0x7F80, 3.4e38: 0x7F80, 2.0 ** -133: 0x0001,
             2.0 ** -135: 0x0000, 0.0: 0x0000}
    got = oracle.bf16_from_f64(np.array(list(cases.keys())))
    assert got.tolist() == list(cases.values())
    v = synth.normal_f32(99, (10000,), 3.0)
    assert np.array_equal(oracle.bf16_from_f64(v.astype(np.float64)), synth.f32_to_bf16_bits(v))
    assert np.array_equal(oracle.bf16_from_f32(v), synth.f32_to_bf16_bits(v))


def test_expert_backward_grouped_matches_core_and_weight_grad_fd():
    """The grouped bf16 backward applies the fp64 core expert by expert over the
    valid rows only; experts without rows get zero weight gradient."""
    cfg = synth.CONFIGS["tiny"].with_(T=24, d=16, h=8, N=4, K=1, cf_num=1, cf_den=1)
    idx = np.array([[0]] * 10 + [[2]] * 14, dtype=np.int32)
    row, count, offset, demand = oracle.route_slots(idx, cfg.N, 14)
    R = cfg.N * 14
    x = synth.gen_bf16(1, (R, cfg.d), "xd")
    wg, wu, wd = synth.gen_expert_weights(cfg.with_(seed=5))
    h, gs, us, y = oracle.expert_ffn(x, count, offset, wg, wu, wd, save=True)
    dyd = synth.gen_bf16(2, (R, cfg.d), "dyd")
    dx, dwg, dwu, dwd = oracle.expert_ffn_bwd(count, offset, x, gs, us, h, dyd, wg, wu, wd,
                                              fill=0x4242)
    assert np.all(dwg[1] == 0) and np.all(dwd[3] == 0)
    assert np.all(dx[int(offset[-1]):] == 0x4242)
    f = lambda b: oracle.bf16_to_f32(b).astype(np.float64)
    e, r0, n = 2, int(offset[2]), int(count[2])
    cdx, cdwg, cdwu, cdwd = oracle.ffn_bwd_f64(f(x[r0:r0 + n]), f(gs[r0:r0 + n]), f(us[r0:r0 + n]),
                                               f(h[r0:r0 + n]), f(dyd[r0:r0 + n]), f(wg[e]),
                                               f(wu[e]), f(wd[e]), round_dgu=True)
    assert np.array_equal(dx[r0:r0 + n], oracle.bf16_from_f64(cdx))
    np.testing.assert_allclose(dwg[e], cdwg.astype(np.float32), rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(dwd[e], cdwd.astype(np.float32), rtol=1e-6, atol=1e-12)


def test_expert_backward_bf16_intermediates_stay_within_rounding():
    """With dG, dU rounded to bf16 the backward differs from the unrounded fp64
    one by no more than that rounding (half an ulp, 2^-9 relative, per term);
    dW_down, which never sees dG or dU, is unchanged."""
    rng = np.random.default_rng(4)
    n, d, h = 6, 16, 12
    x = rng.standard_normal((n, d))
    wg, wu, wd = (rng.standard_normal((h, d)) * 0.3, rng.standard_normal((h, d)) * 0.3,
                  rng.standard_normal((d, h)) * 0.3)
    dy = rng.standard_normal((n, d))
    g, u, a, y = oracle.ffn_fwd_f64(x, wg, wu, wd)
    exact = oracle.ffn_bwd_f64(x, g, u, a, dy, wg, wu, wd)
    rounded = oracle.ffn_bwd_f64(x, g, u, a, dy, wg, wu, wd, round_dgu=True)
    assert np.array_equal(exact[3], rounded[3])
    # the same products evaluated by hand from the rounded intermediates
    s = 1 / (1 + np.exp(-g))
    da = dy @ wd
    du = da * g * s
    dg = da * u * s * (1 + g * (1 - s))
    q = lambda v: oracle.bf16_to_f32(oracle.bf16_from_f64(v)).astype(np.float64)
    for got, want in [(rounded[0], q(dg) @ wg + q(du) @ wu), (rounded[1], q(dg).T @ x),
                      (rounded[2], q(du).T @ x)]:
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    for e_, r_ in zip(exact[:3], rounded[:3]):
        assert np.max(np.abs(e_ - r_)) <= 2.0 ** -8 * np.max(np.abs(e_)) * max(d, h)


def test_router_backward_finite_difference():
    """Router backward against central differences of L = sum_{t,k} c[t,k] g[t,k]
    with g the softmax over the chosen logits of x W_r^T + bias (selection held
    fixed; the perturbation is too small to change it)."""
    rng = np.random.default_rng(11)
    T, d, N, K = 6, 8, 5, 3
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    w = rng.standard_normal((N, d)) * 0.5
    b = rng.standard_normal(N) * 0.3
    c = rng.standard_normal((T, K))

    def gates(xv, wv, bv):
        l = xv @ wv.T + bv
        idx = np.argsort(-l, axis=1, kind="stable")[:, :K]
        sel = np.take_along_axis(l, idx, 1)
        e = np.exp(sel - sel[:, :1])
        return idx, e / e.sum(1, keepdims=True)

    idx, g = gates(xf, w, b)
    L = lambda xv, wv, bv: float(np.sum(c * gates(xv, wv, bv)[1]))
    dl, dx, dw, db = oracle.router_bwd(x, w.astype(np.float32), idx.astype(np.int32),
                                       g.astype(np.float32), c.astype(np.float32))
    # the oracle reads W_r as fp32: evaluate with the same rounded weights
    w = w.astype(np.float32).astype(np.float64)
    eps = 1e-6
    for (t, j) in [(0, 0), (3, 5), (5, 7)]:
        e_ = np.zeros_like(xf); e_[t, j] = eps
        fd = (L(xf + e_, w, b) - L(xf - e_, w, b)) / (2 * eps)
        assert abs(fd - dx[t, j]) <= 1e-4 * (1 + abs(fd))
    for (ee, j) in [(0, 1), (2, 6), (4, 0)]:
        e_ = np.zeros_like(w); e_[ee, j] = eps
        fd = (L(xf, w + e_, b) - L(xf, w - e_, b)) / (2 * eps)
        assert abs(fd - dw[ee, j]) <= 1e-4 * (1 + abs(fd))
    for ee in range(N):
        e_ = np.zeros_like(b); e_[ee] = eps
        fd = (L(xf, w, b + e_) - L(xf, w, b - e_)) / (2 * eps)
        assert abs(fd - db[ee]) <= 1e-4 * (1 + abs(fd))


def test_router_backward_closed_forms():
    """The logit gradients of a token sum to zero (softmax is shift-invariant);
    K = 1 gives no gradient at all; equal dgate on all routes gives none; and
    dx is added to the dx passed in."""
    rng = np.random.default_rng(12)
    T, d, N, K = 20, 16, 8, 4
    x = synth.gen_bf16(1, (T, d), "x")
    w = rng.standard_normal((N, d)).astype(np.float32)
    idx = synth.gen_topk_idx(3, T, N, K)
    g = rng.random((T, K)).astype(np.float32)
    g /= g.sum(1, keepdims=True)
    dg = rng.standard_normal((T, K)).astype(np.float32)
    dl, dx, dw, db = oracle.router_bwd(x, w, idx, g, dg)
    np.testing.assert_allclose(dl.astype(np.float64).sum(1), 0, atol=1e-6)
    np.testing.assert_allclose(db.astype(np.float64).sum(), 0, atol=1e-5)
    dl1, dx1, dw1, db1 = oracle.router_bwd(x, w, idx[:, :1], np.ones((T, 1), np.float32), dg[:, :1])
    assert np.all(dl1 == 0) and np.all(dx1 == 0) and np.all(dw1 == 0)
    same = np.repeat(dg[:, :1], K, 1)
    dl2, _, _, _ = oracle.router_bwd(x, w, idx, g, same)
    np.testing.assert_allclose(dl2, 0, atol=1e-6)
    base = rng.standard_normal((T, d)).astype(np.float32)
    _, dx3, _, _ = oracle.router_bwd(x, w, idx, g, dg, dx=base)
    np.testing.assert_allclose(dx3, base + dx, rtol=1e-6, atol=1e-6)

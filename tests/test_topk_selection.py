"""The router's top-K selection procedure, restated on the CPU.

The GPU splits each token's experts over four lanes (lane s takes experts
s, s + 4, ...), sorts them MAXK at a time with a bitonic network, merges each
batch into the lane's sorted list, and merges the four lists over two lane
shuffles.  This restates that procedure step by step in plain Python and checks
that it picks exactly the oracle's top K (logit descending, lower expert first
on ties, NaN as -inf) on random logits full of ties and infinities, for the
list lengths the kernel is built with (8 and 16).  It tests the procedure, not
the kernel: the GPU tests compare the kernel's output with the oracle.
"""
import math

import numpy as np
import pytest

import oracle

UNFILLED = (-math.inf, 2 ** 31 - 1)  # any expert beats it


def _beats(a, b):
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


def _bitonic_sort(v):
    """Best first; the compare-exchange pattern of a bitonic sorting network."""
    m = len(v)
    k = 2
    while k <= m:
        j = k >> 1
        while j:
            for i in range(m):
                l = i ^ j
                if l > i:
                    swap = _beats(v[l], v[i]) if (i & k) == 0 else _beats(v[i], v[l])
                    if swap:
                        v[i], v[l] = v[l], v[i]
            j >>= 1
        k <<= 1
    return v


def _merge(mine, other):
    """Best len(mine) of two lists sorted best first: the better of entry q and
    the other list's entry m - 1 - q form a bitonic sequence, then a bitonic
    merge network sorts it."""
    m = len(mine)
    v = [other[m - 1 - q] if _beats(other[m - 1 - q], mine[q]) else mine[q] for q in range(m)]
    s = m // 2
    while s:
        for q in range(m):
            if not q & s and _beats(v[q + s], v[q]):
                v[q], v[q + s] = v[q + s], v[q]
        s //= 2
    return v


def _select(logits, maxk):
    """The kernel's procedure for one token: returns its best maxk pairs."""
    n = len(logits)
    canon = [(-math.inf if math.isnan(x) else float(x), e) for e, x in enumerate(logits)]
    lanes = []
    for sub in range(4):
        mine = [UNFILLED] * maxk
        ids = list(range(sub, n, 4))
        for i0 in range(0, len(ids), maxk):
            batch = [canon[e] for e in ids[i0:i0 + maxk]]
            batch += [UNFILLED] * (maxk - len(batch))
            batch = _bitonic_sort(batch)
            mine = batch if i0 == 0 else _merge(mine, batch)
        lanes.append(mine)
    pair01 = _merge(lanes[0], lanes[1])
    pair23 = _merge(lanes[2], lanes[3])
    assert pair01 == _merge(lanes[1], lanes[0])  # both lanes of a pair agree
    return _merge(pair01, pair23)


@pytest.mark.parametrize("maxk", [8, 16])
def test_lane_split_selection_picks_the_oracle_top_k(maxk):
    rng = np.random.default_rng(11 + maxk)
    specials = np.array([0.0, 1.0, -1.0, np.inf, -np.inf, np.nan], dtype=np.float32)
    for _ in range(300):
        n = int(rng.integers(1, 140))
        k = int(rng.integers(1, min(maxk, n) + 1))
        logits = rng.standard_normal(n).astype(np.float32)
        mask = rng.random(n) < 0.3
        logits[mask] = rng.choice(specials, size=int(mask.sum()))
        idx, _ = oracle.topk_gates(logits[None, :], k)
        got = [e for _, e in _select(logits.tolist(), maxk)[:k]]
        assert got == idx[0].tolist(), (logits.tolist(), k)


def test_merge_keeps_the_best_of_both_lists():
    a = _bitonic_sort([(3.0, 5), (1.0, 2), (1.0, 9), UNFILLED])
    b = _bitonic_sort([(2.0, 7), (1.0, 1), (-math.inf, 4), (5.0, 0)])
    assert _merge(a, b) == [(5.0, 0), (3.0, 5), (2.0, 7), (1.0, 1)]

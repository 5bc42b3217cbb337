"""The GPU's slot-assignment procedure, restated on the CPU.

The kernels give every accepted route its row in three launches: per block of
256 tokens, each route's rank among the block's earlier routes to its expert
(per-warp bitmasks of the tokens choosing each expert, counted with popc) and
the block's count per expert; a scan of those counts with up to 32 threads per
expert, each over a contiguous chunk of blocks; and row = offset[e] + block
base + rank, or -1 when that slot is past capacity.  This restates the
procedure step by step and checks it against the oracle's token-order rule
(OLMo-core MoE report, "Section 05: Expert Parallelism", 5.4 and Figure 16)
on shapes the GPU tests do not reach: one expert, 1024 experts, token counts
that leave a ragged last block, block counts that leave empty chunks, zero
capacity and no tokens.  It tests the decomposition, not the kernels: the GPU
tests compare the kernels' output with the oracle.
"""
import numpy as np
import pytest

import oracle

RANK_BLOCK = 256
MAX_N = 1024


def _popc(v):
    return bin(v).count("1")


def _block_rank(idx, N):
    """Ranks inside each 256-token block and the block counts [nblk][N]."""
    T, K = idx.shape
    nblk = (T + RANK_BLOCK - 1) // RANK_BLOCK
    rank = np.zeros((T, K), dtype=np.int64)
    block_count = np.zeros((nblk, N), dtype=np.int64)
    for b in range(nblk):
        masks = [[0] * N for _ in range(RANK_BLOCK // 32)]
        for t in range(b * RANK_BLOCK, min(T, (b + 1) * RANK_BLOCK)):
            w, lane = (t % RANK_BLOCK) // 32, t % 32
            for k in range(K):
                masks[w][idx[t, k]] |= 1 << lane
        wpre = [[0] * N for _ in masks]
        for e in range(N):
            run = 0
            for w in range(len(masks)):
                wpre[w][e] = run
                run += _popc(masks[w][e])
            block_count[b, e] = run
        for t in range(b * RANK_BLOCK, min(T, (b + 1) * RANK_BLOCK)):
            w, lane = (t % RANK_BLOCK) // 32, t % 32
            for k in range(K):
                e = idx[t, k]
                rank[t, k] = wpre[w][e] + _popc(masks[w][e] & ((1 << lane) - 1))
    return rank, block_count


def _lanes_per_expert(nblk, N):
    return max(1, min(32, MAX_N // N, nblk // 4))


def _scan(block_count, N, cap):
    """Block bases (in place of the counts), demand, count and offsets."""
    nblk = block_count.shape[0]
    P = _lanes_per_expert(nblk, N)
    chunk = (nblk + P - 1) // P
    assert P * N <= MAX_N  # one CTA of 1024 threads, one shared-memory slot each
    bounds = [(min(p * chunk, nblk), min(min(p * chunk, nblk) + chunk, nblk)) for p in range(P)]
    chunk_sum = np.array([[block_count[b0:b1, e].sum() for e in range(N)] for b0, b1 in bounds])
    base = block_count.copy()
    for p, (b0, b1) in enumerate(bounds):
        for e in range(N):
            run = int(chunk_sum[:p, e].sum())
            for b in range(b0, b1):
                base[b, e] = run
                run += int(block_count[b, e])
    covered = sorted(b for b0, b1 in bounds for b in range(b0, b1))
    assert covered == list(range(nblk))  # the chunks tile the blocks exactly once
    demand = chunk_sum.sum(axis=0)
    count = np.minimum(demand, cap)
    offset = np.concatenate([[0], np.cumsum(count)])
    return base, demand, count, offset


def _assign(idx, rank, base, offset, cap):
    T, K = idx.shape
    row = np.empty((T, K), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            slot = base[t // RANK_BLOCK, e] + rank[t, k]
            row[t, k] = offset[e] + slot if slot < cap else -1
    return row


def _routes(rng, T, N, K, zipf_s):
    """Distinct experts per token; Zipf-skewed choices by the Gumbel top-K trick."""
    if T == 0:
        return np.zeros((0, K), dtype=np.int32)
    logp = -zipf_s * np.log(rng.permutation(N) + 1.0)
    keys = logp[None, :] + rng.gumbel(size=(T, N))
    return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)


CASES = [
    # (T, N, K, cap, zipf_s)
    (0, 8, 2, 4, 0.0),
    (1, 1, 1, 1, 0.0),
    (300, 1, 1, 7, 0.0),          # one expert, ragged last block
    (256, 8, 2, 80, 0.0),
    (1000, 16, 4, 0, 0.0),        # zero capacity: every route dropped
    (2049, 64, 8, 200, 1.2),      # 9 blocks: chunks of 2, one chunk left empty
    (4096, 32, 4, 10 ** 6, 0.0),  # 16 blocks, 4 threads per expert, no drops
    (9000, 16, 2, 900, 1.2),      # 36 blocks, 9 threads per expert
    (1500, 1024, 16, 20, 1.2),    # 1024 experts: one thread per expert
    (3000, 100, 8, 240, 1.2),     # 12 blocks, 3 threads per expert
]


@pytest.mark.parametrize("T,N,K,cap,zipf_s", CASES)
def test_three_launch_slot_assignment_equals_the_token_order_rule(T, N, K, cap, zipf_s):
    rng = np.random.default_rng(1000 + T + N)
    idx = _routes(rng, T, N, K, zipf_s)
    row_o, count_o, offset_o, demand_o = oracle.route_slots(idx, N, cap)
    rank, block_count = _block_rank(idx, N)
    base, demand, count, offset = _scan(block_count, N, cap)
    row = _assign(idx, rank, base, offset, cap)
    np.testing.assert_array_equal(demand, demand_o)
    np.testing.assert_array_equal(count, count_o)
    np.testing.assert_array_equal(offset, offset_o)
    np.testing.assert_array_equal(row, row_o)


def test_threads_per_expert_stay_within_one_cta():
    for N in (1, 2, 3, 7, 8, 31, 32, 33, 64, 100, 128, 1000, 1024):
        for nblk in (0, 1, 3, 4, 5, 31, 32, 33, 127, 128, 129, 4096):
            P = _lanes_per_expert(nblk, N)
            assert 1 <= P <= 32 and P * N <= MAX_N
            assert P == 1 or nblk // P >= 4  # at least 4 blocks for each thread

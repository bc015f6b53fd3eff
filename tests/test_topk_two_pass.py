"""The two-pass top-k selection of the fused verify kernel, restated on the CPU: its
exactness argument against a full sort (CPU only; the GPU kernel itself is checked
against the oracle in test_verify_gpu.py).

Pass 1 records, for each fine block of a row (a fixed partition; 256 elements here), its
largest value, the id of one element at that value and its second largest value (a tie
at the top counts twice).  Pass 2: each of 32 lanes takes the maximum over its share of
the fine blocks (pairs of blocks 2q, 2q + 1 with q = lane + 32 i); tau, the k-th largest
lane maximum, is at most the row's k-th largest value (and no larger bound will do: when
the top k lie one per lane, the k-th of them is a lane maximum).  The block maxima >= tau
form the candidate list, whose k-th value tau2 is again at most the row's k-th largest
value.  An
element of the top k that is not its block's recorded maximum is at most the block's
second value, so every such block has a second value >= tau2 and is read again, adding its
elements >= tau2 other than the recorded one.  The list then holds the top k by (value
descending, id ascending) exactly -- ties, constant rows, masked (-inf) rows and
vocabularies smaller than 32 blocks included, and whichever tied element pass 1 records.
"""
import numpy as np
import pytest

FINE = 256
LANES = 32


def top_k_by_sort(x, k):
    return [int(i) for i in np.argsort(-x, kind="stable")[:k]]


def top_k_two_pass(x, k, rng):
    V = x.size
    nfb = -(-V // FINE)
    blocks = [np.arange(f * FINE, min(V, (f + 1) * FINE)) for f in range(nfb)]
    m1, rid, m2 = [], [], []
    for ids in blocks:
        v = x[ids]
        top = v.max()
        at = ids[v == top]
        r = int(rng.choice(at))                      # any element at the maximum may be recorded
        m1.append(top)
        rid.append(r)
        rest = x[ids[ids != r]]
        m2.append(rest.max() if rest.size else -np.inf)
    lane_max = np.full(LANES, -np.inf)
    for f in range(nfb):
        lane = (f // 2) % LANES
        lane_max[lane] = max(lane_max[lane], m1[f])
    rank = [sum(1 for j in range(LANES) if lane_max[j] > lane_max[l] or (lane_max[j] == lane_max[l] and j < l))
            for l in range(LANES)]
    tau = lane_max[rank.index(k - 1)]
    key = lambda e: (-e[0], e[1])
    cand = sorted(((m1[f], rid[f]) for f in range(nfb) if m1[f] >= tau), key=key)[:k]
    tau2 = cand[k - 1][0] if len(cand) >= k else -np.inf
    extra = [(x[e], int(e)) for f in range(nfb) if m2[f] >= tau2
             for e in blocks[f] if e != rid[f] and x[e] >= tau2]
    return [i for _, i in sorted(cand + extra, key=key)[:k]], sum(1 for f in range(nfb) if m2[f] >= tau2)


def _rows():
    g = np.random.default_rng(0)
    yield "normal 151936", g.normal(0, 3, 151936).astype(np.float32)
    spike = g.normal(0, 3, 151936).astype(np.float32)
    spike[int(g.integers(0, 151936))] += 8.5
    yield "normal + spike", spike
    yield "constant", np.zeros(3001, np.float32)
    yield "three values", g.integers(0, 3, 5000).astype(np.float32)
    crowded = g.normal(0, 1, 20000).astype(np.float32)
    crowded[300:556] = 100 + np.arange(256, dtype=np.float32)     # the whole top in one fine block
    yield "top in one block", crowded
    twin = g.normal(0, 1, 9000).astype(np.float32)
    twin[[17, 18, 4000, 4001, 4002]] = 50.0                         # tied maxima within blocks
    yield "tied maxima", twin
    spread = g.normal(0, 1, 151936).astype(np.float32)
    spread[np.arange(32) * 2 * FINE] = 100 + np.arange(32, dtype=np.float32)   # one top element per lane
    yield "one top element per lane", spread
    masked = np.full(8000, -np.inf, np.float32)
    masked[g.choice(8000, 7, replace=False)] = g.normal(0, 1, 7)
    yield "mostly -inf", masked
    yield "all -inf", np.full(700, -np.inf, np.float32)
    yield "tiny 5", g.normal(0, 1, 5).astype(np.float32)
    yield "tiny 2 tied", np.zeros(2, np.float32)
    yield "ragged 1025", g.integers(0, 4, 1025).astype(np.float32)


@pytest.mark.parametrize("k", [1, 20, 32])
def test_two_pass_selection_equals_full_sort(k):
    rng = np.random.default_rng(1)
    for name, x in _rows():
        kk = min(k, x.size)
        for _ in range(3):                           # different recorded elements among ties
            got, _ = top_k_two_pass(x, kk, rng)
            assert got == top_k_by_sort(x, kk), (name, k)


def test_blocks_read_again_are_few_on_the_benchmark_rows():
    """On N(0, 3^2) rows of 151,936 logits with top-k 20 only a block or so is read again."""
    rng = np.random.default_rng(2)
    g = np.random.default_rng(3)
    reread = [top_k_two_pass(g.normal(0, 3, 151936).astype(np.float32), 20, rng)[1] for _ in range(8)]
    assert max(reread) <= 3

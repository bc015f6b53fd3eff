"""Exact law of the acceptance rule by enumeration (test infrastructure only).

For fixed target rows P_1..P_{K+1} and draft rows Q_1..Q_K (tiny vocabularies), every
draft sequence d in supp(Q_1) x ... x supp(Q_K) is enumerated with weight prod Q_i(d_i).
The acceptance tests split each uniform u[i-1] into the accept cell [0, min(1, r_i)) and
the reject cell [min(1, r_i), 1) with r_i = P_i(d_i) / Q_i(d_i); the oracle's own
``accept_and_resample`` is evaluated at the midpoint of each reachable cell (and must
land in that cell's outcome), and the last token is distributed as the ``final``
distribution it reports.  The result is the exact law of (a, emitted tokens) under
the oracle, which the tests compare with what the mathematics of [MTP-fixes] "The
verify was wrong under sampling" fixes: the first emitted token follows P_1, token i+1
follows P_{i+1} given a >= i, and P(a >= 1) = sum_x min(P_1(x), Q_1(x)).
"""
import itertools
from collections import defaultdict

from .verify import accept_and_resample


def exact_outcome_law(P, Q):
    """P: list of K+1 dicts, Q: list of K dicts (id -> prob).

    Returns dict (a, emitted tuple) -> probability, where emitted = d_1..d_a, next.
    Raises AssertionError when the oracle's decision at a cell midpoint disagrees with
    the cell.
    """
    K = len(Q)
    law = defaultdict(float)
    supports = [sorted(q) for q in Q]
    for d in itertools.product(*supports):
        w = 1.0
        for i in range(K):
            w *= Q[i][d[i]]
        acc = [min(1.0, P[i].get(d[i], 0.0) / Q[i][d[i]]) for i in range(K)]
        reach = 1.0
        for a in range(K + 1):
            if a < K:
                pa = reach * (1.0 - acc[a])
            else:
                pa = reach
            if pa > 0.0:
                u = [acc[i] / 2.0 for i in range(a)]
                if a < K:
                    u.append((acc[a] + 1.0) / 2.0)
                u += [0.5] * (K - len(u))
                u.append(0.5)
                r = accept_and_resample(P, Q, d, u)
                assert r["a"] == a, (d, a, r["a"])
                for x, px in r["final"].items():
                    law[(a, tuple(d[:a]) + (x,))] += w * pa * px
            if a < K:
                reach *= acc[a]
                if reach == 0.0:
                    break
    return dict(law)


def marginal_token(law, position):
    """Law of the emitted token at `position` (0-based), restricted to outcomes that emit
    at least position+1 tokens, and the probability of emitting that many."""
    out = defaultdict(float)
    mass = 0.0
    for (a, toks), p in law.items():
        if len(toks) > position:
            out[toks[position]] += p
            mass += p
    return {k: v / mass for k, v in out.items()}, mass

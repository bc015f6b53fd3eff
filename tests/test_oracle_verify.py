"""Pins of the oracle's acceptance rule against what the pages and the mathematics fix.

* closed forms and special cases of the truncation (textbook softmax, top-k = 1, ties);
* the worked example of "What is Speculative Decoding and How Does a Draft Model Work?"
  section "#2" (three drafts kept, the fourth replaced by the target's word);
* brute-force laws of the rejection rule of "Qwen3.5 and Qwen3.6 MTP head reaches 1.4x
  on Apple Silicon after three fixes", section "The verify was wrong under sampling":
  first emitted token ~ P_1, token i+1 ~ P_{i+1} given a >= i, P(a >= 1) = sum min(P, Q);
* a chi-square test at 10^6 draws of the emitted-token law.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import verify as ov
from oracle.brute import exact_outcome_law, marginal_token

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(seed, n, V, scale=1.5):
    return np.random.default_rng(seed).normal(0, scale, size=(n, V))


def test_textbook_softmax_when_untruncated():
    x = _rows(1, 1, 11)[0]
    for T in (0.5, 1.0, 2.5):
        ids, p, _ = ov.truncated_distribution(x, T, 0, 1.0)
        ref = special.softmax(x / T)
        got = np.zeros_like(ref)
        got[ids] = p
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)
        ids2, p2, _ = ov.truncated_distribution(x, T, 50, 1.0)   # top_k >= V
        np.testing.assert_array_equal(ids, ids2)


def test_truncation_closed_forms():
    d = json.load(open(os.path.join(GOLDEN, "truncation_closed_forms.json")))
    for c in d["cases"]:
        ids, p, _ = ov.truncated_distribution(np.array(c["logits"]), c["temperature"], c["top_k"], c["top_p"])
        got = {str(int(i)): float(v) for i, v in zip(ids, p)}
        assert set(got) == set(c["expected"]), c["derivation"]
        for k, v in c["expected"].items():
            assert abs(got[k] - v) < 1e-12, c["derivation"]


def test_ranking_ties_go_to_lower_id():
    x = np.zeros(9)
    ids, p, _ = ov.truncated_distribution(x, 1.0, 4, 1.0)
    assert list(ids) == [0, 1, 2, 3]
    np.testing.assert_allclose(p, 0.25)
    assert ov.argmax_with_gap(x)[0] == 0
    y = np.array([1.0, 5.0, 2.0, 5.0])
    assert ov.argmax_with_gap(y) == (1, 0.0)


def test_top_p_keeps_first_token_always():
    x = np.array([10.0, 0.0, 0.0])
    ids, p, _ = ov.truncated_distribution(x, 1.0, 20, 0.01)
    assert list(ids) == [0] and p[0] == 1.0


def test_inverse_cdf_ascending_ids():
    dist = {7: 0.3, 1: 0.5, 3: 0.2}            # ascending: 1 (0.5], 3 (0.7], 7 (1.0]
    assert ov.inverse_cdf(dist, 0.1)[0] == 1
    assert ov.inverse_cdf(dist, 0.6)[0] == 3
    assert ov.inverse_cdf(dist, 0.95)[0] == 7
    assert ov.inverse_cdf(dist, 0.5)[0] == 3   # strict: running sum must exceed u*Z
    assert ov.inverse_cdf({4: 2.0, 9: 6.0}, 0.3)[0] == 9   # unnormalised weights


def test_worked_example_raining_cats_and_dogs():
    d = json.load(open(os.path.join(GOLDEN, "worked_example_raining_cats.json")))
    vocab = d["vocab"]
    V = len(vocab)
    rows = np.zeros((len(d["target_choice_per_row"]), V))
    for i, w in enumerate(d["target_choice_per_row"]):
        rows[i, vocab.index(w)] = 6.0
    drafts = [vocab.index(w) for w in d["drafts"]]
    g = ov.verify_greedy(rows, drafts)
    assert g["a"] == d["expected_accepted"] and vocab[g["next"]] == d["expected_next"]
    # the same outcome under the sampling rule with deterministic drafts: the target rows
    # are near one-hot (top_p 0.95 cuts everything but the top token)
    s = ov.verify_sampling(rows, None, drafts, [0.3] * (len(drafts) + 1), 1.0, 20, 0.95)
    assert s["a"] == d["expected_accepted"] and vocab[s["next"]] == d["expected_next"]


def test_greedy_prefix_rule():
    rows = _rows(3, 5, 16)
    g = [int(np.argmax(r)) for r in rows]
    for a in range(5):
        drafts = g[:a] + [(g[a] + 1) % 16] * (4 - a) if a < 4 else g[:4]
        r = ov.verify_greedy(rows, drafts)
        assert r["a"] == a and r["next"] == g[a]


def test_top_k_one_reduces_sampling_to_greedy():
    rng = np.random.default_rng(5)
    for _ in range(50):
        rows = rng.normal(size=(4, 12))
        drafts = list(rng.integers(0, 12, size=3))
        u = rng.random(4)
        s = ov.verify_sampling(rows, None, drafts, u, 0.7, 1, 0.95)
        g = ov.verify_greedy(rows, drafts)
        assert (s["a"], s["next"]) == (g["a"], g["next"])


def test_draft_equal_to_target_accepts_everything():
    rng = np.random.default_rng(6)
    for _ in range(30):
        rows = rng.normal(size=(4, 10))
        P = [ov.as_dict(*ov.truncated_distribution(r, 1.0, 5, 0.9)[:2]) for r in rows]
        drafts = [ov.inverse_cdf(P[i], rng.random())[0] for i in range(3)]
        r = ov.verify_sampling(rows, rows[:3], drafts, rng.random(4), 1.0, 5, 0.9)
        assert r["a"] == 3


def test_disjoint_supports_reject_first_and_draw_from_target():
    P = [{0: 0.6, 1: 0.4}, {2: 1.0}]
    Q = [{3: 0.5, 4: 0.5}]
    r = ov.accept_and_resample(P, Q, [3], [0.0, 0.7])
    assert r["a"] == 0 and r["final"] == {0: 0.6, 1: 0.4} and r["next"] == 1


def test_illegal_draft_raises():
    rows = np.array([[5.0, 0.0, 0.0], [0.0, 5.0, 0.0]])
    drows = np.array([[5.0, 0.0, 0.0]])
    with pytest.raises(ov.IllegalDraft):
        ov.verify_sampling(rows, drows, [2], [0.5, 0.5], 1.0, 1, 1.0)


def test_residual_all_zero_falls_back_to_target():
    # P <= Q everywhere on P's support can only happen when P == Q: then Z == 0
    P = [{0: 0.5, 1: 0.5}, {0: 1.0}]
    Q = [{0: 0.5, 1: 0.5}]
    r = ov.accept_and_resample(P, Q, [1], [0.99999, 0.2])   # u >= ratio = 1 never rejects
    assert r["a"] == 1
    assert ov.accept_and_resample(P, Q, [0], [0.3, 0.2])["a"] == 1


def _random_case(seed, V, K, top_k, top_p):
    rng = np.random.default_rng(seed)
    trows = rng.normal(0, 1.2, size=(K + 1, V))
    drows = trows[:K] + rng.normal(0, 1.0, size=(K, V))   # overlapping but different
    P = [ov.as_dict(*ov.truncated_distribution(r, 1.0, top_k, top_p)[:2]) for r in trows]
    Q = [ov.as_dict(*ov.truncated_distribution(r, 1.0, top_k, top_p)[:2]) for r in drows]
    return P, Q


@pytest.mark.parametrize("seed,V,K,top_k,top_p", [
    (0, 5, 1, 0, 1.0), (1, 6, 2, 0, 1.0), (2, 7, 3, 0, 1.0), (3, 8, 2, 4, 0.9),
    (4, 8, 3, 3, 0.8), (5, 4, 4, 0, 1.0)])
def test_brute_force_laws(seed, V, K, top_k, top_p):
    P, Q = _random_case(seed, V, K, top_k, top_p)
    law = exact_outcome_law(P, Q)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    # first emitted token follows P_1 exactly
    first, mass = marginal_token(law, 0)
    assert abs(mass - 1.0) < 1e-12
    for x in set(first) | set(P[0]):
        assert abs(first.get(x, 0.0) - P[0].get(x, 0.0)) < 1e-12
    # P(a >= 1) = sum_x min(P_1(x), Q_1(x))
    alpha = [sum(min(P[i].get(x, 0.0), q) for x, q in Q[i].items()) for i in range(K)]
    p_a_ge = lambda n: sum(p for (a, _), p in law.items() if a >= n)
    assert abs(p_a_ge(1) - alpha[0]) < 1e-12
    # acceptance events are independent across positions for fixed rows
    for n in range(1, K + 1):
        assert abs(p_a_ge(n) - math.prod(alpha[:n])) < 1e-12
    # given a >= i, token i+1 follows P_{i+1}
    for i in range(1, K + 1):
        cond = {}
        tot = 0.0
        for (a, toks), p in law.items():
            if a >= i:
                cond[toks[i]] = cond.get(toks[i], 0.0) + p
                tot += p
        if tot > 1e-9:
            for x in set(cond) | set(P[i]):
                assert abs(cond.get(x, 0.0) / tot - P[i].get(x, 0.0)) < 1e-10


def test_brute_force_catches_a_wrong_residual(monkeypatch):
    """A planted mistake (residual max(0, Q - P)) must break the law of the first token."""
    P, Q = _random_case(11, 6, 1, 0, 1.0)

    def wrong(P_, Q_, d, u):
        i = 0
        x = int(d[0])
        if float(u[0]) < P_[0].get(x, 0.0) / Q_[0][x]:
            return ov.accept_and_resample(P_, Q_, d, u)
        res = {y: max(0.0, Q_[0].get(y, 0.0) - P_[0].get(y, 0.0)) for y in Q_[0]}
        Z = sum(res.values())
        res = {y: w / Z for y, w in res.items() if w > 0}
        return {"a": i, "next": ov.inverse_cdf(res, u[1])[0], "final": res, "margin": 1.0}

    import oracle.brute as ob
    monkeypatch.setattr(ob, "accept_and_resample", wrong)
    law = ob.exact_outcome_law(P, Q)
    first, _ = marginal_token(law, 0)
    err = max(abs(first.get(x, 0.0) - P[0].get(x, 0.0)) for x in set(first) | set(P[0]))
    assert err > 1e-3


def test_chi_square_emitted_law_1e6():
    """10^6 draws: drafts from Q, the oracle rule with fresh uniforms; first emitted token
    against P_1 and second against P_2 (given a >= 1)."""
    V, K, n = 6, 2, 1_000_000
    P, Q = _random_case(21, V, K, 0, 1.0)
    rng = np.random.default_rng(1234)
    U = rng.random((n, 2 * K + 1))
    first = np.zeros(V)
    second = np.zeros(V)
    for t in range(n):
        u = U[t]
        d = [ov.inverse_cdf(Q[i], u[K + 1 + i])[0] for i in range(K)]
        r = ov.accept_and_resample(P, Q, d, u[:K + 1])
        toks = d[:r["a"]] + [r["next"]]
        first[toks[0]] += 1
        if r["a"] >= 1:
            second[toks[1]] += 1
    for counts, dist in ((first, P[0]), (second, P[1])):
        exp = np.array([dist.get(x, 0.0) for x in range(V)]) * counts.sum()
        m = exp > 0
        assert counts[~m].sum() == 0
        p = stats.chisquare(counts[m], exp[m]).pvalue
        assert p > 1e-4, p


def test_acceptance_is_strict():
    """Reading R5: accept iff u < P(d)/Q(d).  P(0) = 1/4, Q(0) = 1/2: u = 1/2 sits on the
    boundary and rejects; the residual max(0, P - Q) is all on token 1."""
    P = [{0: 0.25, 1: 0.75}, {2: 1.0}]
    Q = [{0: 0.5, 1: 0.5}]
    r = ov.accept_and_resample(P, Q, [0], [0.5, 0.0])
    assert r["a"] == 0 and r["next"] == 1 and r["final"] == {1: 1.0}
    assert ov.accept_and_resample(P, Q, [0], [0.4999, 0.0])["a"] == 1


def test_ratio_uses_the_truncated_draft_distribution():
    """[MTP-fixes] "Truncation has to match on both sides", top-k 2: the target row
    (ln 3, 0, -30) gives P = (3/4, 1/4, 0) and the draft row (0, ln 3, ln 3) gives
    Q = (0, 1/2, 1/2) (its untruncated softmax would be (1, 3, 3) / 7).  Draft token 1 has
    ratio (1/4) / (1/2) = 1/2 (untruncated: 7/12): u = 0.55 rejects, and the residual
    max(0, P - Q) is all on token 0; u = 0.45 accepts."""
    L = math.log(3.0)
    rows = np.array([[L, 0.0, -30.0], [0.0, 0.0, 5.0]])
    drows = np.array([[0.0, L, L]])
    r = ov.verify_sampling(rows, drows, [1], [0.55, 0.5], 1.0, 2, 1.0)
    assert r["a"] == 0 and r["next"] == 0 and r["final"] == {0: 1.0}
    assert ov.verify_sampling(rows, drows, [1], [0.45, 0.5], 1.0, 2, 1.0)["a"] == 1

"""Pins of the oracle's generation loops.

"Speculative Decoding on Apple Silicon..." section "Why this needed a patch to mlx_lm at
all": greedy speculative output is byte-identical to greedy non-speculative output; the
OptiQ docs ("N-gram lookup") say the same in float32.
"""
import itertools

import numpy as np
import pytest

import synth
from oracle import generate as og
from oracle import model as om
from oracle import verify as ov


@pytest.fixture(scope="module")
def pair():
    t = om.Decoder(synth.TINY_TARGET, synth.model_weights(synth.TINY_TARGET, seed=0))
    d = om.Decoder(synth.TINY_DRAFT, synth.model_weights(synth.TINY_DRAFT, seed=0))
    return t, d


def test_spec_greedy_equals_plain_greedy_tiny_config(pair):
    t, d = pair
    prompt = synth.prompt_tokens(1, 64, 1024)
    plain = og.plain_generate(t, prompt, 64)
    spec, stats = og.spec_generate_greedy(t, d, prompt, 64, K=4)
    assert spec == plain
    assert stats["steps"] <= 64


def test_spec_greedy_with_perfect_draft_accepts_everything(pair):
    t, _ = pair
    prompt = synth.prompt_tokens(7, 20, 1024)
    plain = og.plain_generate(t, prompt, 20)
    spec, stats = og.spec_generate_greedy(t, t, prompt, 20, K=4)
    assert spec == plain
    assert stats["accepted"] == 4 * stats["steps"]      # every draft is the target's own choice


def test_scripted_drafter_accepts_exactly_j_and_matches_closed_form(pair):
    """Drafts = j true tokens + a wrong one: greedy verify must accept exactly min(j, K);
    with j ~ Geometric(alpha = 0.7) the mean emitted per step is (1 - a^(K+1)) / (1 - a)."""
    t, _ = pair
    K, alpha = 4, 0.7
    prompt = list(synth.prompt_tokens(3, 16, 1024))
    traj = og.plain_generate(t, prompt, 200)
    seq = prompt + traj
    rng = np.random.default_rng(4)
    cache = t.new_cache()
    t.forward(seq[:len(prompt) - 1], cache)
    pos = len(prompt) - 1                   # index in seq of the pending token
    emitted = []
    while pos + K + 1 < len(seq):
        j = min(int(rng.geometric(1 - alpha)) - 1, K)
        drafts = og.scripted_drafts(seq, pos, K, j, lambda i: (seq[pos + 1 + i] + 1) % 1024)
        rows = t.forward([seq[pos]] + drafts, cache)
        r = ov.verify_greedy(rows, drafts)
        assert r["a"] == j and r["next"] == seq[pos + j + 1]
        cache.trim(pos + r["a"] + 1)
        emitted.append(r["a"] + 1)
        pos += r["a"] + 1
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(closed - 2.7731) < 1e-4
    m = np.mean(emitted)
    se = np.std(emitted) / np.sqrt(len(emitted))
    assert abs(m - closed) < 5 * se + 0.05


def test_ngram_draft_definition():
    ctx = [1, 2, 3, 4, 5, 9, 9, 1, 2, 3]
    assert og.ngram_draft(ctx, n_draft=8) == [4, 5, 9, 9, 1, 2, 3]
    assert og.ngram_draft(ctx, n_draft=2) == [4, 5]
    assert og.ngram_draft([1, 2, 3, 4, 5, 6], n_draft=4) == []     # no repeated 3-gram
    # the longest match wins over a more recent shorter one
    ctx2 = [7, 1, 2, 3, 50, 8, 2, 3, 60, 9, 7, 1, 2, 3]
    assert og.ngram_draft(ctx2, n_draft=3) == [50, 8, 2]
    # the 4-token suffix (7, 1, 2, 3) matches at 0 and is continued, although the 3-token
    # suffix (1, 2, 3) also occurs later, at 6 (it would continue with 60)
    ctx4 = [7, 1, 2, 3, 50, 9, 1, 2, 3, 60, 7, 1, 2, 3]
    assert og.ngram_draft(ctx4, n_draft=3) == [50, 9, 1]
    # of several earlier occurrences the most recent one is continued
    ctx3 = [1, 2, 3, 10, 1, 2, 3, 20, 1, 2, 3]
    assert og.ngram_draft(ctx3, n_draft=4) == [20, 1, 2, 3]


# ---- draft-length gate ------------------------------------------------------------------

@pytest.mark.parametrize("alpha", [0.0, 0.1, 0.5, 0.9, 1.0])
@pytest.mark.parametrize("n", [0, 1, 4, 8])
def test_gate_expected_tokens(alpha, n):
    """Mean emitted tokens against the geometric series in closed form and against a
    brute-force enumeration of every accept/reject pattern of the n drafts (a pass emits
    the accepted prefix plus one target token)."""
    e = og.DraftGate.expected_tokens(alpha, n)
    closed = n + 1.0 if alpha == 1.0 else (1.0 - alpha ** (n + 1)) / (1.0 - alpha)
    assert e == pytest.approx(closed, rel=1e-12, abs=1e-12)
    brute = 0.0
    for pattern in itertools.product((0, 1), repeat=n):
        p = 1.0
        for ok in pattern:
            p *= alpha if ok else 1.0 - alpha
        j = next((i for i, ok in enumerate(pattern) if not ok), n)
        brute += p * (j + 1)
    assert e == pytest.approx(brute, rel=1e-12, abs=1e-12)


def test_gate_hand_worked_decisions():
    # no history: alpha = 1/2.  cost grows by 1/4 of a pass per drafted token:
    # E/cost = 1/1, 1.5/1.25 = 1.2, 1.75/1.5 = 1.1667, 1.875/1.75 = 1.0714 -> 1 draft
    g = og.DraftGate([1.0, 1.25, 1.5, 1.75, 2.0])
    assert g.acceptance() == 0.5
    assert g.choose(4) == 1
    assert g.choose(0) == 0                 # nothing offered, nothing drafted
    # an exact tie (1.5 / 1.5 = 1 / 1) goes to the shorter draft
    assert og.DraftGate([1.0, 1.5, 2.0]).choose(2) == 0
    # free drafts: any alpha > 0 takes the longest draft offered
    h = og.DraftGate([1.0] * 9)
    assert h.choose(8) == 8 and h.choose(3) == 3
    # one accepted token of one (S = 1, F = 0): alpha = 2/3; with cost 1 + n/4:
    # E = 1, 1.6667, 2.1111, 2.4074, 2.6049; E/cost = 1, 1.3333, 1.4074, 1.3757, 1.3025
    # -> 2 drafts
    g.update(1, 1)
    assert g.acceptance() == pytest.approx(2.0 / 3.0)
    assert g.choose(4) == 2


def test_gate_new_prose_then_retry():
    """Rejection after rejection (decay 0.9): F tends to 1 / (1 - 0.9) = 10 and alpha to
    1/12, below the 1/4 that a first draft at cost 1.25 needs ((1 + alpha) / 1.25 > 1), so
    the gate stops drafting.  Rounds without drafts then only decay F: drafting resumes once
    10 * 0.9^r < 2, at r = 16."""
    g = og.DraftGate([1.0, 1.25, 1.5, 1.75, 2.0], decay=0.9)
    for _ in range(200):
        g.update(1, 0)
    assert g.acceptance() == pytest.approx(1.0 / 12.0, rel=1e-6)
    assert g.choose(4) == 0
    for r in range(1, 40):
        g.update(0, 0)
        if g.choose(4) > 0:
            break
    assert r == 16


def test_gate_copying_drafts_long():
    """All 8 drafts accepted every round: S tends to 8 / (1 - 0.9) = 80, alpha to 81/82, and
    with cost 1 + n/4 the full draft wins (E(8) / 3 = 2.86 against E(1) / 1.25 = 1.59)."""
    g = og.DraftGate([1.0 + n / 4 for n in range(9)])
    for _ in range(200):
        g.update(8, 8)
    assert g.acceptance() == pytest.approx(81.0 / 82.0, rel=1e-6)
    assert g.choose(8) == 8
    assert g.choose(5) == 5

"""Pins of the oracle's generation loops.

"Speculative Decoding on Apple Silicon..." section "Why this needed a patch to mlx_lm at
all": greedy speculative output is byte-identical to greedy non-speculative output; the
OptiQ docs ("N-gram lookup") say the same in float32.
"""
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

"""The native n-gram drafter (spec_ngram_*) against the oracle's definition of n-gram
lookup ("Speculative decoding on Apple Silicon" (mlx-optiq docs), section "N-gram lookup:
any model"), on contexts with copied spans; host code only, no GPU."""
import numpy as np
import pytest

import synth
from oracle import generate as og


@pytest.fixture(scope="module")
def ng():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import ngram
    return ngram


@pytest.mark.parametrize("seed,vocab,mm", [(5, 50, (3, 8)), (6, 7, (3, 8)), (7, 1000, (3, 8)), (8, 20, (1, 4)),
                                          (9, 3, (2, 2))])
def test_drafts_match_oracle_while_growing(ng, seed, vocab, mm):
    ctx = synth.ngram_prompt(seed, 400, vocab)
    d = ng.NgramDrafter(*mm)
    rng = np.random.default_rng(seed)
    pos = 0
    while pos < ctx.size:
        step = int(rng.integers(1, 9))
        d.append(ctx[pos:pos + step])
        pos = min(pos + step, ctx.size)
        assert len(d) == pos
        for n_draft in (1, 3, 8):
            exp = og.ngram_draft(ctx[:pos], n_draft=n_draft, min_match=mm[0], max_match=mm[1])
            assert list(d.draft(n_draft)) == exp, (pos, n_draft)


def test_batch_drafts_pad_and_lengths(ng):
    ctxs = [synth.ngram_prompt(s, n, 30) for s, n in ((1, 200), (2, 3), (3, 90))]
    ds = [ng.NgramDrafter() for _ in ctxs]
    for d, c in zip(ds, ctxs):
        d.append(c)
    toks, lens = ng.draft_batch(ds, 8)
    for b, c in enumerate(ctxs):
        exp = og.ngram_draft(c, n_draft=8)
        assert lens[b] == len(exp)
        assert list(toks[b, :lens[b]]) == exp and np.all(toks[b, lens[b]:] == 0)


def test_definition_cases(ng):
    """The oracle's own pinned cases, through the native index."""
    d = ng.NgramDrafter()
    d.append([1, 2, 3, 4, 5, 9, 9, 1, 2, 3])
    assert list(d.draft(8)) == [4, 5, 9, 9, 1, 2, 3]
    assert list(d.draft(2)) == [4, 5]
    e = ng.NgramDrafter()
    e.append([1, 2, 3, 4, 5, 6])
    assert list(e.draft(4)) == []
    g = ng.NgramDrafter()
    g.append([7, 1, 2, 3, 50, 8, 2, 3, 60, 9, 7, 1, 2, 3])     # longest match beats a later shorter one
    assert list(g.draft(3)) == [50, 8, 2]
    h = ng.NgramDrafter()
    h.append([7, 1, 2, 3, 50, 9, 1, 2, 3, 60, 7, 1, 2, 3])     # 4-token match at 0, 3-token also at 6
    assert list(h.draft(3)) == [50, 9, 1]
    m = ng.NgramDrafter()
    m.append([1, 2, 3, 10, 1, 2, 3, 20, 1, 2, 3])              # the most recent occurrence is continued
    assert list(m.draft(4)) == [20, 1, 2, 3]
    f = ng.NgramDrafter()
    f.append([])
    assert list(f.draft(4)) == [] and len(f) == 0


def test_bad_arguments(ng):
    from speculative_decoding_verify_token_gb300 import _lib
    with pytest.raises(_lib.SpecError):
        ng.NgramDrafter(0, 3)
    with pytest.raises(_lib.SpecError):
        ng.NgramDrafter(4, 3)
    with pytest.raises(_lib.SpecError):
        ng.NgramDrafter(3, 9)


@pytest.mark.parametrize("seed,decay", [(0, 0.9), (1, 0.5), (2, 1.0), (3, 0.0)])
def test_gate_matches_oracle(ng, seed, decay):
    """The native draft-length gate (spec_ngram_gate_*) against the oracle's DraftGate over
    random rounds: same acceptance estimate, same draft length (where the oracle's two best
    scores are within rounding of each other, either of them)."""
    rng = np.random.default_rng(seed)
    n_max = 8
    cost = np.cumsum(np.concatenate([[1.0], rng.uniform(0.02, 0.4, n_max)]))
    nat = ng.DraftGate(cost, decay=decay)
    ref = og.DraftGate(cost, decay=decay)
    for r in range(300):
        avail = int(rng.integers(0, n_max + 3))
        n = nat.choose(avail)
        e = ref.choose(avail)
        if n != e:
            sc = ref.scores(avail)
            assert abs(sc[n] - sc[e]) <= 1e-12 * sc[e], (r, n, e)
        assert nat.acceptance() == pytest.approx(ref.acceptance(), rel=1e-12)
        # copied spans are accepted whole, new prose mostly rejected
        acc = n if rng.random() < 0.5 else int(rng.integers(0, n + 1))
        nat.update(n, acc)
        ref.update(n, acc)
    nat.close()


def test_gate_argument_errors(ng):
    from speculative_decoding_verify_token_gb300._lib import SpecError
    with pytest.raises(SpecError):
        ng.DraftGate([1.0, 0.0, 2.0])
    with pytest.raises(SpecError):
        ng.DraftGate([1.0, 2.0], decay=1.5)
    g = ng.DraftGate([1.0, 1.25])
    with pytest.raises(SpecError):
        g.update(2, 3)
    with pytest.raises(SpecError):
        g.update(-1, 0)
    assert g.choose(-4) == 0
    g.close()

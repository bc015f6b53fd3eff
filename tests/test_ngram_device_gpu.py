"""The n-gram drafter on the device ("Speculative decoding on Apple Silicon" (mlx-optiq docs),
section "N-gram lookup: any model") against the oracle's lookup, exactly.

The device drafter reads each slot's context from the token ids the library records as it
embeds them (prefill, verify, decode) up to the slot's KV length, followed by the pending
token.  Checked:
  * after prefill, on contexts of 2 to 1500 tokens (copied spans, a 3-token period whose
    draft runs into the pending token, a 4-letter alphabet where the longest suffix match is
    the cap), for several (n_draft, min_match, max_match): draft_len and the drafted tokens
    equal oracle.generate.ngram_draft, and the rows past draft_len hold the pending token;
  * a per-sequence cap shortens the draft to min(cap, oracle length);
  * across greedy verify rounds fed by the device drafts (the cache trimmed to the accepted
    prefix each round), the drafts still equal the oracle's lookup on the committed tokens;
  * the float32 path (its own embedding kernel instance) records the same context;
  * the draft-length gate on the device (section "N-gram lookup: any model": the draft
    length follows recent acceptance against the timed cost of a verify pass) chooses what
    the oracle's DraftGate chooses over random rounds, and the gated drafter drafts that
    many tokens of each sequence's available continuation.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import generate as og
from oracle import verify as ov

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model
    return model


def contexts(vocab):
    g = np.random.Generator(np.random.PCG64(3))
    period = np.tile(np.array([11, 12, 13], dtype=np.int32), 10)[:29]
    small = g.integers(0, 4, size=400).astype(np.int32) + 100
    return [synth.ngram_prompt(1, 700, vocab), synth.ngram_prompt(2, 1500, vocab),
            synth.ngram_prompt(3, 129, vocab), period, small,
            np.array([5, 5], dtype=np.int32), np.array([7, 8, 7, 8, 7], dtype=np.int32),
            synth.prompt_tokens(4, 300, vocab)]


def check_draft(ctx, drafts, dl, n_draft, min_match, max_match, cap=None):
    ref = og.ngram_draft(ctx, n_draft=n_draft, min_match=min_match, max_match=max_match)
    if cap is not None:
        ref = ref[:max(0, cap)]
    assert int(dl) == len(ref), (len(ctx), int(dl), len(ref))
    assert [int(t) for t in drafts[:len(ref)]] == ref
    assert np.all(drafts[len(ref):] == ctx[-1])


@pytest.mark.parametrize("shape", [synth.SMALL_BF16, synth.TINY_TARGET], ids=["bf16", "f32"])
def test_device_ngram_matches_oracle_after_prefill(M, shape):
    ctxs = contexts(shape.vocab)
    B = len(ctxs)
    w = synth.model_weights(shape, seed=0, device="cuda")
    m = M.SpecModel(shape, w, max_batch=B, max_ctx=1600, max_k=8, prefill_chunk=256)
    for b, c in enumerate(ctxs):
        m.prefill(b, torch.from_numpy(c[:-1]).cuda())
    pending = torch.tensor([int(c[-1]) for c in ctxs], dtype=torch.int32, device="cuda")
    n_hit = 0
    for n_draft, lo, hi in [(8, 3, 8), (4, 1, 1), (16, 2, 4), (1, 1, 8), (64, 8, 8)]:
        drafts, dl = m.ngram_draft(list(range(B)), pending, n_draft, lo, hi)
        drafts, dl = drafts.cpu().numpy(), dl.cpu().numpy()
        for b, c in enumerate(ctxs):
            check_draft(c, drafts[b], dl[b], n_draft, lo, hi)
        n_hit += int((dl > 0).sum())
    assert n_hit > 10
    # slots in another order, and a cap per sequence (including 0 and above n_draft)
    order = [4, 0, 3, 7, 6]
    cap = torch.tensor([2, 0, 5, 100, 1], dtype=torch.int32, device="cuda")
    drafts, dl = m.ngram_draft(order, pending[order].contiguous(), 8, 3, 8, cap=cap)
    drafts, dl = drafts.cpu().numpy(), dl.cpu().numpy()
    for i, b in enumerate(order):
        check_draft(ctxs[b], drafts[i], dl[i], 8, 3, 8, cap=int(cap[i]))
    m.close()


def test_device_ngram_across_verify_rounds(M):
    shape = synth.SMALL_BF16
    w = synth.model_weights(shape, seed=0, device="cuda")
    B, K, rounds = 4, 8, 6
    ctxs = [synth.ngram_prompt(10 + b, n, shape.vocab) for b, n in enumerate((200, 517, 64, 333))]
    m = M.SpecModel(shape, w, max_batch=B, max_ctx=600 + (K + 1) * rounds, max_k=K, prefill_chunk=256)
    for b, c in enumerate(ctxs):
        m.prefill(b, torch.from_numpy(c[:-1]).cuda())
    ctxs = [[int(t) for t in c] for c in ctxs]
    pending = torch.tensor([c[-1] for c in ctxs], dtype=torch.int32, device="cuda")
    u = torch.zeros(B, K + 1, dtype=torch.float32, device="cuda")
    seq = list(range(B))
    drafted = 0
    for r in range(rounds):
        drafts, dl = m.ngram_draft(seq, pending, K)
        hd, hl = drafts.cpu().numpy(), dl.cpu().numpy()
        for b in range(B):
            check_draft(np.array(ctxs[b]), hd[b], hl[b], K, 3, 8)
        drafted += int(hl.sum())
        out = m.verify(seq, pending, drafts, u, 0.0, draft_len=dl, want_logits=True)
        a = out["accepted_len"].cpu().numpy()
        nx = out["next_token"].cpu().numpy()
        lg = out["logits"].double().cpu().numpy()
        for b in range(B):
            ref = ov.verify_greedy(lg[b, :hl[b] + 1], hd[b, :hl[b]])
            assert (int(a[b]), int(nx[b])) == (ref["a"], ref["next"]), (r, b)
            ctxs[b] += [int(t) for t in hd[b, :a[b]]] + [int(nx[b])]
            assert m.seq_len(b) == len(ctxs[b]) - 1
        pending = out["next_token"].clone()
    assert drafted > 0
    m.close()


@pytest.mark.parametrize("decay", [0.9, 0.5, 1.0])
def test_device_gate_matches_oracle(M, decay):
    """The draft-length gate on the device against the oracle's DraftGate, per slot, over
    random rounds (same choice, or where the oracle's two best scores are within rounding,
    either), then applied by the drafter to each sequence's available continuation."""
    shape = synth.TINY_TARGET
    B, n_max = 4, 8
    rng = np.random.default_rng(int(decay * 10))
    cost = np.cumsum(np.concatenate([[1.0], rng.uniform(0.02, 0.4, n_max)]))
    w = synth.model_weights(shape, seed=0, device="cuda")
    ctxs = [np.tile(np.array([11, 12, 13], dtype=np.int32), 12)[:34], synth.ngram_prompt(9, 200, shape.vocab),
            synth.prompt_tokens(5, 60, shape.vocab), np.tile(np.array([40, 41, 42, 43, 44], dtype=np.int32), 9)]
    m = M.SpecModel(shape, w, max_batch=B, max_ctx=256, max_k=8, prefill_chunk=256)
    for b, c in enumerate(ctxs):
        m.prefill(b, torch.from_numpy(c[:-1]).cuda())
    m.gate_config(cost, decay)
    refs = [og.DraftGate(cost, decay=decay) for _ in range(B)]
    seq = list(range(B))

    def same_choice(ref, avail, got):
        e = ref.choose(avail)
        if got != e:
            sc = ref.scores(avail)
            assert abs(sc[got] - sc[e]) <= 1e-12 * sc[e], (avail, got, e)

    for r in range(60):
        avail = rng.integers(0, n_max + 3, size=B).astype(np.int32)
        n = m.gate_choose(seq, torch.from_numpy(avail).cuda()).cpu().numpy()
        for b in range(B):
            same_choice(refs[b], int(avail[b]), int(n[b]))
        acc = np.array([n[b] if rng.random() < 0.5 else rng.integers(0, n[b] + 1) for b in range(B)], dtype=np.int32)
        m.gate_update(seq, torch.from_numpy(n.astype(np.int32)).cuda(), torch.from_numpy(acc).cuda())
        for b in range(B):
            refs[b].update(int(n[b]), int(acc[b]))
    # the drafter with the gate: each sequence's draft length is the gate's choice for the
    # continuation its lookup finds, and the drafted tokens are that continuation's first ones
    pending = torch.tensor([int(c[-1]) for c in ctxs], dtype=torch.int32, device="cuda")
    drafts, dl = m.ngram_draft(seq, pending, 8, 3, 8, gated=True)
    drafts, dl = drafts.cpu().numpy(), dl.cpu().numpy()
    for b in range(B):
        full = og.ngram_draft(ctxs[b], n_draft=8)
        same_choice(refs[b], len(full), int(dl[b]))
        assert [int(t) for t in drafts[b, :dl[b]]] == full[:dl[b]]
    m.close()

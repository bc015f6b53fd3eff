"""Batched serving rounds on the GPU: ragged prompts, drafts from the native n-gram drafter
("Speculative decoding on Apple Silicon" (mlx-optiq docs), section "N-gram lookup: any
model"), one batched verify pass per round with per-sequence draft lengths and the KV cache
trimmed to the accepted prefix ("Speculative Decoding on Apple Silicon: 119% Faster on
Qwen3.8", "Why this needed a patch to mlx_lm at all").

A 2-layer slice of the 8B shape at full width and vocabulary, B=4 with prompts of 129 to
700 tokens, K=8, greedy:
  * every round's drafts equal the oracle's n-gram lookup on the committed tokens;
  * every sequence's accepted length and next token follow the oracle's greedy rule on the
    GPU's own verify rows (argmax ties go to the lower id on both sides, so exact);
  * each sequence's KV length grows by exactly accepted + 1;
  * the first round's verify rows of one sequence match the float64 oracle within 3e-2.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import generate as og
from oracle import model as om
from oracle import verify as ov

pytestmark = pytest.mark.gpu
LOGIT_TOL = 3e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model, ngram
    return model, ngram


class EmbedRows:
    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        return self.t[torch.as_tensor(np.asarray(idx))].double().numpy()


def test_serving_rounds(lib):
    model, ngram = lib
    shape = dataclasses.replace(synth.QWEN_8B, n_layers=2, name="dense-8b-2l")
    w = synth.model_weights(shape, seed=0, device="cuda")
    B, K, rounds = 4, 8, 5
    lens = [300, 517, 129, 700]
    m = model.SpecModel(shape, w, max_batch=B, max_ctx=max(lens) + (K + 1) * rounds + 16, max_k=K,
                        prefill_chunk=256)
    ctx, drafters = [], []
    for b in range(B):
        p = synth.ngram_prompt(5 + b, lens[b], shape.vocab)
        m.prefill(b, torch.from_numpy(p[:-1]).cuda())
        d = ngram.NgramDrafter(3, 8)
        d.append(p)
        ctx.append([int(t) for t in p])
        drafters.append(d)
    u = torch.zeros(B, K + 1, dtype=torch.float32, device="cuda")
    matched = 0
    for r in range(rounds):
        toks, dl = ngram.draft_batch(drafters, K)
        for b in range(B):
            assert list(toks[b, :dl[b]]) == og.ngram_draft(ctx[b], n_draft=K), (r, b)
        matched += int((dl > 0).sum())
        last = torch.tensor([c[-1] for c in ctx], dtype=torch.int32, device="cuda")
        before = [m.seq_len(b) for b in range(B)]
        out = m.verify(list(range(B)), last, torch.from_numpy(toks).cuda(), u, 0.0,
                       draft_len=torch.from_numpy(dl).cuda(), want_logits=True)
        a = out["accepted_len"].cpu().numpy()
        nx = out["next_token"].cpu().numpy()
        lg = out["logits"].double().cpu().numpy()
        assert np.all(out["status"].cpu().numpy() == 0)
        for b in range(B):
            ref = ov.verify_greedy(lg[b, :dl[b] + 1], toks[b, :dl[b]])
            assert (int(a[b]), int(nx[b])) == (ref["a"], ref["next"]), (r, b)
            assert m.seq_len(b) == before[b] + int(a[b]) + 1
        if r == 0:
            # the shortest sequence's rows against the float64 oracle
            b = 2
            host = {k: v.cpu() for k, v in w.items()}
            host["embed"] = EmbedRows(host["embed"])
            o = om.Decoder(shape, host)
            cache = o.new_cache()
            o.forward(ctx[b][:-1], cache, logits_rows=np.zeros(0, dtype=np.int64))
            rows = o.forward([ctx[b][-1]] + [int(t) for t in toks[b, :dl[b]]], cache)
            err = np.max(np.abs(lg[b, :dl[b] + 1] - rows))
            assert err < LOGIT_TOL, err
        for b in range(B):
            new = [int(t) for t in toks[b, :a[b]]] + [int(nx[b])]
            drafters[b].append(np.array(new, dtype=np.int32))
            ctx[b] += new
    assert matched > 0          # the prompts' copied spans give n-gram matches
    m.close()


def test_long_context_attention_bitwise(lib):
    """32 sequences of ~1300 tokens verified in one pass, and the same sequences alone (B=1)
    in a context of the same size (the attention's split length is fixed per context).
    Every split's arithmetic is the same, as is every other stage's per-token arithmetic,
    so the verify rows agree bit for bit."""
    model, _ = lib
    shape = dataclasses.replace(synth.QWEN_8B, n_layers=2, name="dense-8b-2l")
    w = synth.model_weights(shape, seed=0, device="cuda")
    B, K = 32, 8
    g = np.random.Generator(np.random.PCG64(11))
    lens = g.integers(1200, 1400, size=B)
    prompts = [synth.prompt_tokens(20 + b, int(lens[b]), shape.vocab) for b in range(B)]
    drafts = torch.from_numpy(g.integers(0, shape.vocab, size=(B, K)).astype(np.int32)).cuda()
    u = torch.zeros(B, K + 1, dtype=torch.float32, device="cuda")
    m = model.SpecModel(shape, w, max_batch=B, max_ctx=1400 + K + 8, max_k=K, prefill_chunk=256)
    for b in range(B):
        m.prefill(b, torch.from_numpy(prompts[b][:-1]).cuda())
    last = torch.tensor([int(p[-1]) for p in prompts], dtype=torch.int32, device="cuda")
    big = m.verify(list(range(B)), last, drafts, u, 0.0, want_logits=True)["logits"].cpu()
    m.close()
    for b in (0, 17):
        one = model.SpecModel(shape, w, max_batch=B, max_ctx=1400 + K + 8, max_k=K, prefill_chunk=256)
        one.prefill(0, torch.from_numpy(prompts[b][:-1]).cuda())
        r = one.verify([0], last[b:b + 1].clone(), drafts[b:b + 1].clone(), u[b:b + 1].clone(), 0.0,
                       want_logits=True)["logits"].cpu()
        assert torch.equal(r[0], big[b]), b
        one.close()


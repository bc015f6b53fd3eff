"""27B-class dense target with a 0.8B-class draft under sampling (temperature 1, top-k 20,
top-p 0.95): the draft proposes K tokens one at a time, the target checks them in one
batched pass ("Speculative Decoding on Apple Silicon: 119% Faster on Qwen3.8", section
"How speculative decoding works"), with the same truncation on both sides ("Qwen3.5 and
Qwen3.6 MTP head reaches 1.4x on Apple Silicon after three fixes", section "Truncation
has to match on both sides").

* 2-layer slices of both shapes at full width and vocabulary: the draft's decode logits
  and the target's verify logits against the float64 oracle (3e-2 max-abs), every drafted
  token and every round's decision (accepted length, next token) against the oracle rule
  on the GPU's own logits (exact unless within 1e-6 of a boundary), and against the oracle
  rule on the oracle's logits (excused within 0.06 of a boundary: twice the logit
  tolerance);
* the full shapes (64 and 28 layers, 2048-token prompt, K in {1, 4, 16}): every drafted
  token and round decision against the oracle rule on the GPU's own logits, and the
  target's verify rows against single-token decode rows, bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from oracle import verify as ov

pytestmark = pytest.mark.gpu
LOGIT_TOL = 3e-2
EDGE = 1e-6
EDGE_MODEL = 0.06
T, TOP_K, TOP_P = 1.0, 20, 0.95


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model
    return model


def sliced(shape, layers):
    return dataclasses.replace(shape, n_layers=layers, name=f"{shape.name}-{layers}l")


class EmbedRows:
    """Embedding table for the oracle, converted to float64 one gathered row set at a time."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        return self.t[torch.as_tensor(np.asarray(idx))].double().numpy()


def oracle_of(shape, w):
    host = {k: v.cpu() for k, v in w.items()}
    host["embed"] = EmbedRows(host["embed"])
    return om.Decoder(shape, host)


def spec_round(target, draft, pending, K, gd, g, extra):
    """One draft-then-verify round on slot 0; returns drafts, draft logits, uniforms, the
    verify outputs (with logits) and the draft token to ingest next round (if a == K)."""
    dev = target.device
    if extra is not None:
        draft.prefill(0, extra)
    toks, rows, uds = [], [], []
    tok = pending
    for _ in range(K):
        ud = torch.from_numpy(gd.random(1, dtype=np.float32)).to(dev)
        tok, lg = draft.decode([0], tok, ud, T, TOP_K, TOP_P, want_logits=True)
        toks.append(tok)
        rows.append(lg)
        uds.append(float(ud.item()))
    d = torch.stack(toks, dim=1)
    dl = torch.stack(rows, dim=1)
    u = torch.from_numpy(g.random((1, K + 1), dtype=np.float32)).to(dev)
    r = target.verify([0], pending, d, u, T, TOP_K, TOP_P, draft_logits=dl, want_logits=True)
    a = int(r["accepted_len"].item())
    draft.kv_trim([0], K - 1, torch.clamp(r["accepted_len"], max=K - 1))
    nxt_extra = d[0, K - 1:K].clone() if a == K else None
    return d, dl, np.array(uds), u, r, nxt_extra


def check_rule_on_gpu_logits(d, dl, uds, u, r):
    """Drafts sampled from the GPU's truncated q, and the decision from the GPU's rows."""
    drafts = d[0].cpu().numpy()
    drows = dl[0].double().cpu().numpy()
    for i in range(drafts.size):
        tok, margin = ov.sample_token(drows[i], uds[i], T, TOP_K, TOP_P)
        if margin >= EDGE:
            assert int(drafts[i]) == tok, (i, int(drafts[i]), tok)
    ref = ov.verify(r["logits"][0].double().cpu().numpy(), drows, drafts, list(u[0].cpu().numpy()), T, TOP_K, TOP_P)
    if ref["margin"] >= EDGE:
        assert int(r["accepted_len"].item()) == ref["a"]
        assert int(r["next_token"].item()) == ref["next"]
    return ref


def test_27b_and_draft_slices_match_oracle(lib):
    ts, ds = sliced(synth.QWEN_27B, 2), sliced(synth.DRAFT_0P8B, 2)
    wt = synth.model_weights(ts, seed=0, device="cuda")
    wd = synth.model_weights(ds, seed=0, device="cuda")
    V = ts.vocab
    K = 4
    prompt = synth.prompt_tokens(1, 40, V)
    target = lib.SpecModel(ts, wt, max_ctx=256, max_k=K)
    draft = lib.SpecModel(ds, wd, max_ctx=256, max_k=K)
    target.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    draft.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    o_t, o_d = oracle_of(ts, wt), oracle_of(ds, wd)
    committed = [int(x) for x in prompt]
    pending = torch.tensor([committed[-1]], dtype=torch.int32, device="cuda")
    gd, g = np.random.Generator(np.random.PCG64(4)), np.random.Generator(np.random.PCG64(2))
    extra = None
    excused = 0
    for _ in range(3):
        d, dl, uds, u, r, extra = spec_round(target, draft, pending, K, gd, g, extra)
        drafts = [int(x) for x in d[0].cpu()]
        # oracle logits of the same inputs (both contexts hold every committed token)
        c_t, c_d = o_t.new_cache(), o_d.new_cache()
        o_t.forward(committed[:-1], c_t, logits_rows=np.zeros(0, dtype=np.int64))
        o_d.forward(committed[:-1], c_d, logits_rows=np.zeros(0, dtype=np.int64))
        ref_t = o_t.forward([committed[-1]] + drafts, c_t)
        ref_d = o_d.forward([committed[-1]] + drafts[:-1], c_d)
        assert np.max(np.abs(r["logits"][0].cpu().numpy() - ref_t)) < LOGIT_TOL
        assert np.max(np.abs(dl[0].cpu().numpy() - ref_d)) < LOGIT_TOL
        check_rule_on_gpu_logits(d, dl, uds, u, r)
        ref = ov.verify(ref_t, ref_d, np.array(drafts), list(u[0].cpu().numpy()), T, TOP_K, TOP_P)
        a, nxt = int(r["accepted_len"].item()), int(r["next_token"].item())
        if (a, nxt) != (ref["a"], ref["next"]):
            assert ref["margin"] < EDGE_MODEL, (a, nxt, ref["a"], ref["next"], ref["margin"])
            excused += 1
        committed += drafts[:a] + [nxt]
        pending = r["next_token"].clone()
    assert excused <= 1
    target.close()
    draft.close()


@pytest.fixture(scope="module")
def full_models(lib):
    wt = synth.model_weights(synth.QWEN_27B, seed=0, device="cuda")
    wd = synth.model_weights(synth.DRAFT_0P8B, seed=0, device="cuda")
    yield wt, wd
    del wt, wd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("K", [1, 4, 16])
def test_27b_full_rounds_follow_rule(lib, full_models, K):
    wt, wd = full_models
    V = synth.QWEN_27B.vocab
    prompt = torch.from_numpy(synth.prompt_tokens(1, 2048, V)).cuda()
    target = lib.SpecModel(synth.QWEN_27B, wt, max_ctx=2048 + 160, max_k=16, prefill_chunk=256)
    draft = lib.SpecModel(synth.DRAFT_0P8B, wd, max_ctx=2048 + 160, max_k=16, prefill_chunk=256)
    target.prefill(0, prompt[:-1])
    draft.prefill(0, prompt[:-1])
    pending = prompt[-1:].clone()
    gd, g = np.random.Generator(np.random.PCG64(4)), np.random.Generator(np.random.PCG64(2))
    extra = None
    first = None
    for rnd in range(4):
        d, dl, uds, u, r, extra = spec_round(target, draft, pending, K, gd, g, extra)
        check_rule_on_gpu_logits(d, dl, uds, u, r)
        if rnd == 0:
            first = (pending.clone(), d.clone(), r["logits"].clone())
        pending = r["next_token"].clone()
    target.close()
    draft.close()
    # the first verify pass's rows against decode steps of the same tokens
    dec = lib.SpecModel(synth.QWEN_27B, wt, max_ctx=2048 + 160, max_k=16, prefill_chunk=256)
    dec.prefill(0, prompt[:-1])
    p0, d0, lg0 = first
    toks = torch.cat([p0, d0[0]])
    for i in range(K + 1):
        _, lg = dec.decode([0], toks[i:i + 1].contiguous(), want_logits=True)
        assert torch.equal(lg[0], lg0[0, i]), i
    dec.close()

"""GPU parity of the decoder pass, the paged KV cache and the trim, on the tiny float32
configuration (target: 2 layers, d=256, 4/2 heads, head_dim 64, FFN 768, vocab 1024;
draft: 1 layer, d=128, 2/1 heads; weights N(0, 0.02^2) from seed 0).

Bars: logits within 1e-4 of the float64 oracle; greedy tokens equal to the oracle's
(a position whose float64 top-2 gap is below 1e-5 is excused); speculative greedy output
bit-identical to plain greedy on the GPU; after a trim the next pass equals a fresh
prefill of the kept prefix bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import generate as og
from oracle import model as om
from oracle import verify as ov

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model, generate
    return model, generate


@pytest.fixture(scope="module")
def weights():
    wt = synth.model_weights(synth.TINY_TARGET, seed=0)
    wd = synth.model_weights(synth.TINY_DRAFT, seed=0)
    return wt, wd


def make(lib, shape, w, **kw):
    model, _ = lib
    return model.SpecModel(shape, {k: v.cuda() for k, v in w.items()}, **kw)


def test_prefill_logits_match_oracle(lib, weights):
    wt, _ = weights
    m = make(lib, synth.TINY_TARGET, wt, max_ctx=512, prefill_chunk=16)
    prompt = synth.prompt_tokens(1, 64, 1024)
    got = m.prefill(0, torch.from_numpy(prompt).cuda(), want_logits=True).cpu().numpy()
    o = om.Decoder(synth.TINY_TARGET, wt)
    ref = o.forward(prompt, o.new_cache(), logits_rows=[63])[0]
    assert np.max(np.abs(got - ref)) < 1e-4
    m.close()


def test_verify_logits_rows_match_oracle_and_decode_bitwise(lib, weights):
    wt, _ = weights
    m = make(lib, synth.TINY_TARGET, wt, max_ctx=512, max_k=4)
    prompt = synth.prompt_tokens(2, 40, 1024)
    drafts = np.array([[5, 77, 900, 3]], dtype=np.int32)
    m.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    u = torch.full((1, 5), 0.5, device="cuda")
    r = m.verify([0], torch.tensor([prompt[-1]], dtype=torch.int32, device="cuda"), torch.from_numpy(drafts).cuda(),
                 u, 0.0, auto_trim=False, want_logits=True)
    rows = r["logits"][0].cpu().numpy()
    o = om.Decoder(synth.TINY_TARGET, wt)
    ref = o.forward(list(prompt) + list(drafts[0]), o.new_cache())[-5:]
    assert np.max(np.abs(rows - ref)) < 1e-4
    # the same tokens decoded one at a time give bit-identical rows
    m2 = make(lib, synth.TINY_TARGET, wt, max_ctx=512, max_k=4)
    m2.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    seq = [prompt[-1]] + list(drafts[0])
    for i, t in enumerate(seq):
        _, lg = m2.decode([0], torch.tensor([t], dtype=torch.int32, device="cuda"), want_logits=True)
        assert torch.equal(lg[0], r["logits"][0, i]), i
    m.close()
    m2.close()


def test_plain_greedy_matches_oracle(lib, weights):
    _, gen = lib
    wt, _ = weights
    m = make(lib, synth.TINY_TARGET, wt, max_ctx=256)
    prompt = synth.prompt_tokens(1, 64, 1024)
    got = gen.plain_generate(m, torch.from_numpy(prompt), 64).cpu().tolist()
    o = om.Decoder(synth.TINY_TARGET, wt)
    # teacher-forced: the oracle's argmax given the GPU's own prefix
    cache = o.new_cache()
    logits = o.forward(prompt, cache, logits_rows=[63])[0]
    for t, tok in enumerate(got):
        g, gap = ov.argmax_with_gap(logits)
        assert tok == g or gap < 1e-5, (t, tok, g, gap)
        logits = o.forward([tok], cache)[0]
    m.close()


def test_spec_greedy_equals_plain_greedy_bitwise(lib, weights):
    """Tiny fp32 configuration: B=1, prompt 64, K=4, 64 tokens greedy."""
    _, gen = lib
    wt, wd = weights
    prompt = torch.from_numpy(synth.prompt_tokens(1, 64, 1024))
    m = make(lib, synth.TINY_TARGET, wt, max_ctx=256, max_k=4)
    plain = gen.plain_generate(m, prompt, 64).cpu().tolist()
    m.close()
    t = make(lib, synth.TINY_TARGET, wt, max_ctx=256, max_k=4)
    d = make(lib, synth.TINY_DRAFT, wd, max_ctx=256, max_k=4)
    spec, stats = gen.spec_generate(t, d, prompt, 64, K=4)
    assert spec == plain
    # and the oracle's speculative loop gives the same tokens
    ot = om.Decoder(synth.TINY_TARGET, wt)
    od = om.Decoder(synth.TINY_DRAFT, wd)
    ospec, _ = og.spec_generate_greedy(ot, od, prompt.numpy(), 64, K=4)
    assert ospec == spec
    assert stats["steps"] <= 64
    # the target's length equals prompt + emitted tokens - 1 (pending excluded)
    assert t.seq_len(0) == 64 - 1 + stats["accepted"] + stats["steps"]
    t.close()
    d.close()


def test_trim_invariant_bitwise(lib, weights):
    """After a verify pass whose drafts are rejected, the kept cache equals a fresh prefill
    of the kept prefix: the next pass gives the same logits bit for bit."""
    wt, _ = weights
    prompt = synth.prompt_tokens(5, 30, 1024)
    m = make(lib, synth.TINY_TARGET, wt, max_ctx=256, max_k=6)
    m.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    last = torch.tensor([prompt[-1]], dtype=torch.int32, device="cuda")
    # drafts: first = the target's own greedy token, then junk
    g0 = int(m.decode([0], last).item())
    m.reset(0)
    m.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    drafts = torch.tensor([[g0, 1, 2, 3, 4, 5]], dtype=torch.int32, device="cuda")
    r = m.verify([0], last, drafts, torch.full((1, 7), 0.5, device="cuda"), 0.0)
    a = int(r["accepted_len"].item())
    nxt = r["next_token"]
    assert a >= 1
    kept = list(prompt) + [g0] + [int(x) for x in drafts[0, 1:a].tolist()]
    assert m.seq_len(0) == len(kept)
    _, lg = m.decode([0], nxt, want_logits=True)
    f = make(lib, synth.TINY_TARGET, wt, max_ctx=256, max_k=6)
    f.prefill(0, torch.tensor(kept, dtype=torch.int32, device="cuda"))
    _, lg2 = f.decode([0], nxt, want_logits=True)
    assert torch.equal(lg, lg2)
    m.close()
    f.close()


def test_batched_ragged_paged_verify(lib, weights):
    """B=3 slots of different lengths (pages interleaved in the pool), ragged draft_len:
    logits per sequence against the oracle, decisions exact on the GPU's own logits."""
    wt, _ = weights
    m = make(lib, synth.TINY_TARGET, wt, max_batch=4, max_ctx=300, max_k=5, num_pages=80)
    lens = [37, 130, 5]
    prompts = [synth.prompt_tokens(10 + i, n, 1024) for i, n in enumerate(lens)]
    slots = [2, 0, 3]
    for p, s in zip(prompts, slots):
        m.prefill(s, torch.from_numpy(p[:-1]).cuda())
    rng = np.random.default_rng(3)
    drafts = rng.integers(0, 1024, size=(3, 5)).astype(np.int32)
    dlen = np.array([5, 2, 0], dtype=np.int32)
    last = torch.tensor([p[-1] for p in prompts], dtype=torch.int32, device="cuda")
    u = torch.from_numpy(synth.uniforms(7, (3, 6))).cuda()
    r = m.verify(slots, last, torch.from_numpy(drafts).cuda(), u, 1.0, 20, 0.95,
                 draft_len=torch.from_numpy(dlen).cuda(), want_logits=True)
    logits = r["logits"].cpu().numpy()
    o = om.Decoder(synth.TINY_TARGET, wt)
    for b in range(3):
        ref = o.forward(list(prompts[b]) + list(drafts[b]), o.new_cache())[-6:]
        assert np.max(np.abs(logits[b] - ref)) < 1e-4
        kb = int(dlen[b])
        res = ov.verify(logits[b, :kb + 1], None, drafts[b, :kb], list(u[b, :kb].cpu().numpy()) + [u[b, 5].item()],
                        1.0, 20, 0.95)
        if res["margin"] < 1e-6:
            continue
        assert r["accepted_len"][b].item() == res["a"]
        assert r["next_token"][b].item() == res["next"]
    for s, p, b in zip(slots, prompts, range(3)):
        assert m.seq_len(s) == len(p) + int(r["accepted_len"][b].item())
    m.close()


def test_sampling_spec_generate_runs_and_matches_oracle_rule(lib, weights):
    """Sampling mode with a draft model: each verify decision equals the oracle's rule on
    the GPU's own logits (checked inside the loop by re-running one step)."""
    _, gen = lib
    wt, wd = weights
    prompt = torch.from_numpy(synth.prompt_tokens(1, 64, 1024))
    t = make(lib, synth.TINY_TARGET, wt, max_ctx=256, max_k=4)
    d = make(lib, synth.TINY_DRAFT, wd, max_ctx=256, max_k=4)
    out, stats = gen.spec_generate(t, d, prompt, 48, K=4, temperature=1.0, top_k=20, top_p=0.95)
    assert len(out) == 48 and all(0 <= x < 1024 for x in out)
    assert stats["steps"] >= 10
    t.close()
    d.close()


def test_errors_are_reported(lib, weights):
    from speculative_decoding_verify_token_gb300 import _lib
    wt, _ = weights
    m = make(lib, synth.TINY_TARGET, wt, max_batch=2, max_ctx=40, max_k=4)
    with pytest.raises(_lib.SpecError) as e:
        m.verify([0, 0], torch.zeros(2, dtype=torch.int32, device="cuda"), torch.zeros(2, 4, dtype=torch.int32,
                 device="cuda"), torch.zeros(2, 5, device="cuda"))
    assert e.value.code == _lib.SPEC_E_INVAL
    with pytest.raises(_lib.SpecError) as e:
        m.prefill(0, torch.zeros(41, dtype=torch.int32, device="cuda"))
    assert e.value.code == _lib.SPEC_E_RANGE
    m.sync()                        # host-side rejections leave the device status clean
    m.close()

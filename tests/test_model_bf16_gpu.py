"""GPU parity of the bf16 decoder pass on the tensor-core (tcgen05) GEMMs.

A small bf16 model with the 8B-class head geometry (head_dim 128, GQA 2:1) exercises
every GEMM kind (QKV + RoPE + KV append, O + residual, gate/up + SwiGLU, down + residual,
lm_head), split tiles of the stream-K schedule and token tiles of 16..256 columns.
Bars: logits within 3e-2 of the float64 oracle on the bf16-rounded weights; rows of a
verify pass bit-identical to single-token decode rows; greedy tokens equal to the
oracle's unless its top-2 gap is below 1e-2.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from oracle import verify as ov

pytestmark = pytest.mark.gpu
LOGIT_TOL = 3e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model, generate
    return model, generate


@pytest.fixture(scope="module")
def w():
    return synth.model_weights(synth.SMALL_BF16, seed=0)


def make(lib, w, **kw):
    model, _ = lib
    return model.SpecModel(synth.SMALL_BF16, {k: v.cuda() for k, v in w.items()}, **kw)


def test_tensor_core_path_is_used(lib, w):
    m = make(lib, w, max_ctx=512, max_k=4)
    n0 = m.launches()
    m.prefill(0, torch.arange(10, dtype=torch.int32, device="cuda"))
    # one pass of 2 layers: embed + 2 x (4 tensor-core GEMMs with the RMSNorms folded into
    # them + attention splits + attention combine) + advance
    assert m.launches() - n0 == 1 + 2 * 6 + 1
    m.close()


def test_prefill_logits_match_oracle(lib, w):
    m = make(lib, w, max_ctx=512, prefill_chunk=64)
    prompt = synth.prompt_tokens(1, 150, synth.SMALL_BF16.vocab)
    got = m.prefill(0, torch.from_numpy(prompt).cuda(), want_logits=True).cpu().numpy()
    o = om.Decoder(synth.SMALL_BF16, w)
    ref = o.forward(prompt, o.new_cache(), logits_rows=[149])[0]
    err = np.max(np.abs(got - ref))
    assert err < LOGIT_TOL, err
    m.close()


@pytest.mark.parametrize("B,K", [(1, 4), (3, 7), (8, 15), (16, 15), (32, 8), (20, 15)])
def test_verify_rows_match_oracle_and_decode_bitwise(lib, w, B, K):
    V = synth.SMALL_BF16.vocab
    m = make(lib, w, max_batch=B, max_ctx=512, max_k=K)
    dec = make(lib, w, max_batch=B, max_ctx=512, max_k=K)
    prompts = [synth.prompt_tokens(20 + b, 17 + 9 * b, V) for b in range(B)]
    for b, p in enumerate(prompts):
        m.prefill(b, torch.from_numpy(p[:-1]).cuda())
        dec.prefill(b, torch.from_numpy(p[:-1]).cuda())
    drafts = np.random.default_rng(B).integers(0, V, size=(B, K)).astype(np.int32)
    last = torch.tensor([p[-1] for p in prompts], dtype=torch.int32, device="cuda")
    r = m.verify(list(range(B)), last, torch.from_numpy(drafts).cuda(), torch.full((B, K + 1), 0.5, device="cuda"),
                 0.0, auto_trim=False, want_logits=True)
    logits = r["logits"]
    # decode the same tokens one at a time for all B slots together (M = B)
    toks = torch.cat([last[:, None], torch.from_numpy(drafts).cuda()], dim=1)
    for i in range(K + 1):
        _, lg = dec.decode(list(range(B)), toks[:, i].contiguous(), want_logits=True)
        assert torch.equal(lg, logits[:, i]), i
    o = om.Decoder(synth.SMALL_BF16, w)
    for b in (0, B - 1):
        ref = o.forward(list(prompts[b]) + list(drafts[b]), o.new_cache())[-(K + 1):]
        err = np.max(np.abs(logits[b].cpu().numpy() - ref))
        assert err < LOGIT_TOL, (b, err)
    m.close()
    dec.close()


def test_spec_greedy_equals_plain_and_oracle(lib, w):
    _, gen = lib
    V = synth.SMALL_BF16.vocab
    prompt = torch.from_numpy(synth.prompt_tokens(3, 40, V))
    t = make(lib, w, max_ctx=256, max_k=4)
    plain = gen.plain_generate(t, prompt, 48).cpu().tolist()
    t.close()
    t = make(lib, w, max_ctx=256, max_k=4)
    d = make(lib, w, max_ctx=256, max_k=4)     # the target as its own draft: every draft accepted
    spec, stats = gen.spec_generate(t, d, prompt, 48, K=4)
    assert spec == plain
    assert stats["accepted"] >= 4 * (stats["steps"] - 1)
    o = om.Decoder(synth.SMALL_BF16, w)
    cache = o.new_cache()
    logits = o.forward(prompt.numpy(), cache, logits_rows=[39])[0]
    bad = 0
    for tok in plain:
        g, gap = ov.argmax_with_gap(logits)
        if tok != g and gap >= 1e-2:
            bad += 1
        logits = o.forward([tok], cache)[0]
    assert bad == 0
    t.close()
    d.close()


def test_graphs_and_pdl_change_no_bits(lib, w):
    """The decoder pass replayed from a CUDA graph, with programmatic dependent launch, gives
    the same logits bit for bit as eager launches without PDL."""
    from speculative_decoding_verify_token_gb300 import _lib
    V = synth.SMALL_BF16.vocab
    prompt = synth.prompt_tokens(9, 50, V)
    drafts = torch.from_numpy(np.random.default_rng(1).integers(0, V, size=(1, 4)).astype(np.int32)).cuda()
    last = torch.tensor([prompt[-1]], dtype=torch.int32, device="cuda")
    u = torch.full((1, 5), 0.5, device="cuda")
    res = []
    for graphs, pdl in ((0, 0), (1, 1), (1, 0), (0, 1)):
        m = make(lib, w, max_ctx=256, max_k=4)
        m.set_option(_lib.SPEC_OPT_GRAPHS, graphs)
        m.set_option(_lib.SPEC_OPT_PDL, pdl)
        m.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
        outs = []
        for rep in range(3):        # replays of the same graph along a growing context
            r = m.verify([0], last, drafts, u, 0.0, auto_trim=False, want_logits=True)
            outs.append(r["logits"].clone())
        m.sync()                    # no device-side wait gave up
        res.append(outs)
        m.close()
    for outs in res[1:]:
        for a, b in zip(res[0], outs):
            assert torch.equal(a, b)


def test_device_wait_that_runs_out_is_reported(lib, w):
    """A bounded device wait that runs out (the GEMM kernels' wait helper on a barrier that
    nothing completes, no copy in flight) is reported by the next sync as SPEC_E_TIMEOUT,
    stays reported (the context is spent), and leaves the GPU usable: the kernel returned
    after its budget and a fresh context still verifies correctly."""
    import time
    from speculative_decoding_verify_token_gb300 import _lib
    m = make(lib, w, max_batch=1, max_ctx=64, max_k=4)
    m.sync()                                     # nothing has run out yet
    with pytest.raises(_lib.SpecError) as e:
        m.check_wait_timeout(0)                  # budget outside [1, 2000] ms
    assert e.value.code == _lib.SPEC_E_INVAL
    t0 = time.perf_counter()
    m.check_wait_timeout(50)
    with pytest.raises(_lib.SpecError) as e:
        m.sync()
    assert e.value.code == _lib.SPEC_E_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    with pytest.raises(_lib.SpecError) as e:
        m.sync()
    assert e.value.code == _lib.SPEC_E_TIMEOUT
    m.close()
    m2 = make(lib, w, max_batch=1, max_ctx=64, max_k=4)
    p = synth.prompt_tokens(1, 20, synth.SMALL_BF16.vocab)
    m2.prefill(0, torch.from_numpy(p[:-1]).cuda())
    r = m2.verify([0], torch.tensor(p[-1:], dtype=torch.int32, device="cuda"),
                  torch.zeros(1, 4, dtype=torch.int32, device="cuda"), torch.zeros(1, 5, device="cuda"), 0.0,
                  want_logits=True)
    m2.sync()
    g = ov.verify_greedy(r["logits"][0].double().cpu().numpy(), [0, 0, 0, 0])
    assert (int(r["accepted_len"].item()), int(r["next_token"].item())) == (g["a"], g["next"])
    m2.close()


@pytest.mark.parametrize("temperature,graphs", [(0.0, 1), (1.0, 1), (1.0, 0)])
def test_draft_loop_equals_per_token_decodes(lib, w, temperature, graphs):
    """spec_draft's device-resident loop gives the drafts and draft logits of K separate
    decode calls bit for bit (greedy and sampled, two sequences of different lengths, from a
    graph and eagerly), leaves the same KV lengths, and a second call continues the same way."""
    from speculative_decoding_verify_token_gb300 import _lib
    V, K, B = synth.SMALL_BF16.vocab, 5, 2
    prompts = [synth.prompt_tokens(60 + b, 20 + 9 * b, V) for b in range(B)]
    u = torch.from_numpy(synth.uniforms(61, (2, B, K))).cuda()
    res = []
    for mode in ("loop", "calls"):
        m = make(lib, w, max_batch=B, max_ctx=128, max_k=K)
        m.set_option(_lib.SPEC_OPT_GRAPHS, graphs)
        for b, p in enumerate(prompts):
            m.prefill(b, torch.from_numpy(p[:-1]).cuda())
        pend = torch.tensor([int(p[-1]) for p in prompts], dtype=torch.int32, device="cuda")
        outs = []
        for r in range(2):
            if mode == "loop":
                d, lg = m.draft(list(range(B)), pend, K, u[r].contiguous(), temperature, 20, 0.95, want_logits=True)
            else:
                toks, rows = [], []
                tok = pend
                for i in range(K):
                    tok, l1 = m.decode(list(range(B)), tok, u[r, :, i].contiguous(), temperature, 20, 0.95,
                                       want_logits=True)
                    toks.append(tok)
                    rows.append(l1)
                d, lg = torch.stack(toks, 1), torch.stack(rows, 1)
            outs.append((d.clone(), lg.clone()))
            pend = d[:, -1].contiguous()
        m.sync()
        res.append((outs, [m.seq_len(b) for b in range(B)]))
        m.close()
    (lo, ll), (co, cl) = res
    assert ll == cl == [len(p) - 1 + 2 * K for p in prompts]
    for (dl_, gl), (dc, gc) in zip(lo, co):
        assert torch.equal(dl_, dc)
        assert torch.equal(gl, gc)


@pytest.mark.parametrize("B,K", [(1, 4), (3, 7), (8, 15)])
def test_lm_head_fused_greedy_equals_logits_path(lib, w, B, K):
    """Greedy verify without logits keeps only each 128-row lm_head tile's argmax per token
    ([MTP-fixes] "Truncation has to match on both sides": greedy needs the argmax alone)
    and merges them; its decisions, tokens, output distributions and statuses equal the
    full-logits path exactly: drafts that copy 0..K tokens of the greedy continuation, an
    illegal id, ragged draft lengths; and single-token decode."""
    V = synth.SMALL_BF16.vocab
    prompts = [synth.prompt_tokens(70 + b, 23 + 11 * b, V) for b in range(B)]
    seq = list(range(B))
    # the greedy continuation of every prompt (fused decode on a helper context)
    helper = make(lib, w, max_batch=B, max_ctx=256, max_k=K)
    for b, p in enumerate(prompts):
        helper.prefill(b, torch.from_numpy(p[:-1]).cuda())
    tok = torch.tensor([int(p[-1]) for p in prompts], dtype=torch.int32, device="cuda")
    cont = []
    for _ in range(K):
        tok = helper.decode(seq, tok)
        cont.append(tok.clone())
    helper.close()
    cont = torch.stack(cont, dim=1)                                  # [B, K]
    rng = np.random.default_rng(B * 100 + K)
    drafts = cont.clone()
    for b in range(B):
        j = K if b == 0 else int(rng.integers(0, K + 1))             # first j drafts are the argmax
        if j < K:
            drafts[b, j] = int((int(cont[b, j]) + 1 + rng.integers(0, V - 1)) % V)
    if B > 1:
        drafts[1, 0] = V + 5                                         # an illegal id: rejected at once
    dl = torch.tensor([K - (b % 3) for b in range(B)], dtype=torch.int32, device="cuda")
    last = torch.tensor([int(p[-1]) for p in prompts], dtype=torch.int32, device="cuda")
    u = torch.zeros(B, K + 1, dtype=torch.float32, device="cuda")
    outs = []
    for want in (False, True):
        m = make(lib, w, max_batch=B, max_ctx=256, max_k=K)
        for b, p in enumerate(prompts):
            m.prefill(b, torch.from_numpy(p[:-1]).cuda())
        r = m.verify(seq, last, drafts, u, 0.0, draft_len=dl, want_logits=want)
        d = m.decode(seq, r["next_token"].clone(), want_logits=want)
        d_tok = d[0] if want else d
        outs.append(({k: v.cpu() for k, v in r.items() if k != "logits"}, d_tok.cpu(), [m.seq_len(b) for b in seq]))
        m.close()
    (fa, fd, fl), (ra, rd, rl) = outs
    for k in ("accepted_len", "next_token", "out_ids", "out_probs", "status"):
        assert torch.equal(fa[k], ra[k]), (k, fa[k], ra[k])
    assert torch.equal(fd, rd)
    assert fl == rl
    assert int(fa["accepted_len"].sum()) > 0                         # some drafts were accepted

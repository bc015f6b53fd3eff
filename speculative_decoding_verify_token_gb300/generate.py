"""Draft-then-verify loops over the C ABI (host logic; every forward runs in the library).

"Speculative Decoding on Apple Silicon..." section "How speculative decoding works": a
draft model proposes K tokens one at a time, the target checks them in one batched pass,
the agreeing prefix is kept and the first mismatch is replaced by the target's token.

KV bookkeeping per round (both contexts hold every committed token except `pending`):
  * the draft decodes pending, d1, ..., d_{K-1} (K entries) and proposes d1..dK;
  * the target verify pass appends K+1 entries and keeps a+1 of them (auto trim);
  * the draft keeps min(a+1, K) of its K entries; when a == K it still has to ingest
    d_K before the next round.
"""
import numpy as np
import torch


def plain_generate(model, prompt, n_new, seq=0, temperature=0.0, top_k=20, top_p=0.95, uniforms=None):
    """Plain token-by-token decoding; tokens stay on the device (one sync at the end)."""
    dev = model.device
    prompt = prompt.to(dev, torch.int32)
    if prompt.numel() > 1:
        model.prefill(seq, prompt[:-1])
    pending = prompt[-1:].clone()
    out = torch.empty(n_new, dtype=torch.int32, device=dev)
    for t in range(n_new):
        u = None if uniforms is None else uniforms[t:t + 1]
        nxt = model.decode([seq], pending, u, temperature, top_k, top_p)
        out[t:t + 1].copy_(nxt)
        pending = nxt
    return out


def spec_generate(target, draft, prompt, n_new, K, seq=0, temperature=0.0, top_k=20, top_p=0.95, seed=2,
                  draft_seed=4):
    """Speculative generation with a draft model.  Greedy when temperature == 0; otherwise
    the draft samples from its truncated distribution and the target runs rejection
    sampling with the same truncation.  Returns (tokens [n_new] host, stats)."""
    dev = target.device
    prompt = prompt.to(dev, torch.int32)
    if prompt.numel() > 1:
        target.prefill(seq, prompt[:-1])
        draft.prefill(seq, prompt[:-1])
    pending = prompt[-1:].clone()
    g = np.random.Generator(np.random.PCG64(seed))
    gd = np.random.Generator(np.random.PCG64(draft_seed))
    out = []
    steps = accepted = 0
    extra = None
    while len(out) < n_new:
        if extra is not None:
            draft.prefill(seq, extra)
        # the draft's K tokens in one device-resident loop (K decode steps, no host round trip)
        ud = torch.from_numpy(gd.random((1, K), dtype=np.float32)).to(dev)
        d, dl = draft.draft([seq], pending, K, ud, temperature, top_k, top_p, want_logits=temperature > 0)
        u = torch.from_numpy(g.random((1, K + 1), dtype=np.float32)).to(dev)
        r = target.verify([seq], pending, d, u, temperature, top_k, top_p, draft_logits=dl)
        a = int(r["accepted_len"].item())
        nxt = r["next_token"]
        out += d[0, :a].tolist() + [int(nxt.item())]
        steps += 1
        accepted += a
        keep = torch.clamp(r["accepted_len"], max=K - 1)
        draft.kv_trim([seq], K - 1, keep)
        extra = d[0, K - 1:K].clone() if a == K else None
        pending = nxt.clone()
    return out[:n_new], {"steps": steps, "accepted": accepted, "attempted": steps * K}

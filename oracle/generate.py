"""Plain and speculative generation loops (test infrastructure only).

[SD-Apple] "How speculative decoding works": a draft proposes K tokens one at a time,
the target checks them in one batched pass, the agreeing prefix is kept and the first
mismatch is replaced by the target's token.  KV convention used here and by the CUDA
library: before a verify pass the cache holds every committed token except the pending
one; the pass appends K+1 entries (pending token + drafts); the trim keeps
len + a + 1 of them, and the emitted token becomes the new pending one.

Drafters defined here (inputs to the verify step, not part of it):
  * scripted -- copy j tokens of a recorded trajectory, then one token that differs,
    with j ~ Geometric (P(j = n) = (1 - alpha) alpha^n) capped at K;
  * n-gram -- [OptiQ] "N-gram lookup": when the last >= 3 tokens match earlier in the
    context, draft the tokens that followed (longest match of 8 down to 3 tokens, most
    recent occurrence, at most n_draft tokens).
A draft-length gate (DraftGate) picks how many of those tokens to verify each step.

Parity status: pinned -- greedy speculative output equals plain greedy output
([SD-Apple] "Why this needed a patch", [OptiQ] "In float32 the output is identical"),
and the scripted drafter's mean emitted tokens per step against its closed form; the draft
gate's expected tokens against the geometric closed form and brute-force enumeration, and
its decisions on hand-worked cost tables.
"""
import numpy as np

from .verify import verify, sample_token


def plain_generate(model, prompt, n_new, temperature=0.0, top_k=0, top_p=1.0, uniforms=None):
    """Token-by-token decoding of the target alone, the output speculative decoding must
    reproduce under greedy decoding ([SD-Apple] "Why this needed a patch to mlx_lm at all").
    Sampling draws token t from the truncated row with uniforms[t]."""
    cache = model.new_cache()
    logits = model.forward(prompt, cache, logits_rows=[len(prompt) - 1])[0]
    out = []
    for t in range(n_new):
        u = 0.5 if uniforms is None else uniforms[t]
        tok, _ = sample_token(logits, u, temperature, top_k, top_p)
        out.append(tok)
        if t + 1 < n_new:
            logits = model.forward([tok], cache)[0]
    return out


def greedy_trajectory_logits(model, prompt, n_new):
    """Plain greedy decode that also returns every step's logits row."""
    cache = model.new_cache()
    logits = model.forward(prompt, cache, logits_rows=[len(prompt) - 1])[0]
    toks, rows = [], []
    for t in range(n_new):
        rows.append(logits)
        tok = int(np.argmax(logits))
        toks.append(tok)
        if t + 1 < n_new:
            logits = model.forward([tok], cache)[0]
    return toks, rows


def spec_generate_greedy(target, draft, prompt, n_new, K):
    """Greedy speculative generation with a greedy draft model; returns (tokens, stats)."""
    tc, dc = target.new_cache(), draft.new_cache()
    prompt = [int(t) for t in prompt]
    # both caches hold the prompt except its last token, which is pending
    if len(prompt) > 1:
        target.forward(prompt[:-1], tc)
        draft.forward(prompt[:-1], dc)
    pending = prompt[-1]
    out, steps, accepted = [], 0, 0
    while len(out) < n_new:
        # draft K tokens one at a time (the draft cache catches up on committed tokens)
        base = len(tc)
        committed = (prompt + out)
        dc.trim(min(len(dc), base))
        draft_in = committed[len(dc):base] + [pending]
        drafts = []
        for i in range(K):
            lg = draft.forward(draft_in, dc)[-1]
            d = int(np.argmax(lg))
            drafts.append(d)
            draft_in = [d]
        rows = target.forward([pending] + drafts, tc)              # K+1 rows
        r = verify(rows, None, drafts, None, 0.0, 0, 1.0)
        a, nxt = r["a"], r["next"]
        tc.trim(base + a + 1)
        out.extend(drafts[:a] + [nxt])
        pending = nxt
        steps += 1
        accepted += a
    return out[:n_new], {"steps": steps, "accepted": accepted}


def scripted_drafts(trajectory, pos, K, j, wrong_token):
    """Drafts for a verify step whose pending token is trajectory[pos]: the next j tokens
    of the trajectory, then (if j < K) wrong_token(i) != the true token for the rest."""
    out = []
    for i in range(K):
        if i < j:
            out.append(int(trajectory[pos + 1 + i]))
        else:
            out.append(int(wrong_token(i)))
    return out


def ngram_draft(context, n_draft=8, min_match=3, max_match=8):
    """[OptiQ] "N-gram lookup": longest suffix (max_match down to min_match tokens) that
    occurred earlier in context; draft the tokens that followed its most recent earlier
    occurrence, at most n_draft.  Returns [] when nothing matches."""
    ctx = [int(t) for t in context]
    n = len(ctx)
    for m in range(min(max_match, n - 1), min_match - 1, -1):
        suffix = ctx[n - m:]
        for start in range(n - m - 1, -1, -1):      # most recent earlier occurrence
            if ctx[start:start + m] == suffix:
                follow = ctx[start + m:start + m + n_draft]
                if follow:
                    return follow
    return []


class DraftGate:
    """[OptiQ] "N-gram lookup": the draft length of a step follows how often recent drafts
    were accepted, set against the timed cost of a verify pass; long drafts while text is
    copied, none during new prose.

    Reading (the pages give no formula): a drafted token is accepted with probability
    alpha = (S + 1) / (S + F + 2) -- a uniform prior over alpha updated with S accepted draft
    tokens and F first rejections -- where every round first multiplies S and F by `decay`
    (so that alpha drifts back to 1/2 while nothing is drafted, and drafting is retried).
    With acceptance alpha a verify pass over n drafts emits j + 1 tokens when the first j
    drafts are accepted, so its mean is expected_tokens(alpha, n); the gate drafts the
    n <= min(n_max, available) with the largest expected_tokens / cost[n], the smaller n on
    ties."""

    def __init__(self, cost, decay=0.9):
        self.cost = [float(c) for c in cost]
        self.n_max = len(self.cost) - 1
        self.decay = float(decay)
        self.S = 0.0
        self.F = 0.0

    def acceptance(self):
        return (self.S + 1.0) / (self.S + self.F + 2.0)

    @staticmethod
    def expected_tokens(alpha, n):
        """Mean tokens emitted by a verify pass with n drafts: the j accepted drafts plus the
        target's own token, j = n with probability alpha^n, else j < n with probability
        alpha^j (1 - alpha)."""
        total = 0.0
        for j in range(n + 1):
            p = alpha ** j * ((1.0 - alpha) if j < n else 1.0)
            total += p * (j + 1)
        return total

    def scores(self, available):
        lim = max(0, min(self.n_max, int(available)))
        a = self.acceptance()
        return [self.expected_tokens(a, n) / self.cost[n] for n in range(lim + 1)]

    def choose(self, available):
        s = self.scores(available)
        best = 0
        for n in range(1, len(s)):
            if s[n] > s[best]:
                best = n
        return best

    def update(self, drafted, accepted):
        self.S *= self.decay
        self.F *= self.decay
        if drafted > 0:
            self.S += accepted
            if accepted < drafted:
                self.F += 1.0

"""Acceptance rule of speculative decoding, plain float64 (test infrastructure only).

Sources:
  * [MTP-fixes] "The verify was wrong under sampling": accept a drafted token t with
    probability min(1, p(t)/q(t)); on rejection draw a replacement from the clipped,
    renormalised difference max(0, p - q).
  * [MTP-fixes] "Truncation has to match on both sides": p and q are restricted by the
    same sampler -- the top 20 tokens and the top 0.95 of cumulative mass -- before the
    ratio is taken.
  * [Draft] "#2" and "#3": greedy (temperature 0) keeps a drafted token only when it is
    the target's own most likely token; the first disagreement is replaced by the
    target's token and the rest of the draft is discarded, so every target pass emits
    at least one token.
  * [OptiQ] "MTP head": Qwen's production sampler is temperature 1.0, top_p 0.95,
    top_k 20.

Readings where the pages are silent (each is restated in the design notes):
  R1 a full acceptance emits a bonus token drawn from the last target row;
  R2 uniforms u[0..K-1] drive the K acceptance tests, u[K] drives the one final draw;
  R3 top-k first, then top-p on the renormalised top-k mass, keeping a token while the
     mass before it is below top_p (the first token is always kept); top_p >= 1 keeps
     all top-k tokens;
  R4 ties in ranking go to the lower token id (argmax included);
  R5 acceptance is the strict test u < P/Q;
  R6 the final draw is an inverse CDF over the support in ascending token id: the first
     x whose running sum exceeds u * Z;
  R7 a drafted token outside its own truncated draft distribution (Q(d) = 0) is an
     error; a missing draft distribution means a deterministic draft (Q = one-hot).
  R8 the ranking is done on the raw logits (division by a positive temperature keeps
     the order).

Parity status: pinned (closed forms, special cases, brute-force laws, the worked
example of [Draft] "#2", chi-square) -- see tests/test_oracle_verify.py.
"""
import math

import numpy as np


class IllegalDraft(ValueError):
    """A drafted token has zero probability under its own truncated draft distribution."""


def truncated_distribution(logits, temperature, top_k, top_p):
    """Sampling distribution of one row after temperature, top-k and top-p.

    Returns (ids, probs, top_p_margin): ids in ranking order (logit descending, lower
    id first on ties), probs renormalised over the kept tokens (float64), and the
    smallest distance between a cumulative mass the top-p cut compared and top_p
    (inf when no comparison was made).  temperature == 0 gives the one-hot argmax.
    top_k <= 0 means no top-k limit.
    """
    x = np.asarray(logits, dtype=np.float64)
    order = np.argsort(-x, kind="stable")           # R4, R8
    if temperature == 0:
        return order[:1].astype(np.int64), np.ones(1), math.inf
    k = x.size if top_k <= 0 else min(int(top_k), x.size)
    cand = order[:k]
    z = x[cand] / float(temperature)
    e = np.exp(z - z[0])
    p = e / e.sum()
    kept = k
    margin = math.inf
    if top_p < 1.0:                                 # R3
        before = 0.0
        for j in range(k):
            if j > 0:
                margin = min(margin, abs(before - top_p))
                if not before < top_p:
                    kept = j
                    break
            before += p[j]
    keep_p = p[:kept]
    return cand[:kept].astype(np.int64), keep_p / keep_p.sum(), margin


def as_dict(ids, probs):
    return {int(i): float(v) for i, v in zip(ids, probs)}


def inverse_cdf(dist, u):
    """R6: first token (ascending id) whose running sum of weights exceeds u * Z.

    dist maps token id -> non-negative weight (need not sum to one).  Returns
    (token, margin) with margin = min_j |cumsum_j - u Z| / Z.
    """
    ids = sorted(dist)
    w = np.array([dist[i] for i in ids], dtype=np.float64)
    c = np.cumsum(w)
    Z = c[-1]
    target = float(u) * Z
    margin = float(np.min(np.abs(c - target)) / Z)
    for i, ci in zip(ids, c):
        if ci > target:
            return i, margin
    return ids[-1], margin


def argmax_with_gap(logits):
    """Argmax (lower id on ties) and the gap between the two largest logits."""
    x = np.asarray(logits, dtype=np.float64)
    order = np.argsort(-x, kind="stable")
    gap = float(x[order[0]] - x[order[1]]) if x.size > 1 else math.inf
    return int(order[0]), gap


def verify_greedy(target_rows, draft_tokens):
    """[Draft] "#2": keep drafts while each equals the target's argmax on the row before it.

    target_rows [K+1, V]; draft_tokens [K].  Returns dict(a, next, min_gap) where min_gap
    is the smallest top-2 logit gap among the rows that decided the outcome.
    """
    K = len(draft_tokens)
    a = 0
    min_gap = math.inf
    while True:
        g, gap = argmax_with_gap(target_rows[a])
        min_gap = min(min_gap, gap)
        if a < K and int(draft_tokens[a]) == g:
            a += 1
            continue
        return {"a": a, "next": g, "min_gap": min_gap, "final": {g: 1.0}}


def truncate_rows(target_rows, draft_rows, draft_tokens, temperature, top_k, top_p):
    """Truncated target distributions P_1..P_{K+1} (rows 0..K) and draft Q_1..Q_K.

    Both sides go through the same truncation ([MTP-fixes] "Truncation has to match on
    both sides").  Returns (P, Q, margin) with P, Q lists of dicts id -> prob.
    """
    K = len(draft_tokens)
    margin = math.inf
    P = []
    for i in range(K + 1):
        ids, pr, m = truncated_distribution(target_rows[i], temperature, top_k, top_p)
        P.append(as_dict(ids, pr))
        margin = min(margin, m)
    Q = []
    for i in range(K):
        if draft_rows is None:
            Q.append({int(draft_tokens[i]): 1.0})
        else:
            ids, pr, m = truncated_distribution(draft_rows[i], temperature, top_k, top_p)
            Q.append(as_dict(ids, pr))
            margin = min(margin, m)
    return P, Q, margin


def accept_and_resample(P, Q, draft_tokens, u):
    """[MTP-fixes] "The verify was wrong under sampling", on truncated distributions.

    For i = 1..K accept d_i iff u[i-1] < P_i(d_i) / Q_i(d_i); at the first rejection draw
    the next token from max(0, P_i - Q_i) renormalised (P_i itself if that is all zero)
    with u[K]; when all K are accepted draw the bonus token from P_{K+1} with u[K].
    """
    K = len(draft_tokens)
    margin = math.inf
    for i in range(K):                      # draft token d_{i+1} checked against row i
        d = int(draft_tokens[i])
        p = P[i].get(d, 0.0)
        q = Q[i].get(d, 0.0)
        if q == 0.0:
            raise IllegalDraft(f"draft token {d} at position {i} has q = 0")
        ratio = p / q
        margin = min(margin, abs(float(u[i]) - ratio))
        if float(u[i]) < ratio:             # R5: accept with probability min(1, p/q)
            continue
        residual = {x: max(0.0, px - Q[i].get(x, 0.0)) for x, px in P[i].items()}
        Z = sum(residual.values())
        if Z == 0.0:
            residual = dict(P[i])
            Z = 1.0
        residual = {x: w / Z for x, w in residual.items() if w > 0.0}
        nxt, m = inverse_cdf(residual, u[K])
        return {"a": i, "next": nxt, "final": residual, "margin": min(margin, m)}
    nxt, m = inverse_cdf(P[K], u[K])        # R1, R2: bonus token from the last row
    return {"a": K, "next": nxt, "final": P[K], "margin": min(margin, m)}


def verify_sampling(target_rows, draft_rows, draft_tokens, u, temperature, top_k, top_p):
    """Rejection-sampling acceptance with matched truncation, from logits.

    target_rows [K+1, V] logits; draft_rows [K, V] logits or None (deterministic
    drafts, R7); draft_tokens [K]; u [K+1] uniforms.  Returns dict(a, next, final,
    margin): final is the distribution the last token was drawn from (id -> prob),
    margin the smallest distance of any floating-point decision to its boundary
    (acceptance ratio, top-p cut, inverse-CDF step), used to excuse ties.
    """
    P, Q, m0 = truncate_rows(target_rows, draft_rows, draft_tokens, temperature, top_k, top_p)
    r = accept_and_resample(P, Q, draft_tokens, u)
    r["margin"] = min(r["margin"], m0)
    return r


def verify(target_rows, draft_rows, draft_tokens, u, temperature, top_k, top_p):
    if temperature == 0:
        return verify_greedy(target_rows, draft_tokens)
    return verify_sampling(target_rows, draft_rows, draft_tokens, u, temperature, top_k, top_p)


def sample_token(logits, u, temperature, top_k, top_p):
    """Draw one token from the truncated distribution of a row by inverse CDF (R6).

    Returns (token, margin); greedy when temperature == 0 (margin = top-2 gap).
    """
    if temperature == 0:
        return argmax_with_gap(logits)
    ids, pr, m = truncated_distribution(logits, temperature, top_k, top_p)
    tok, m2 = inverse_cdf(as_dict(ids, pr), u)
    return tok, min(m, m2)

"""The 27B-class target at full depth (64 layers) against the float64 oracle, on a sample of
positions: a 256-token prompt and the next 32 greedy tokens, teacher-forced against ONE
oracle forward of prompt + trajectory (the oracle generates each float64 weight tensor on
the CPU when its layer needs it).

* greedy: every GPU token is the oracle's argmax given the GPU's own prefix unless the
  oracle's top-2 gap is below 1e-2 ("What is Speculative Decoding and How Does a Draft
  Model Work?", section "#3": the output is the target's);
* sampling at temperature 1, top-k 20, top-p 0.95 ("Qwen3.5 and Qwen3.6 MTP head reaches
  1.4x on Apple Silicon after three fixes", section "Truncation has to match on both
  sides"): each position's token drawn by the GPU's sampler from its own row with a seeded
  uniform equals the oracle's draw from the float64 row with the same uniform, unless the
  oracle's draw lies within 0.06 of a truncation or inverse-CDF boundary (twice the logit
  tolerance, as in the 2-layer tests);
* logits within 3e-2 max-abs: an expected failure at this depth, for the reason the 8B
  full-depth test gives (the bf16 rounding of keys and values computed with fp32
  accumulation differs from the oracle's on ~0.1% of them, and the difference compounds
  over the layers); the numbers are printed.

The prompt is short because the depth is what is checked here (long contexts are checked
on the 8B shape's first layer); kept in a file collected after the other GPU tests but the
allocation-free entry point's.
"""
import numpy as np
import pytest
import torch

import synth
from synth import fastgen
from oracle import model as om
from oracle import verify as ov

pytestmark = pytest.mark.gpu
LOGIT_TOL = 3e-2
GAP_EXCUSE = 1e-2
EDGE_MODEL = 0.06
T, TOP_K, TOP_P = 1.0, 20, 0.95
P, N = 256, 32
_RES = {}


def run_27b():
    if _RES:
        return _RES
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import model as M
    from speculative_decoding_verify_token_gb300 import verify as sv
    shape = synth.QWEN_27B
    V = shape.vocab
    prompt = synth.prompt_tokens(1, P, V)
    w = synth.model_weights(shape, seed=0, device="cuda")
    m = M.SpecModel(shape, w, max_batch=1, max_ctx=P + N + 16, max_k=4, prefill_chunk=256)
    del w
    m.prefill(0, torch.from_numpy(prompt[:-1]).cuda())
    tok = torch.tensor(prompt[-1:], dtype=torch.int32, device="cuda")
    traj, rows = [], []
    for _ in range(N):
        tok, lg = m.decode([0], tok, want_logits=True)
        rows.append(lg[0].clone())
        traj.append(int(tok.item()))
    gpu_rows = torch.stack(rows)                                            # [N, V] fp32
    u = torch.from_numpy(synth.uniforms(7, N)).cuda()
    sampled = sv.sample_logits(gpu_rows, u, T, TOP_K, TOP_P).cpu().numpy()
    m.sync()
    m.close()
    gpu_rows = gpu_rows.double().cpu().numpy()
    torch.cuda.empty_cache()

    seq = np.concatenate([prompt, np.array(traj, dtype=np.int32)])
    dec = om.Decoder(shape, fastgen.WeightsF64(shape))
    ref = dec.forward(seq[:P + N - 1], dec.new_cache(), logits_rows=np.arange(P - 1, P + N - 1))   # [N, V]
    top2 = np.sort(ref, axis=1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]
    agree = np.argmax(ref, axis=1) == np.array(traj)
    uu = u.cpu().numpy()
    draws = [ov.sample_token(ref[i], float(uu[i]), T, TOP_K, TOP_P) for i in range(N)]
    s_agree = np.array([int(sampled[i]) == d[0] for i, d in enumerate(draws)])
    s_margin = np.array([d[1] for d in draws])
    _RES.update({"greedy_agreement": float(np.mean(agree)),
                 "greedy_unexcused": int(np.sum(~agree & (gap >= GAP_EXCUSE))),
                 "sample_agreement": float(np.mean(s_agree)),
                 "sample_unexcused": int(np.sum(~s_agree & (s_margin >= EDGE_MODEL))),
                 "max_abs_logit_err": float(np.max(np.abs(gpu_rows - ref))),
                 "positions_over_tol": int(np.sum(np.max(np.abs(gpu_rows - ref), axis=1) >= LOGIT_TOL))})
    print("27B full depth, 32 teacher-forced positions:", _RES)
    return _RES


def test_dense_27b_full_depth_greedy_and_sampled_tokens():
    """64 layers: greedy tokens are the oracle's argmax (excused under a 1e-2 top-2 gap), and
    tokens sampled from the truncated rows with shared uniforms are the oracle's draws
    (excused within 0.06 of a boundary)."""
    r = run_27b()
    assert r["greedy_unexcused"] == 0, r
    assert r["sample_unexcused"] == 0, r


@pytest.mark.xfail(strict=False, reason="64-layer logits exceed 3e-2 max-abs against the oracle's bf16-KV "
                   "reading: bf16 keys and values from fp32 accumulation round differently from the oracle's "
                   "on ~0.1% of them, and the difference compounds with depth")
def test_dense_27b_full_depth_logits():
    """64 layers: every teacher-forced position's logits within 3e-2 of the oracle."""
    r = run_27b()
    assert r["max_abs_logit_err"] < LOGIT_TOL, r

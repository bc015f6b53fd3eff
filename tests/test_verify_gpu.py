"""GPU parity of the fused verify kernel (spec_verify_logits / spec_sample_logits) with
the CPU oracle, on seeded synthetic logits.

Bar: accepted lengths and emitted tokens bit-exact (a sequence whose oracle decision lies
within 1e-6 of a boundary -- acceptance ratio, top-p cut or inverse-CDF step -- is
excused), final-distribution ids exact and probabilities within 1e-5 absolute.

The module runs on a created stream, where the per-row pass of the kernel starts while the
streaming pass still runs (programmatic dependent launch); the full-size case also runs on
the legacy default stream, where the two passes serialise.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import verify as ov

pytestmark = pytest.mark.gpu
TOL_P = 1e-5
EDGE = 1e-6


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import verify
    prev = torch.cuda.current_stream()
    torch.cuda.set_stream(torch.cuda.Stream())
    yield verify
    torch.cuda.synchronize()
    torch.cuda.set_stream(prev)


def oracle_drafts(draft, u_draft, T, k, p):
    B, K, V = draft.shape
    out = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            out[b, i] = ov.sample_token(draft[b, i], u_draft[b, i], T, k, p)[0]
    return out


def oracle_batch(target, draft, drafts, u, T, k, p, draft_len=None):
    B, K1, V = target.shape
    K = K1 - 1
    res = []
    for b in range(B):
        kb = K if draft_len is None else int(draft_len[b])
        uu = list(u[b, :kb]) + [u[b, K]]
        dr = None if draft is None else draft[b, :kb]
        try:
            r = ov.verify(target[b, :kb + 1], dr, drafts[b, :kb], uu, T, k, p)
        except ov.IllegalDraft:
            r = {"illegal": True}
        res.append(r)
    return res


def compare(res, out, greedy=False):
    a = out["accepted_len"].cpu().numpy()
    nxt = out["next_token"].cpu().numpy()
    ids = out["out_ids"].cpu().numpy()
    probs = out["out_probs"].cpu().numpy()
    st = out["status"].cpu().numpy()
    excused = 0
    for b, r in enumerate(res):
        if r.get("illegal"):
            assert st[b] == -7 and nxt[b] == -1
            continue
        assert st[b] == 0
        if not greedy and r["margin"] < EDGE:
            excused += 1
            continue
        assert a[b] == r["a"], (b, a[b], r["a"])
        assert nxt[b] == r["next"], (b, nxt[b], r["next"])
        exp_ids = sorted(r["final"])
        n = len(exp_ids)
        assert list(ids[b, :n]) == exp_ids and np.all(ids[b, n:] == -1), (b, ids[b], exp_ids)
        np.testing.assert_allclose(probs[b, :n], [r["final"][i] for i in exp_ids], atol=TOL_P, rtol=0)
        assert np.all(probs[b, n:] == 0)
    return excused


def run_case(sv, seed, B, K, V, T=1.0, k=20, p=0.95, with_q=True, draft_len=None, base_offset=0):
    case = synth.verify_logits_case(seed, B, K, V)
    tgt, dft = case["target"], case["draft"]
    if T == 0:
        drafts = np.argmax(dft, axis=-1).astype(np.int32) if K > 0 else np.zeros((B, 0), np.int32)
        # make roughly half the drafts agree with the target's argmax
        g = np.argmax(tgt[:, :K], axis=-1)
        drafts = np.where(np.random.default_rng(seed).random((B, K)) < 0.7, g, drafts).astype(np.int32)
    elif with_q:
        drafts = oracle_drafts(dft, case["u_draft"], T, k, p)
    else:
        drafts = np.array([[ov.sample_token(tgt[b, i], case["u_draft"][b, i], T, k, p)[0]
                            if (b + i) % 3 else (b * 7 + i) % V for i in range(K)] for b in range(B)],
                          dtype=np.int32).reshape(B, K)
    dev = "cuda"
    if base_offset:
        flat = torch.zeros(tgt.size + base_offset, dtype=torch.float32, device=dev)
        t_dev = flat[base_offset:].view(B, K + 1, V)
        t_dev.copy_(torch.from_numpy(tgt))
    else:
        t_dev = torch.from_numpy(tgt).to(dev)
    d_dev = torch.from_numpy(dft).to(dev) if (with_q and K > 0) else None
    dl = None if draft_len is None else torch.from_numpy(np.asarray(draft_len, np.int32)).to(dev)
    out = sv.verify_logits(t_dev, d_dev, torch.from_numpy(drafts).to(dev), torch.from_numpy(case["u"]).to(dev),
                           T, k, p, draft_len=dl)
    torch.cuda.synchronize()
    res = oracle_batch(tgt, dft if with_q else None, drafts, case["u"], T, k, p, draft_len)
    return res, out


@pytest.mark.parametrize("B,K,V", [(6, 4, 3000), (5, 3, 3001), (3, 1, 20000), (4, 0, 777), (2, 4, 5), (3, 2, 2)])
def test_sampling_parity_small(sv, B, K, V):
    res, out = run_case(sv, 10 + V, B, K, V)
    assert compare(res, out) <= 1


@pytest.mark.parametrize("T,k,p", [(0.5, 20, 0.95), (2.0, 20, 0.95), (1.0, 1, 0.95), (1.0, 32, 1.0), (1.0, 7, 0.5)])
def test_sampling_parity_sampler_settings(sv, T, k, p):
    res, out = run_case(sv, 99, 8, 4, 4099, T, k, p)
    assert compare(res, out) <= 1


@pytest.mark.parametrize("V,off", [(1000, 0), (1001, 1), (70001, 3)])
def test_greedy_parity(sv, V, off):
    res, out = run_case(sv, 5, 7, 4, V, T=0.0, base_offset=off)
    compare(res, out, greedy=True)


def test_deterministic_drafts_and_ragged_lengths(sv):
    res, out = run_case(sv, 7, 9, 5, 12345, with_q=False, draft_len=[0, 1, 2, 3, 4, 5, 5, 3, 0])
    assert compare(res, out) <= 1


def test_unaligned_rows_sampling(sv):
    res, out = run_case(sv, 8, 5, 4, 40003, base_offset=2)
    assert compare(res, out) <= 1


def test_illegal_draft_status(sv):
    B, K, V = 3, 2, 500
    case = synth.verify_logits_case(3, B, K, V)
    tgt, dft = case["target"], case["draft"]
    drafts = oracle_drafts(dft, case["u_draft"], 1.0, 20, 0.95)
    drafts[1, 0] = int(np.argmin(dft[1, 0]))          # outside the draft's top-20
    dev = "cuda"
    out = sv.verify_logits(torch.from_numpy(tgt).to(dev), torch.from_numpy(dft).to(dev),
                           torch.from_numpy(drafts).to(dev), torch.from_numpy(case["u"]).to(dev))
    torch.cuda.synchronize()
    res = oracle_batch(tgt, dft, drafts, case["u"], 1.0, 20, 0.95)
    assert res[1].get("illegal")
    compare(res, out)
    assert out["accepted_len"][1].item() == 0


@pytest.mark.parametrize("default_stream", [False, True])
def test_full_size_standalone_verify_config(sv, default_stream):
    """The standalone-verify workload at full size: B=64, K=4, V=151936, T=1, k=20, p=0.95."""
    side = torch.cuda.current_stream()
    if default_stream:
        torch.cuda.synchronize()
        torch.cuda.set_stream(torch.cuda.default_stream())
    try:
        res, out = run_case(sv, 3, 64, 4, 151936)
    finally:
        torch.cuda.synchronize()
        torch.cuda.set_stream(side)
    assert compare(res, out) <= 2
    a = out["accepted_len"].cpu().numpy()
    assert a.min() >= 0 and a.max() <= 4


def test_repeatable_bitwise(sv):
    B, K, V = 16, 4, 50000
    case = synth.verify_logits_case(4, B, K, V)
    drafts = oracle_drafts(case["draft"], case["u_draft"], 1.0, 20, 0.95)
    args = [torch.from_numpy(x).cuda() for x in (case["target"], case["draft"], drafts, case["u"])]
    ws = sv.verify_workspace(B, K, V)
    first = {k: v.clone() for k, v in sv.verify_logits(*args, workspace=ws).items()}
    for _ in range(5):
        o = sv.verify_logits(*args, workspace=ws)
        for k in first:
            assert torch.equal(first[k], o[k]), k


def test_sample_logits_parity(sv):
    R, V = 40, 30011
    x = synth.verify_logits_case(12, 1, R - 1, V)["target"][0]           # [R, V]
    u = synth.uniforms(13, (R,))
    for T, k, p in ((1.0, 20, 0.95), (0.0, 20, 0.95), (0.7, 5, 0.8)):
        tok = sv.sample_logits(torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda(), T, k, p)
        torch.cuda.synchronize()
        tok = tok.cpu().numpy()
        for r in range(R):
            exp, margin = ov.sample_token(x[r], u[r], T, k, p)
            if T > 0 and margin < EDGE:
                continue
            assert tok[r] == exp, (T, k, p, r)


def test_chi_square_gpu_emitted_law():
    """10^6 sequences on the GPU with the same rows and fresh uniforms: the first emitted
    token follows the truncated target distribution P_1."""
    from scipy import stats
    from speculative_decoding_verify_token_gb300 import verify as svm
    V, K, n = 64, 2, 1 << 20
    rng = np.random.default_rng(31)
    trow = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    drow = (trow[:K] + rng.normal(0, 1.0, size=(K, V))).astype(np.float32)
    dev = "cuda"
    tgt = torch.from_numpy(trow).to(dev).expand(n, K + 1, V).contiguous()
    dft = torch.from_numpy(drow).to(dev).expand(n, K, V).contiguous()
    g = torch.Generator(device=dev).manual_seed(5)
    ud = torch.rand(n * K, device=dev, generator=g)
    drafts = svm.sample_logits(dft.view(n * K, V), ud, 1.0, 20, 0.95).view(n, K)
    u = torch.rand(n, K + 1, device=dev, generator=g)
    out = svm.verify_logits(tgt, dft, drafts, u, 1.0, 20, 0.95)
    torch.cuda.synchronize()
    first = torch.where(out["accepted_len"] > 0, drafts[:, 0], out["next_token"]).cpu().numpy()
    P1 = ov.as_dict(*ov.truncated_distribution(trow[0], 1.0, 20, 0.95)[:2])
    counts = np.bincount(first, minlength=V).astype(np.float64)
    exp = np.array([P1.get(x, 0.0) for x in range(V)]) * n
    m = exp > 0
    assert counts[~m].sum() == 0
    assert stats.chisquare(counts[m], exp[m]).pvalue > 1e-4
    # acceptance rate of the first draft = sum_x min(P_1, Q_1)
    Q1 = ov.as_dict(*ov.truncated_distribution(drow[0], 1.0, 20, 0.95)[:2])
    alpha = sum(min(P1.get(x, 0.0), q) for x, q in Q1.items())
    rate = (out["accepted_len"] > 0).float().mean().item()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / n) + 1e-4


def test_row_without_finite_logit(sv):
    """A sequence whose target rows are all -inf: sampling has nothing to draw the final
    token from (status SPEC_E_INVAL, next token -1, no final distribution); greedy takes
    the lowest id (argmax ties go to the lower id).  The other sequences keep their oracle
    results, and the sampler does the same per row."""
    B, K, V = 3, 3, 5000
    case = synth.verify_logits_case(21, B, K, V)
    tgt, dft = case["target"].copy(), case["draft"]
    tgt[1] = -np.inf
    drafts = oracle_drafts(dft, case["u_draft"], 1.0, 20, 0.95)
    args = [torch.from_numpy(x).cuda() for x in (tgt, dft, drafts, case["u"])]
    out = sv.verify_logits(*args, 1.0, 20, 0.95)
    torch.cuda.synchronize()
    assert out["status"][1].item() == -1 and out["next_token"][1].item() == -1
    assert torch.all(out["out_ids"][1] == -1)
    keep = [0, 2]
    res = oracle_batch(tgt[keep], dft[keep], drafts[keep], case["u"][keep], 1.0, 20, 0.95)
    compare(res, {k: v[keep] for k, v in out.items()})
    g = sv.verify_logits(*args, 0.0, 20, 0.95)
    torch.cuda.synchronize()
    a1 = int(np.argmax(drafts[1] != 0)) if np.any(drafts[1] != 0) else K
    assert g["status"][1].item() == 0 and g["next_token"][1].item() == 0
    assert g["accepted_len"][1].item() == a1
    x = synth.verify_logits_case(22, 1, 3, 3000)["target"][0]
    x[1] = -np.inf
    u = synth.uniforms(23, (4,))
    tok = sv.sample_logits(torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda(), 1.0, 20, 0.95).cpu().numpy()
    assert tok[1] == -1
    for r in (0, 2, 3):
        exp, margin = ov.sample_token(x[r], u[r], 1.0, 20, 0.95)
        assert margin < EDGE or tok[r] == exp
    tok0 = sv.sample_logits(torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda(), 0.0, 20, 0.95).cpu().numpy()
    assert tok0[1] == 0

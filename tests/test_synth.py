"""The seeded inputs follow their stated recipes (CPU only).

* standalone-verify logits: fp32 N(0, 3^2), one spike per row of height 8 + Gumbel(0, 1)
  drawn per side, the draft row i sharing target row i's spike token;
* prompts: uniform token ids; uniforms: fp32 in [0, 1);
* n-gram prompts: spans of U[8, 64] tokens, 40% of them copied from earlier in the
  sequence (seen here as the share of trigrams that occurred before, on a vocabulary
  large enough that fresh tokens almost never repeat one);
* every generator returns the same values for the same seed.
"""
import numpy as np

import synth


def test_verify_logits_recipe():
    B, K, V = 64, 4, 20000
    c = synth.verify_logits_case(3, B, K, V)
    t, d, s = c["target"], c["draft"], c["spikes"]
    assert t.shape == (B, K + 1, V) and d.shape == (B, K, V) and s.shape == (B, K + 1)
    assert t.dtype == np.float32 and d.dtype == np.float32
    assert c["u"].shape == (B, K + 1) and c["u_draft"].shape == (B, K)
    off = np.ones(t.shape, bool)
    off[np.arange(B)[:, None], np.arange(K + 1)[None, :], s] = False
    n = off.sum()
    assert abs(t[off].mean()) < 4 * 3.0 / np.sqrt(n)
    assert abs(t[off].std() - 3.0) < 0.01 and abs(d.std() - 3.0) < 0.01
    # spike height: N(0, 9) noise + 8 + Gumbel(0, 1) (mean 8 + Euler's gamma, variance 9 + pi^2/6)
    h = t[np.arange(B)[:, None], np.arange(K + 1)[None, :], s].ravel()
    se = np.sqrt((9.0 + np.pi ** 2 / 6.0) / h.size)
    assert abs(h.mean() - (8.0 + np.euler_gamma)) < 4 * se
    # draft row i carries target row i's spike token, with its own Gumbel height
    hd = d[np.arange(B)[:, None], np.arange(K)[None, :], s[:, :K]].ravel()
    assert abs(hd.mean() - (8.0 + np.euler_gamma)) < 4 * np.sqrt((9.0 + np.pi ** 2 / 6.0) / hd.size)
    assert not np.array_equal(hd, t[np.arange(B)[:, None], np.arange(K)[None, :], s[:, :K]].ravel())
    for u in (c["u"], c["u_draft"]):
        assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0


def test_prompts_and_uniforms():
    V = 1000
    p = synth.prompt_tokens(1, 200000, V)
    assert p.dtype == np.int32 and p.min() == 0 and p.max() == V - 1
    counts = np.bincount(p, minlength=V)
    exp = p.size / V
    chi2 = np.sum((counts - exp) ** 2 / exp)
    assert chi2 < V + 6 * np.sqrt(2 * V)                 # chi-square with V - 1 degrees of freedom
    u = synth.uniforms(2, (100000,))
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005


def test_ngram_prompt_copied_spans():
    for seed in (5, 6):
        p = synth.ngram_prompt(seed, 20000, 1_000_000)
        assert p.dtype == np.int32 and p.size == 20000
        seen, rep = set(), 0
        for i in range(2, p.size):
            tri = (int(p[i - 2]), int(p[i - 1]), int(p[i]))
            rep += tri in seen
            seen.add(tri)
        # 40% of spans (mean length 36) copied; the first two tokens of a copied span start
        # no repeated trigram: about 0.4 * (1 - 2/36) = 0.378
        assert 0.33 < rep / (p.size - 2) < 0.42
        assert synth.ngram_prompt(seed, 2000, 50).tolist() == synth.ngram_prompt(seed, 2000, 50).tolist()


def test_generators_are_seeded():
    a, b = synth.verify_logits_case(7, 2, 2, 300), synth.verify_logits_case(7, 2, 2, 300)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["target"], synth.verify_logits_case(8, 2, 2, 300)["target"])
    assert np.array_equal(synth.prompt_tokens(1, 50, 99), synth.prompt_tokens(1, 50, 99))
    assert np.array_equal(synth.uniforms(2, (3, 4)), synth.uniforms(2, (3, 4)))


def test_c_weight_generator_matches_torch_generator():
    """The C generator behind the float64 oracle copies of large models gives the torch
    generator's values bit for bit (bf16 and fp32 models, several tensors and offsets)."""
    from synth import fastgen
    for shape, name in ((synth.QWEN_8B, "layers.3.wk"), (synth.SMALL_BF16, "lm_head"),
                        (synth.TINY_TARGET, "layers.1.wg"), (synth.DRAFT_0P8B, "layers.0.wo")):
        ref = synth.model_weight(shape, name).double().numpy()
        got = fastgen.model_weight_f64(shape, name)
        assert got.shape == ref.shape
        assert np.array_equal(got, ref), (shape.name, name)
    key = synth.tensor_key(5, "x", "y")
    ref = synth.normal_tensor(key, (3, 1000), 0.5, dtype=__import__("torch").float32).double().numpy()
    buf = np.empty(5000)
    assert np.array_equal(fastgen.normal_f64(key, (3, 1000), 0.5, bf16=False, out=buf), ref)


def test_oracle_weight_providers_match_generator():
    """The on-demand float64 providers the oracle reads large models through give the
    generator's values: gathered embedding rows (repeats, any order) and whole tensors
    through a reused buffer."""
    from synth import fastgen
    s = synth.SMALL_BF16
    w = fastgen.WeightsF64(s)
    ref = synth.model_weight(s, "embed").double().numpy()
    idx = np.array([[5, 7, 5], [4095, 0, 7]])
    assert np.array_equal(w("embed")[idx], ref[idx])
    for name in ("layers.1.wd", "layers.0.wo", "layers.0.wq", "lm_head"):
        assert np.array_equal(w(name), synth.model_weight(s, name).double().numpy()), name
    assert np.array_equal(w("layers.0.attn_norm"), np.ones(s.d_model))

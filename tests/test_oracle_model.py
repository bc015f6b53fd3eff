"""Pins of the oracle decoder: library routines, closed forms and invariants."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as om


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(0)
    S, T, Hq, Hkv, hd = 37, 6, 8, 2, 16
    q = rng.normal(size=(T, Hq, hd))
    k = rng.normal(size=(S, Hkv, hd))
    v = rng.normal(size=(S, Hkv, hd))
    pos = np.arange(S - T, S)
    got = om.causal_gqa_attention(q, k, v, pos)
    qt = torch.tensor(q).permute(1, 0, 2)[None]                     # [1, Hq, T, hd]
    kt = torch.tensor(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
    vt = torch.tensor(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
    mask = torch.tensor(np.arange(S)[None, :] <= pos[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_rmsnorm_closed_forms():
    x = np.array([[3.0, 4.0]])
    np.testing.assert_allclose(om.rmsnorm(x, np.ones(2), 0.0), x / np.sqrt(12.5))
    c = np.full((1, 64), -2.5)
    np.testing.assert_allclose(om.rmsnorm(c, np.full(64, 0.5), 0.0), np.full((1, 64), -0.5))


def test_rope_identity_rotation_and_relative_position():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(1, 3, 8))
    np.testing.assert_allclose(om.rope(x, [0], 1e6), x)
    # one frequency pair is a plain 2-D rotation by pos * theta^0 = pos radians
    y = np.array([[[1.0, 0.0]]])
    np.testing.assert_allclose(om.rope(y, [2.0], 1e6), [[[np.cos(2.0), np.sin(2.0)]]], atol=1e-15)
    r = om.rope(np.repeat(x, 5, 0), np.arange(5) * 17, 1e4)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(np.repeat(x, 5, 0), axis=-1))
    q = rng.normal(size=(1, 1, 16))
    k = rng.normal(size=(1, 1, 16))
    dots = [np.sum(om.rope(q, [m + s], 1e4) * om.rope(k, [n + s], 1e4))
            for (m, n, s) in ((9, 4, 0), (9, 4, 31), (9, 4, 1000))]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


@pytest.fixture(scope="module")
def tiny():
    w = synth.model_weights(synth.TINY_TARGET, seed=0)
    return om.Decoder(synth.TINY_TARGET, w)


def test_incremental_equals_full_forward(tiny):
    toks = synth.prompt_tokens(1, 12, tiny.s.vocab)
    full = tiny.forward(toks, tiny.new_cache())
    c = tiny.new_cache()
    inc = [tiny.forward(toks[:5], c)]
    for t in toks[5:]:
        inc.append(tiny.forward([t], c))
    np.testing.assert_allclose(np.concatenate(inc), full, rtol=1e-10, atol=1e-12)


def test_trim_invariant(tiny):
    """After trimming rejected entries the next pass equals a fresh prefill of the prefix."""
    a = list(synth.prompt_tokens(2, 10, tiny.s.vocab))
    rejected = [5, 6, 7]
    nxt = [11, 12]
    c = tiny.new_cache()
    tiny.forward(a + rejected, c)
    c.trim(len(a))
    got = tiny.forward(nxt, c)
    ref = tiny.forward(a + nxt, tiny.new_cache())[-2:]
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_zero_blocks_reduce_to_embedding_readout():
    s = synth.TINY_TARGET
    w = {k: om.to_f64(v) for k, v in synth.model_weights(s, seed=3).items()}
    for l in range(s.n_layers):
        w[f"layers.{l}.wo"] = np.zeros_like(w[f"layers.{l}.wo"])
        w[f"layers.{l}.wd"] = np.zeros_like(w[f"layers.{l}.wd"])
    m = om.Decoder(s, w)
    toks = [3, 99, 500]
    got = m.forward(toks, m.new_cache())
    e = w["embed"][toks]
    ref = (e / np.sqrt(np.mean(e * e, axis=-1, keepdims=True) + s.rms_eps)) @ w["lm_head"].T
    np.testing.assert_allclose(got, ref, rtol=1e-12)


def test_generator_reproducible_and_distribution():
    s = synth.TINY_DRAFT
    a = synth.model_weight(s, "layers.0.wq", seed=0)
    b = synth.model_weight(s, "layers.0.wq", seed=0)
    c = synth.model_weight(s, "layers.0.wq", seed=1)
    assert torch.equal(a, b) and not torch.equal(a, c)
    big = synth.normal_tensor(synth.tensor_key(0, "x", "y"), (1 << 20,), 1.0, dtype=torch.float32)
    assert abs(big.mean().item()) < 5e-3 and abs(big.std().item() - 1.0) < 5e-3
    # chunking does not change values
    small_chunks = synth.normal_tensor(synth.tensor_key(0, "x", "y"), (1 << 12,), 1.0,
                                       dtype=torch.float32, chunk=1000)
    assert torch.equal(small_chunks, big[:1 << 12])


def test_round_bf16_ties_and_library():
    """Nearest bfloat16 with ties to even: hand-worked cases at 1 (spacing 2^-7), then the
    same rounding as torch's float32 -> bfloat16 conversion on float32 values."""
    r = om.round_bf16
    assert r(1.0 + 2.0 ** -8) == 1.0                               # tie, even mantissa below
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6               # tie, even mantissa above
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7      # just above the tie
    assert r(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert r(0.0) == 0.0 and r(3.0) == 3.0 and r(1.0 / 3.0) == 0.333984375
    x = np.random.default_rng(5).standard_normal(100000).astype(np.float32) * 7.0
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(r(x.astype(np.float64)), ref)


def test_bf16_shape_caches_rounded_keys():
    """A bf16 model's cache holds bf16 keys and values; the float32 model's does not."""
    s = synth.SMALL_BF16
    w = {n: synth.model_weight(s, n) for n in synth.weight_names(s)}
    o = om.Decoder(s, w)
    c = o.new_cache()
    o.forward([1, 2, 3], c, logits_rows=np.zeros(0, dtype=np.int64))
    assert np.array_equal(c.k[0], om.round_bf16(c.k[0])) and np.array_equal(c.v[1], om.round_bf16(c.v[1]))
    t = synth.TINY_TARGET
    o32 = om.Decoder(t, synth.model_weights(t))
    c32 = o32.new_cache()
    o32.forward([1, 2, 3], c32)
    assert not np.array_equal(c32.k[0], om.round_bf16(c32.k[0]))

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



def test_f64_kv_reading_keeps_unrounded_keys():
    """kv="f64" skips the bf16 rounding of keys and values and nothing else: the cache holds
    keys that are not all bf16 values, rounding them gives the default cache exactly, the
    incremental forward still equals the full one, and the logits move by far less than
    the 3e-2 logit tolerance but not by nothing."""
    s = synth.SMALL_BF16
    w = {n: synth.model_weight(s, n) for n in synth.weight_names(s)}
    toks = synth.prompt_tokens(3, 9, s.vocab)
    o16, o64 = om.Decoder(s, w), om.Decoder(s, w, kv="f64")
    c16, c64 = o16.new_cache(), o64.new_cache()
    l16 = o16.forward(toks, c16)
    l64 = o64.forward(toks, c64)
    assert not np.array_equal(c64.k[0], om.round_bf16(c64.k[0]))
    np.testing.assert_array_equal(om.round_bf16(c64.k[0]), c16.k[0])
    np.testing.assert_array_equal(om.round_bf16(c64.v[0]), c16.v[0])
    d = np.max(np.abs(l16 - l64))
    assert 0 < d < 1e-2, d
    c = o64.new_cache()
    inc = np.concatenate([o64.forward(toks[:4], c)] + [o64.forward([t], c) for t in toks[4:]])
    np.testing.assert_allclose(inc, l64, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("kv", ["model", "f64"])
def test_first_layer_cache_builder_equals_forward(kv):
    """append_first_layer_kv builds the cache forward() builds on a one-layer model: the rows
    of a verify pass after it equal the same rows of one forward over the whole sequence."""
    import dataclasses
    s = dataclasses.replace(synth.SMALL_BF16, n_layers=1)
    w = {n: synth.model_weight(synth.SMALL_BF16, n) for n in synth.weight_names(s)}
    o = om.Decoder(s, w, kv=kv)
    toks = synth.prompt_tokens(4, 40, s.vocab)
    full_cache = o.new_cache()
    full = o.forward(toks, full_cache)
    c = o.new_cache()
    o.append_first_layer_kv(toks[:30], c)
    o.append_first_layer_kv(toks[30:35], c)
    rows = o.forward(toks[35:], c)
    np.testing.assert_array_equal(c.k[0], full_cache.k[0])
    np.testing.assert_array_equal(c.v[0], full_cache.v[0])
    np.testing.assert_allclose(rows, full[35:], rtol=0, atol=1e-12)


# ---- hand-worked closed forms of the layer ----------------------------------------------

def test_rope_pairs_and_frequencies():
    """head_dim 4, theta 1e4: dimension j pairs with j + 2 (rotate-half), pair 0 turns by
    the position in radians, pair 1 by position * theta^(-2/4) = position / 100."""
    p = 3.0
    e = np.eye(4).reshape(4, 1, 4)                                   # the four basis vectors
    got = om.rope(e, [p] * 4, 1e4)[:, 0, :]
    c0, s0, c1, s1 = np.cos(p), np.sin(p), np.cos(p / 100), np.sin(p / 100)
    ref = np.array([[c0, 0, s0, 0],
                    [0, c1, 0, s1],
                    [-s0, 0, c0, 0],
                    [0, -s1, 0, c1]])
    np.testing.assert_allclose(got, ref, atol=1e-15)


def test_rmsnorm_epsilon_inside_the_root_and_gains():
    x = np.array([[3.0, 4.0]])                                      # mean square 12.5
    np.testing.assert_allclose(om.rmsnorm(x, np.array([2.0, -1.0]), 0.5), [[6 / np.sqrt(13), -4 / np.sqrt(13)]],
                               rtol=1e-15)


def _layer_shape(d, hq, hkv, hd, f, v):
    return synth.ModelShape("closed-form", 1, d, hq, hkv, hd, f, v, rope_theta=1e4, rms_eps=0.0, dtype="f32")


def test_two_token_attention_closed_form():
    """d = 2, one head of dimension 2 (one RoPE pair turning 1 rad per position), identity
    projections, no FFN.  Token 0 = (1, 0) at position 0, token 1 = (0, 1) at position 1.
    Normed: h0 = (sqrt2, 0), h1 = (0, sqrt2).  Token 0 sees itself: x0 = (1 + sqrt2, 0).
    Token 1: q1 = k1 = R(1) h1 = sqrt2 (-sin 1, cos 1), v1 = h1 (values are not rotated);
    scores (scale 1/sqrt2) are q1.k0 = -sqrt2 sin 1 and q1.k1 = sqrt2, so the weight on
    key 1 is w = 1 / (1 + exp(-sqrt2 (1 + sin 1))) and x1 = (sqrt2 (1 - w), 1 + sqrt2 w).
    The logits (final norm, identity head) are x / rms(x)."""
    s = _layer_shape(2, 1, 1, 2, 2, 2)
    I2 = np.eye(2)
    z = np.zeros((2, 2))
    w = {"embed": I2, "lm_head": I2, "final_norm": np.ones(2), "layers.0.attn_norm": np.ones(2),
         "layers.0.ffn_norm": np.ones(2), "layers.0.wq": I2, "layers.0.wk": I2, "layers.0.wv": I2,
         "layers.0.wo": I2, "layers.0.wg": z, "layers.0.wu": z, "layers.0.wd": z}
    m = om.Decoder(s, w)
    got = m.forward([0, 1], m.new_cache())
    r2 = np.sqrt(2.0)
    wk1 = 1.0 / (1.0 + np.exp(-r2 * (1.0 + np.sin(1.0))))
    x0 = np.array([1.0 + r2, 0.0])
    x1 = np.array([r2 * (1.0 - wk1), 1.0 + r2 * wk1])
    ref = np.stack([x / np.sqrt(np.mean(x * x)) for x in (x0, x1)])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_single_token_layer_closed_form():
    """One token at position 0 (attention over one key returns its value, whatever W_q and
    W_k are).  d = 4, two q heads sharing one kv head of dimension 2, F = 4, vocabulary 3.
    e = (1, -1, 1, -1) has mean square 1, so h = e; v = (h_0, h_2) = (1, 1), both q heads
    read it, and W_o = diag(-2, 2, 0, 0) adds (-2, 2, 0, 0): x1 = (-1, 1, 1, -1) = h2 (its
    mean square is 1).  Gate W_g = ln3 I, up W_u = I: silu(+ln3) = (3/4) ln3 and
    silu(-ln3) = -(1/4) ln3, so silu(gate) * up = ln3 (1/4, 3/4, 3/4, 1/4).  W_d is the
    cyclic shift (row i reads column i + 1): x2 = x1 + ln3 (3/4, 3/4, 1/4, 1/4).  The head
    sums dimensions 1 and 2 into the middle logit."""
    s = _layer_shape(4, 2, 1, 2, 4, 3)
    rng = np.random.default_rng(9)
    L = np.log(3.0)
    wd = np.roll(np.eye(4), 1, axis=1)                    # wd[i, (i + 1) % 4] = 1
    lm = np.array([[1.0, 0, 0, 0], [0, 1, 1, 0], [0, 0, 0, 1]])
    w = {"embed": np.array([[1.0, -1, 1, -1], [0.0, 0, 0, 0], [0.0, 0, 0, 0]]), "lm_head": lm,
         "final_norm": np.ones(4), "layers.0.attn_norm": np.ones(4), "layers.0.ffn_norm": np.ones(4),
         "layers.0.wq": rng.normal(size=(4, 4)), "layers.0.wk": rng.normal(size=(2, 4)),
         "layers.0.wv": np.array([[1.0, 0, 0, 0], [0, 0, 1, 0]]), "layers.0.wo": np.diag([-2.0, 2, 0, 0]),
         "layers.0.wg": L * np.eye(4), "layers.0.wu": np.eye(4), "layers.0.wd": wd}
    m = om.Decoder(s, w)
    got = m.forward([0], m.new_cache())[0]
    x2 = np.array([-1.0, 1, 1, -1]) + L * np.array([0.75, 0.75, 0.25, 0.25])
    y = x2 / np.sqrt(np.mean(x2 * x2))
    np.testing.assert_allclose(got, [y[0], y[1] + y[2], y[3]], rtol=1e-14, atol=1e-15)

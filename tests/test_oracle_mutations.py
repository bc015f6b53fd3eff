"""Planted mistakes in the oracle: every one must fail at least one of its pins.

Each mutant is the oracle's own source with one plausible mistake written in -- a dropped
term, a flipped comparison, a transposed operand, a wrong index, a wrong reading of the
rule -- loaded as a module of its own and swapped in for the real one (CPU only, inside
this process).  The pins of tests/test_oracle_*.py then run against it, in order, until
one fails; a mutant that passes every pin is a hole in the pins and fails this test.  A
control run with no mistake planted must pass every pin, so that the harness itself is
shown to change nothing.
"""
import functools
import importlib
import inspect
import types

import numpy as np
import pytest

import synth
import test_oracle_generate as tg
import test_oracle_model as tm
import test_oracle_verify as tv
from oracle import brute as ob
from oracle import generate as og
from oracle import model as om
from oracle import verify as ov


# ---- the pins, as plain callables ---------------------------------------------------------

@functools.lru_cache(maxsize=None)
def _tiny_weights(shape_name):
    shape = {"tiny-target": synth.TINY_TARGET, "tiny-draft": synth.TINY_DRAFT}[shape_name]
    return {k: om.to_f64(v) for k, v in synth.model_weights(shape, seed=0).items()}


def _tiny(shape=synth.TINY_TARGET):
    return om.Decoder(shape, _tiny_weights(shape.name))   # om.Decoder as currently swapped in


def verify_pins():
    pins = [tv.test_textbook_softmax_when_untruncated, tv.test_truncation_closed_forms,
            tv.test_ranking_ties_go_to_lower_id, tv.test_top_p_keeps_first_token_always,
            tv.test_inverse_cdf_ascending_ids, tv.test_worked_example_raining_cats_and_dogs,
            tv.test_greedy_prefix_rule, tv.test_top_k_one_reduces_sampling_to_greedy,
            tv.test_draft_equal_to_target_accepts_everything,
            tv.test_disjoint_supports_reject_first_and_draw_from_target, tv.test_illegal_draft_raises,
            tv.test_residual_all_zero_falls_back_to_target, tv.test_acceptance_is_strict,
            tv.test_ratio_uses_the_truncated_draft_distribution]
    for args in ((0, 5, 1, 0, 1.0), (1, 6, 2, 0, 1.0), (2, 7, 3, 0, 1.0), (3, 8, 2, 4, 0.9),
                 (4, 8, 3, 3, 0.8), (5, 4, 4, 0, 1.0)):
        pins.append(functools.partial(tv.test_brute_force_laws, *args))
    return pins


def model_pins():
    return [tm.test_attention_matches_torch_sdpa, tm.test_rmsnorm_closed_forms,
            tm.test_rope_identity_rotation_and_relative_position, tm.test_rope_pairs_and_frequencies,
            tm.test_rmsnorm_epsilon_inside_the_root_and_gains, tm.test_two_token_attention_closed_form,
            tm.test_single_token_layer_closed_form, tm.test_round_bf16_ties_and_library,
            lambda: tm.test_incremental_equals_full_forward(_tiny()),
            lambda: tm.test_trim_invariant(_tiny()),
            tm.test_zero_blocks_reduce_to_embedding_readout, tm.test_bf16_shape_caches_rounded_keys,
            tm.test_f64_kv_reading_keeps_unrounded_keys,
            functools.partial(tm.test_first_layer_cache_builder_equals_forward, "model"),
            functools.partial(tm.test_first_layer_cache_builder_equals_forward, "f64")]


def generate_pins():
    pair = lambda: (_tiny(), _tiny(synth.TINY_DRAFT))
    pins = [tg.test_ngram_draft_definition, tg.test_gate_hand_worked_decisions,
            tg.test_gate_new_prose_then_retry, tg.test_gate_copying_drafts_long,
            lambda: tg.test_spec_greedy_equals_plain_greedy_tiny_config(pair()),
            lambda: tg.test_spec_greedy_with_perfect_draft_accepts_everything(pair()),
            lambda: tg.test_scripted_drafter_accepts_exactly_j_and_matches_closed_form(pair())]
    for alpha in (0.0, 0.5, 0.9, 1.0):
        for n in (0, 1, 4):
            pins.append(functools.partial(tg.test_gate_expected_tokens, alpha, n))
    return pins


PINS = {"oracle.verify": verify_pins, "oracle.model": model_pins, "oracle.generate": generate_pins}


# ---- mutants ------------------------------------------------------------------------------

def _mutant(modname, edits):
    """The module's source with each (old, new) edit applied; every `old` names exactly one
    place, so an edit that no longer matches the oracle fails loudly instead of silently
    planting nothing."""
    real = importlib.import_module(modname)
    src = inspect.getsource(real)
    for old, new in edits:
        assert src.count(old) == 1, f"{modname}: the edit target occurs {src.count(old)} times: {old!r}"
        src = src.replace(old, new)
    m = types.ModuleType(modname)
    m.__package__ = "oracle"
    m.__file__ = real.__file__
    exec(compile(src, f"<mutant of {modname}>", "exec"), m.__dict__)
    return m


def _swap_in(monkeypatch, modname, mutant):
    real = importlib.import_module(modname)
    for name, val in vars(mutant).items():
        if isinstance(val, (types.FunctionType, type)) and getattr(val, "__module__", None) == modname:
            monkeypatch.setattr(real, name, val)
    if modname == "oracle.verify":        # modules that imported names from it
        monkeypatch.setattr(ob, "accept_and_resample", mutant.accept_and_resample)
        monkeypatch.setattr(og, "verify", mutant.verify)
        monkeypatch.setattr(og, "sample_token", mutant.sample_token)


def _first_failing_pin(modname):
    with np.errstate(all="ignore"):
        for pin in PINS[modname]():
            try:
                pin()
            except (Exception, pytest.fail.Exception) as e:   # an assertion, pytest.raises or a crash
                return pin, e
    return None


VERIFY_MUTANTS = [
    ("top-p drops the token that crosses the mass",
     [("                if not before < top_p:", "                if not before + p[j] < top_p:")]),
    ("ranking ties go to the higher id",
     [('    order = np.argsort(-x, kind="stable")           # R4, R8',
       '    order = x.size - 1 - np.argsort(-x[::-1], kind="stable")')]),
    ("argmax ties go to the higher id",
     [('    order = np.argsort(-x, kind="stable")\n    gap',
       '    order = x.size - 1 - np.argsort(-x[::-1], kind="stable")\n    gap')]),
    ("temperature multiplies the logits",
     [("    z = x[cand] / float(temperature)", "    z = x[cand] * float(temperature)")]),
    ("kept tokens not renormalised",
     [("    return cand[:kept].astype(np.int64), keep_p / keep_p.sum(), margin",
       "    return cand[:kept].astype(np.int64), keep_p, margin")]),
    ("top-k keeps one token too many", [("    cand = order[:k]", "    cand = order[:k + 1]")]),
    ("inverse CDF walks descending ids", [("    ids = sorted(dist)", "    ids = sorted(dist, reverse=True)")]),
    ("inverse CDF step not strict", [("        if ci > target:", "        if ci >= target:")]),
    ("greedy compares a draft with the argmax of its own row",
     [("        g, gap = argmax_with_gap(target_rows[a])",
       "        g, gap = argmax_with_gap(target_rows[min(a + 1, K)])")]),
    ("ratio inverted (q / p)", [("        ratio = p / q", "        ratio = q / p if p > 0 else math.inf")]),
    ("acceptance test not strict", [("        if float(u[i]) < ratio:", "        if float(u[i]) <= ratio:")]),
    ("residual not clipped at zero",
     [("        residual = {x: max(0.0, px - Q[i].get(x, 0.0)) for x, px in P[i].items()}",
       "        residual = {x: px - Q[i].get(x, 0.0) for x, px in P[i].items()}")]),
    ("residual ignores the draft",
     [("        residual = {x: max(0.0, px - Q[i].get(x, 0.0)) for x, px in P[i].items()}",
       "        residual = dict(P[i])")]),
    ("residual is max(0, Q - P)",
     [("        residual = {x: max(0.0, px - Q[i].get(x, 0.0)) for x, px in P[i].items()}",
       "        residual = {x: max(0.0, Q[i].get(x, 0.0) - px) for x, px in P[i].items()}")]),
    ("resample uses the rejected position's uniform",
     [("        nxt, m = inverse_cdf(residual, u[K])", "        nxt, m = inverse_cdf(residual, u[i])")]),
    ("bonus token drawn from the row before the last",
     [("    nxt, m = inverse_cdf(P[K], u[K])", "    nxt, m = inverse_cdf(P[K - 1], u[K])"),
      ('    return {"a": K, "next": nxt, "final": P[K],', '    return {"a": K, "next": nxt, "final": P[K - 1],')]),
    ("illegal draft accepted silently",
     [('            raise IllegalDraft(f"draft token {d} at position {i} has q = 0")', "            q = 1.0")]),
    ("draft token checked against the next target row",
     [("        p = P[i].get(d, 0.0)", "        p = P[min(i + 1, K)].get(d, 0.0)")]),
    ("draft distribution not truncated like the target's",
     [("            ids, pr, m = truncated_distribution(draft_rows[i], temperature, top_k, top_p)",
       "            ids, pr, m = truncated_distribution(draft_rows[i], temperature, 0, 1.0)")]),
]

MODEL_MUTANTS = [
    ("epsilon outside the square root",
     [("    return x / np.sqrt(ms + eps) * g", "    return x / (np.sqrt(ms) + eps) * g")]),
    ("sum of squares instead of the mean",
     [("    ms = np.mean(x * x, axis=-1, keepdims=True)", "    ms = np.sum(x * x, axis=-1, keepdims=True)")]),
    ("norm gains ignored", [("    return x / np.sqrt(ms + eps) * g", "    return x / np.sqrt(ms + eps)")]),
    ("RoPE pairs adjacent dimensions",
     [("    x1, x2 = x[..., :half], x[..., half:]", "    x1, x2 = x[..., 0::2], x[..., 1::2]")]),
    ("RoPE frequency exponent -j/hd",
     [("    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)",
       "    inv_freq = theta ** (-1.0 * np.arange(half, dtype=np.float64) / hd)")]),
    ("RoPE turns the other way",
     [("[x1 * cos - x2 * sin, x2 * cos + x1 * sin]", "[x1 * cos + x2 * sin, x2 * cos - x1 * sin]")]),
    ("attention scale 1/hd", [("        s = (q[:, h, :] @ kh.T) / np.sqrt(hd)", "        s = (q[:, h, :] @ kh.T) / hd")]),
    ("causal mask excludes the query's own key",
     [("key_pos[None, :] <= np.asarray(q_pos)[:, None]", "key_pos[None, :] < np.asarray(q_pos)[:, None]")]),
    ("q head h reads kv head h mod n_kv",
     [("        kh = k[:, h // group, :]\n        vh = v[:, h // group, :]",
       "        kh = k[:, h % Hkv, :]\n        vh = v[:, h % Hkv, :]")]),
    ("SiLU replaced by the sigmoid", [("    return x / (1.0 + np.exp(-x))", "    return 1.0 / (1.0 + np.exp(-x))")]),
    ("SwiGLU gate and up swapped",
     [('(silu(h2 @ w(p + "wg").T) * (h2 @ w(p + "wu").T))', '(silu(h2 @ w(p + "wu").T) * (h2 @ w(p + "wg").T))')]),
    ("FFN norm taken before the attention residual",
     [('            x = x + o.reshape(T, s.q_dim) @ w(p + "wo").T\n'
       '            h2 = rmsnorm(x, w(p + "ffn_norm"), s.rms_eps)',
       '            h2 = rmsnorm(x, w(p + "ffn_norm"), s.rms_eps)\n'
       '            x = x + o.reshape(T, s.q_dim) @ w(p + "wo").T')]),
    ("RoPE not applied to the keys", [("            k = rope(k, pos, s.rope_theta)\n", "")]),
    ("RoPE applied to the values too",
     [("            k = rope(k, pos, s.rope_theta)\n",
       "            k = rope(k, pos, s.rope_theta)\n            v = rope(v, pos, s.rope_theta)\n")]),
    ("attention residual dropped",
     [('            x = x + o.reshape(T, s.q_dim) @ w(p + "wo").T', '            x = o.reshape(T, s.q_dim) @ w(p + "wo").T')]),
    ("FFN residual dropped", [("            x = x + (silu(", "            x = (silu(")]),
    ("final norm missing", [('        hf = rmsnorm(x, w("final_norm"), s.rms_eps)', "        hf = x")]),
    ("lm_head tied to the embedding", [('        return hf @ w("lm_head").T', '        return hf @ w("embed").T')]),
    ("positions ignore the cache",
     [("        pos = len(cache) + np.arange(T)\n        x = w(", "        pos = np.arange(T)\n        x = w(")]),
    ("trim keeps one entry too many",
     [("                self.k[l] = self.k[l][:n]\n                self.v[l] = self.v[l][:n]",
       "                self.k[l] = self.k[l][:n + 1]\n                self.v[l] = self.v[l][:n + 1]")]),
    ("bf16 rounding keeps 7 bits",
     [("    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)", "    return np.ldexp(np.round(np.ldexp(m, 7)), e - 7)")]),
    ("bf16 ties rounded away from zero",
     [("    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)",
       "    return np.ldexp(np.sign(m) * np.floor(np.abs(np.ldexp(m, 8)) + 0.5), e - 8)")]),
    ("bf16 cache keeps unrounded keys", [("            if self.kv_bf16:", "            if False:")]),
    ("float64-KV reading still rounds the cache",
     [('        self.kv_bf16 = shape.dtype == "bf16" and kv == "model"', '        self.kv_bf16 = shape.dtype == "bf16"')]),
    ("first-layer cache builder ignores the cache length",
     [("        pos = len(cache) + np.arange(T)\n        h = rmsnorm(", "        pos = np.arange(T)\n        h = rmsnorm(")]),
    ("first-layer cache builder skips the attention norm",
     [('        h = rmsnorm(w("embed")[tokens], w("layers.0.attn_norm"), s.rms_eps)', '        h = w("embed")[tokens]')]),
    ("first-layer cache builder keeps unrounded keys",
     [("        if self.kv_bf16:\n            k, v = round_bf16(k), round_bf16(v)\n        cache.append(0, k, v)",
       "        cache.append(0, k, v)")]),
    ("first-layer cache builder skips RoPE",
     [('        k = rope((h @ w("layers.0.wk").T).reshape(T, s.n_kv_heads, s.head_dim), pos, s.rope_theta)',
       '        k = (h @ w("layers.0.wk").T).reshape(T, s.n_kv_heads, s.head_dim)')]),
]

GENERATE_MUTANTS = [
    ("speculative loop trims one entry too few", [("        tc.trim(base + a + 1)", "        tc.trim(base + a)")]),
    ("speculative loop emits the rejected draft",
     [("        out.extend(drafts[:a] + [nxt])", "        out.extend(drafts[:a + 1] if a < K else drafts + [nxt])")]),
    ("scripted drafter copies one token too many", [("        if i < j:", "        if i <= j:")]),
    ("n-gram lookup continues the earliest occurrence",
     [("        for start in range(n - m - 1, -1, -1):      # most recent earlier occurrence",
       "        for start in range(0, n - m):")]),
    ("n-gram lookup tries the shortest match first",
     [("    for m in range(min(max_match, n - 1), min_match - 1, -1):",
       "    for m in range(min_match, min(max_match, n - 1) + 1):")]),
    ("draft gate ties go to the longer draft", [("            if s[n] > s[best]:", "            if s[n] >= s[best]:")]),
    ("draft gate prior (S + 1) / (S + F + 1)",
     [("        return (self.S + 1.0) / (self.S + self.F + 2.0)", "        return (self.S + 1.0) / (self.S + self.F + 1.0)")]),
    ("draft gate decays only on rounds with drafts",
     [("        self.S *= self.decay\n        self.F *= self.decay\n        if drafted > 0:\n",
       "        if drafted > 0:\n            self.S *= self.decay\n            self.F *= self.decay\n")]),
    ("expected tokens without the target's own token", [("            total += p * (j + 1)", "            total += p * j")]),
]

CASES = ([("oracle.verify",) + m for m in VERIFY_MUTANTS] + [("oracle.model",) + m for m in MODEL_MUTANTS]
         + [("oracle.generate",) + m for m in GENERATE_MUTANTS])


@pytest.mark.parametrize("modname", sorted(PINS))
def test_control_without_a_mistake_passes_every_pin(monkeypatch, modname):
    _swap_in(monkeypatch, modname, _mutant(modname, []))
    assert _first_failing_pin(modname) is None


@pytest.mark.parametrize("modname,mistake,edits", CASES, ids=[c[1] for c in CASES])
def test_planted_mistake_fails_a_pin(monkeypatch, modname, mistake, edits):
    _swap_in(monkeypatch, modname, _mutant(modname, edits))
    assert _first_failing_pin(modname) is not None, f"no pin of {modname} catches: {mistake}"

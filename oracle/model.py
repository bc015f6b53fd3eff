"""Dense decoder forward in float64 with a per-token KV list (test infrastructure only).

The verify pass of speculative decoding is one batched forward of the target over the
pending token and the K drafts ([SD-Apple] "How speculative decoding works"; [Draft]
"#2": the target checks the drafts "the same way it reads a prompt").  The KV cache of a
plain attention layer is rolled back by slicing off the rejected entries ([SD-Apple]
"Why this needed a patch to mlx_lm at all").

For the bf16 model configurations the KV cache holds keys and values in the model's
dtype: the batched-serving workload keeps them in a paged bf16 cache, and the same cache
holds the keys of the other bf16 models (the pages' bf16 runtimes attend in bf16 too:
mlx-optiq "Speculative decoding on Apple Silicon", section "Assistant drafter: Gemma-4").
Each key and value is rounded to bfloat16 (nearest, ties to even) when it enters the
cache; everything else stays float64.  kv="f64" keeps the cache in float64 as well (the
all-float64 reading, against which the bf16 results are also reported).

The decoder itself is not printed on the pages; it is the plain Llama/Qwen-style
reading: x = E[tok]; per layer h = RMSNorm(x), q,k,v = h W_q^T, h W_k^T, h W_v^T,
rotate-half RoPE on q and k at absolute positions, causal GQA softmax attention with
scale 1/sqrt(head_dim) (q head h reads kv head h // (n_q/n_kv)), x += attn W_o^T,
h2 = RMSNorm(x), x += (silu(h2 W_g^T) * (h2 W_u^T)) W_d^T; logits = RMSNorm(x) W_lm^T.
RMSNorm(x) = g * x / sqrt(mean(x^2) + eps).  RoPE pairs dims (j, j + hd/2) with
inverse frequency theta^(-2j/hd).

Parity status: pinned -- attention against torch's scaled_dot_product_attention
(float64, CPU), RMSNorm and RoPE against closed forms and invariants (norm
preservation, relative-position dependence, the pairing and frequencies of head_dim 4),
hand-worked closed forms of a two-token attention layer and a one-token layer through
SwiGLU and the lm_head, incremental decoding against a full forward, the trim invariant,
and the bfloat16 rounding against hand-worked ties and torch's conversion -- see
tests/test_oracle_model.py; tests/test_oracle_mutations.py checks that planted mistakes
fail these pins.
"""
import numpy as np


def to_f64(t):
    """torch tensor (fp32/bf16, any device) or numpy array -> float64 numpy array."""
    if hasattr(t, "detach"):
        return t.detach().to("cpu").float().double().numpy()
    return np.asarray(t, dtype=np.float64)


def rmsnorm(x, g, eps):
    """g * x / sqrt(mean(x^2) + eps) over the last axis.  The pages name Llama/Qwen-style
    models without printing their layers; this is the plain reading of their norm."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x, positions, theta):
    """Rotate-half RoPE on x [T, H, hd] at absolute positions [T] (the plain Llama/Qwen
    reading: dimension j pairs with j + hd/2 and turns by position * theta^(-2j/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]   # [T, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def causal_gqa_attention(q, k, v, q_pos):
    """q [T, Hq, hd] at absolute positions q_pos; k, v [S, Hkv, hd] for positions 0..S-1.

    Query t attends keys 0..q_pos[t] with weights softmax(q.k / sqrt(hd)); q head h reads kv
    head h // (Hq / Hkv).  The K+1 rows of a verify pass are such queries at consecutive
    positions ([Draft] "#2": the target checks the drafts the way it reads a prompt).
    Returns [T, Hq, hd].
    """
    T, Hq, hd = q.shape
    S, Hkv, _ = k.shape
    group = Hq // Hkv
    out = np.empty_like(q)
    key_pos = np.arange(S)
    for h in range(Hq):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        s = (q[:, h, :] @ kh.T) / np.sqrt(hd)                       # [T, S]
        s = np.where(key_pos[None, :] <= np.asarray(q_pos)[:, None], s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


def silu(x):
    """x * sigmoid(x), the gate of the SwiGLU feed-forward of the Llama/Qwen reading."""
    return x / (1.0 + np.exp(-x))


def round_bf16(x):
    """Nearest bfloat16 value (8 significant bits, ties to even), as float64.

    x = m 2^e with 1/2 <= |m| < 1 (frexp); m 2^8 rounded to an integer (half to even)
    keeps 8 significant bits.  Values here are far from bfloat16's range limits.
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


class KVList:
    """Per-layer lists of keys and values [T, Hkv, hd]; trimmed by slicing."""

    def __init__(self, n_layers):
        self.k = [None] * n_layers
        self.v = [None] * n_layers

    def __len__(self):
        return 0 if self.k[0] is None else self.k[0].shape[0]

    def append(self, layer, k, v):
        if self.k[layer] is None:
            self.k[layer], self.v[layer] = k, v
        else:
            self.k[layer] = np.concatenate([self.k[layer], k], axis=0)
            self.v[layer] = np.concatenate([self.v[layer], v], axis=0)

    def trim(self, n):
        """Keep the first n positions (the rejected tail is sliced off)."""
        for l in range(len(self.k)):
            if self.k[l] is not None:
                self.k[l] = self.k[l][:n]
                self.v[l] = self.v[l][:n]


class Decoder:
    """shape: synth.ModelShape; weights: callable name -> float64 array (or a dict);
    kv: "model" (bf16 keys and values for bf16 models) or "f64"."""

    def __init__(self, shape, weights, kv="model"):
        assert kv in ("model", "f64")
        self.s = shape
        self.kv_bf16 = shape.dtype == "bf16" and kv == "model"     # the cache stores the model dtype
        if isinstance(weights, dict):
            cache = {}

            def get(name, _w=weights, _c=cache):
                if name not in _c:
                    v = _w[name]
                    _c[name] = v if hasattr(v, "__getitem__") and not hasattr(v, "shape") else to_f64(v)
                return _c[name]
            self.w = get
        else:
            self.w = weights

    def new_cache(self):
        return KVList(self.s.n_layers)

    def append_first_layer_kv(self, tokens, cache):
        """One-layer models: append the keys and values of `tokens` at positions
        len(cache).. without computing their attention outputs or logits.  A layer's keys
        and values depend only on that layer's input, which for the first layer is the
        embedding, so this is the cache forward() would build; it lets long contexts be set
        up without the O(T^2) attention of every prompt position."""
        s, w = self.s, self.w
        assert s.n_layers == 1
        tokens = np.asarray(tokens, dtype=np.int64)
        T = tokens.size
        pos = len(cache) + np.arange(T)
        h = rmsnorm(w("embed")[tokens], w("layers.0.attn_norm"), s.rms_eps)
        k = rope((h @ w("layers.0.wk").T).reshape(T, s.n_kv_heads, s.head_dim), pos, s.rope_theta)
        v = (h @ w("layers.0.wv").T).reshape(T, s.n_kv_heads, s.head_dim)
        if self.kv_bf16:
            k, v = round_bf16(k), round_bf16(v)
        cache.append(0, k, v)

    def forward(self, tokens, cache, logits_rows=None):
        """Run tokens at positions len(cache).. and append their K/V to cache.

        Returns logits [T, V] (or only the rows listed in logits_rows).
        """
        s, w = self.s, self.w
        tokens = np.asarray(tokens, dtype=np.int64)
        T = tokens.size
        pos = len(cache) + np.arange(T)
        x = w("embed")[tokens]                                            # [T, d]
        for l in range(s.n_layers):
            p = f"layers.{l}."
            h = rmsnorm(x, w(p + "attn_norm"), s.rms_eps)
            q = (h @ w(p + "wq").T).reshape(T, s.n_q_heads, s.head_dim)
            k = (h @ w(p + "wk").T).reshape(T, s.n_kv_heads, s.head_dim)
            v = (h @ w(p + "wv").T).reshape(T, s.n_kv_heads, s.head_dim)
            q = rope(q, pos, s.rope_theta)
            k = rope(k, pos, s.rope_theta)
            if self.kv_bf16:
                k, v = round_bf16(k), round_bf16(v)
            cache.append(l, k, v)
            o = causal_gqa_attention(q, cache.k[l], cache.v[l], pos)
            x = x + o.reshape(T, s.q_dim) @ w(p + "wo").T
            h2 = rmsnorm(x, w(p + "ffn_norm"), s.rms_eps)
            x = x + (silu(h2 @ w(p + "wg").T) * (h2 @ w(p + "wu").T)) @ w(p + "wd").T
        hf = rmsnorm(x, w("final_norm"), s.rms_eps)
        if logits_rows is not None:
            hf = hf[np.asarray(logits_rows)]
        return hf @ w("lm_head").T

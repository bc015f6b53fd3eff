"""Seeded generators.  No arithmetic of the verify method lives here.

Weights use a counter-based generator written with 64-bit integer tensor ops only, so
that the same (seed, tensor name, element index) gives the same value on the CPU and
on a GPU:

* a 64-bit key per tensor = blake2b(seed, model name, tensor name);
* per element i and j in {1, 2, 3}: h_j = splitmix64(key + (3 i + j) * 0x9E3779B97F4A7C15);
* the twelve 16-bit fields k of h_1..h_3 give the Irwin-Hall sum
  n = 2 * sum(k) - 12 * 65535, an integer below 2**24 in magnitude, so exact in fp32;
* value = fp32(n) * fp32(std / 131072), one correctly rounded IEEE multiply, which is
  an approximately normal draw of standard deviation std (twelve uniforms), then
  rounded to bf16 (round-to-nearest-even) for bf16 models.

Prompts, uniforms and synthetic logits come from numpy's PCG64 with fixed seeds.
"""
import hashlib

import numpy as np
import torch

from .shapes import ModelShape, weight_names, weight_shape

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(u):
    """Reinterpret an unsigned 64-bit constant as a signed int64 (torch has no uint64 math)."""
    return u - (1 << 64) if u >= (1 << 63) else u


def _lsr(z, s):
    return torch.bitwise_and(torch.bitwise_right_shift(z, s), (1 << (64 - s)) - 1)


def _splitmix64(z):
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _s64(_M1)
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _s64(_M2)
    return torch.bitwise_xor(z, _lsr(z, 31))


def tensor_key(seed: int, model: str, name: str) -> int:
    h = hashlib.blake2b(f"{seed}/{model}/{name}".encode(), digest_size=8).digest()
    return _s64(int.from_bytes(h, "little"))


def normal_tensor(key: int, shape, std: float, dtype=torch.bfloat16, device="cpu",
                  chunk: int = 1 << 25) -> torch.Tensor:
    """Approximately N(0, std^2) values, bit-identical on every device for the same key."""
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype, device=device)
    scale = torch.tensor(np.float32(std / 131072.0), dtype=torch.float32, device=device)
    for start in range(0, numel, chunk):
        n = min(chunk, numel - start)
        idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
        total = torch.zeros(n, dtype=torch.int64, device=device)
        for j in (1, 2, 3):
            h = _splitmix64((idx * 3 + j) * _s64(_GOLDEN) + key)  # wrapping int64 arithmetic
            for f in range(4):
                total += torch.bitwise_and(_lsr(h, 16 * f) if f else h, 0xFFFF)
        num = (total * 2 - 12 * 65535).to(torch.float32)
        out[start:start + n] = (num * scale).to(dtype)
    return out.view(*shape)


def model_weight(shape: ModelShape, name: str, seed: int = 0, device="cpu", std: float = 0.02):
    dtype = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    shp = weight_shape(shape, name)
    if name.endswith("norm"):
        return torch.ones(shp, dtype=dtype, device=device)
    return normal_tensor(tensor_key(seed, shape.name, name), shp, std, dtype=dtype, device=device)


def model_weights(shape: ModelShape, seed: int = 0, device="cpu", std: float = 0.02):
    return {n: model_weight(shape, n, seed, device, std) for n in weight_names(shape)}


def prompt_tokens(seed: int, n: int, vocab: int) -> np.ndarray:
    return np.random.Generator(np.random.PCG64(seed)).integers(0, vocab, size=n).astype(np.int32)


def uniforms(seed: int, shape) -> np.ndarray:
    """fp32 U(0,1) draws (24-bit resolution, never 1.0)."""
    return np.random.Generator(np.random.PCG64(seed)).random(shape, dtype=np.float32)


def verify_logits_case(seed: int, B: int, K: int, V: int, std: float = 3.0, spike: float = 8.0):
    """Synthetic target/draft logits with a shared spike per row.

    target [B, K+1, V] and draft [B, K, V] are fp32 N(0, std^2).  For each (b, i < K) a
    token s ~ U[0, V) gets +spike + g on both sides, g ~ Gumbel(0, 1) drawn
    independently per side; target row K gets its own spike.  Also returns the
    uniforms used to draw the drafts [B, K] and the verification uniforms [B, K+1].
    """
    g = np.random.Generator(np.random.PCG64(seed))
    target = (g.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(std))
    draft = (g.standard_normal((B, K, V), dtype=np.float32) * np.float32(std))
    spikes = g.integers(0, V, size=(B, K + 1))
    gum_t = -np.log(-np.log(g.random((B, K + 1))))
    gum_d = -np.log(-np.log(g.random((B, K))))
    for b in range(B):
        for i in range(K + 1):
            target[b, i, spikes[b, i]] += np.float32(spike + gum_t[b, i])
            if i < K:
                draft[b, i, spikes[b, i]] += np.float32(spike + gum_d[b, i])
    u_draft = g.random((B, K), dtype=np.float32)
    u_verify = g.random((B, K + 1), dtype=np.float32)
    return {"target": target, "draft": draft, "spikes": spikes.astype(np.int32),
            "u_draft": u_draft, "u": u_verify}


def ngram_prompt(seed: int, n: int, vocab: int, copy_prob: float = 0.4,
                 span_lo: int = 8, span_hi: int = 64) -> np.ndarray:
    """Random tokens in spans of U[span_lo, span_hi] tokens; with probability copy_prob a
    span copies an earlier window of the same sequence instead of drawing new tokens."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < n:
        ln = int(g.integers(span_lo, span_hi + 1))
        if len(out) >= span_lo and g.random() < copy_prob:
            src = int(g.integers(0, len(out) - 1))
            ln = min(ln, len(out) - src)
            out.extend(out[src:src + ln])
        else:
            out.extend(int(t) for t in g.integers(0, vocab, size=ln))
    return np.asarray(out[:n], dtype=np.int32)

"""Decoder shapes of the workloads (dense Llama/Qwen-style decoder, untied lm_head).

The shapes are the ones the speculative-decoding write-ups measure on: a tiny fp32
pair for end-to-end checks, an 8B-class and a 27B-class dense target, and a
0.8B-class draft.  No biases, no QK-norm, RMSNorm gains of one, RoPE theta 1e6.
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    dtype: str = "bf16"          # "f32" or "bf16": storage type of weights and KV

    @property
    def q_dim(self):
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    def n_params(self):
        d, f, v = self.d_model, self.ffn_dim, self.vocab
        per_layer = d * (self.q_dim + 2 * self.kv_dim) + self.q_dim * d + 3 * d * f + 2 * d
        return self.n_layers * per_layer + 2 * v * d + d

    def layer_matrix_params(self):
        d, f = self.d_model, self.ffn_dim
        return d * (self.q_dim + 2 * self.kv_dim) + self.q_dim * d + 3 * d * f

    def kv_bytes_per_token(self):
        esize = 4 if self.dtype == "f32" else 2
        return self.n_layers * 2 * self.kv_dim * esize


TINY_TARGET = ModelShape("tiny-target", 2, 256, 4, 2, 64, 768, 1024, dtype="f32")
TINY_DRAFT = ModelShape("tiny-draft", 1, 128, 2, 1, 64, 384, 1024, dtype="f32")
SMALL_BF16 = ModelShape("small-bf16", 2, 512, 4, 2, 128, 1536, 4096)
QWEN_8B = ModelShape("dense-8b", 36, 4096, 32, 8, 128, 12288, 151936)
QWEN_27B = ModelShape("dense-27b", 64, 5120, 40, 8, 128, 17408, 151936)
DRAFT_0P8B = ModelShape("draft-0.8b", 28, 1024, 16, 8, 128, 3072, 151936)


def weight_names(shape: ModelShape):
    names = ["embed"]
    for l in range(shape.n_layers):
        names += [f"layers.{l}.{n}" for n in
                  ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")]
    names += ["final_norm", "lm_head"]
    return names


def weight_shape(shape: ModelShape, name: str):
    d, f, v = shape.d_model, shape.ffn_dim, shape.vocab
    base = name.split(".")[-1]
    return {
        "embed": (v, d), "lm_head": (v, d), "final_norm": (d,),
        "attn_norm": (d,), "ffn_norm": (d,),
        "wq": (shape.q_dim, d), "wk": (shape.kv_dim, d), "wv": (shape.kv_dim, d),
        "wo": (d, shape.q_dim), "wg": (f, d), "wu": (f, d), "wd": (d, f),
    }[base]

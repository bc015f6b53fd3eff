"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package holds no arithmetic of the speculative-decoding method: it only draws
weights, prompts, uniforms and synthetic logits from fixed seeds.  Both sides of every
parity test take their inputs from here, so that neither side feeds the other.
"""
from .shapes import ModelShape, TINY_TARGET, TINY_DRAFT, SMALL_BF16, QWEN_8B, QWEN_27B, DRAFT_0P8B, weight_names, weight_shape
from .gen import (normal_tensor, model_weights, model_weight, prompt_tokens, uniforms,
                  verify_logits_case, tensor_key, ngram_prompt)

__all__ = [
    "ModelShape", "TINY_TARGET", "TINY_DRAFT", "SMALL_BF16", "QWEN_8B", "QWEN_27B", "DRAFT_0P8B",
    "weight_names", "weight_shape", "normal_tensor", "model_weights", "model_weight",
    "prompt_tokens", "uniforms", "verify_logits_case", "tensor_key", "ngram_prompt",
]

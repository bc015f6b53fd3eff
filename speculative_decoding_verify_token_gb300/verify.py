"""Python binding of the fused verify and sampling calls (argument marshalling only).

Every step runs in the CUDA library; this module checks tensor devices, dtypes and
shapes, allocates outputs and the workspace with PyTorch, and passes raw pointers.
"""
import ctypes

import torch

from . import _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape, name):
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def sampling(temperature, top_k, top_p):
    return _lib.SpecSampling(float(temperature), int(top_k), float(top_p))


def verify_workspace(B, K, V, device="cuda"):
    n = _lib.load().spec_verify_logits_workspace_bytes(B, K, V)
    if n == 0:
        raise ValueError("bad sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def verify_logits(target, draft, draft_tokens, uniforms, temperature=1.0, top_k=20, top_p=0.95,
                  draft_len=None, workspace=None, stream=None, out=None):
    """Fused verify (spec_verify_logits).  target [B, K+1, V] fp32, draft [B, K, V] fp32 or
    None, draft_tokens [B, K] int32, uniforms [B, K+1] fp32.  Returns a dict of device
    tensors: accepted_len [B], next_token [B], out_ids [B, 32], out_probs [B, 32], status [B].
    """
    lib = _lib.load()
    B, K1, V = target.shape
    K = K1 - 1
    _need(target, torch.float32, (B, K + 1, V), "target")
    if draft is not None:
        _need(draft, torch.float32, (B, K, V), "draft")
    _need(draft_tokens, torch.int32, (B, K), "draft_tokens")
    _need(uniforms, torch.float32, (B, K + 1), "uniforms")
    if draft_len is not None:
        _need(draft_len, torch.int32, (B,), "draft_len")
    dev = target.device
    if out is None:
        out = {
            "accepted_len": torch.empty(B, dtype=torch.int32, device=dev),
            "next_token": torch.empty(B, dtype=torch.int32, device=dev),
            "out_ids": torch.empty(B, _lib.SPEC_TOPK_MAX, dtype=torch.int32, device=dev),
            "out_probs": torch.empty(B, _lib.SPEC_TOPK_MAX, dtype=torch.float32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    if workspace is None:
        workspace = verify_workspace(B, K, V, dev)
    s = sampling(temperature, top_k, top_p)
    _lib.check(lib.spec_verify_logits(
        B, K, V, _ptr(target), _ptr(draft), _ptr(draft_tokens), _ptr(draft_len), _ptr(uniforms),
        ctypes.byref(s), _ptr(out["accepted_len"]), _ptr(out["next_token"]), _ptr(out["out_ids"]),
        _ptr(out["out_probs"]), _ptr(out["status"]), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def sample_workspace(R, V, device="cuda"):
    n = _lib.load().spec_sample_logits_workspace_bytes(R, V)
    if n == 0:
        raise ValueError("bad sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def sample_logits(logits, uniforms, temperature=1.0, top_k=20, top_p=0.95, workspace=None,
                  stream=None, out=None):
    """Draw one token per row of logits [R, V] fp32 under the truncated distribution
    (spec_sample_logits).  uniforms [R] fp32.  Returns int32 tokens [R]."""
    lib = _lib.load()
    R, V = logits.shape
    _need(logits, torch.float32, (R, V), "logits")
    _need(uniforms, torch.float32, (R,), "uniforms")
    if out is None:
        out = torch.empty(R, dtype=torch.int32, device=logits.device)
    if workspace is None:
        workspace = sample_workspace(R, V, logits.device)
    s = sampling(temperature, top_k, top_p)
    _lib.check(lib.spec_sample_logits(R, V, _ptr(logits), _ptr(uniforms), ctypes.byref(s), _ptr(out),
                                      _ptr(workspace), workspace.numel(), _stream(stream)))
    return out

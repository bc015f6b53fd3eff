"""Python binding of the model context (spec_create / spec_verify / ...): marshalling only.

A SpecModel owns one spec_ctx bound to a CUDA stream and keeps the borrowed weight
tensors alive.  All tensors are CUDA tensors; seq_ids are host ints.
"""
import ctypes

import numpy as np

import torch

from . import _lib
from .verify import _need, _ptr, sampling


def _ids(seq_ids):
    arr = (ctypes.c_int32 * len(seq_ids))(*[int(s) for s in seq_ids])
    return arr


class SpecModel:
    def __init__(self, shape, weights, max_batch=1, max_ctx=2048, max_k=8, num_pages=0, prefill_chunk=0,
                 stream=None, device="cuda"):
        lib = _lib.load()
        self.lib = lib
        self.shape = shape
        self.device = torch.device(device)
        self.stream = torch.cuda.current_stream(self.device) if stream is None else stream
        dt = _lib.SPEC_BF16 if shape.dtype == "bf16" else _lib.SPEC_F32
        self.tdtype = torch.bfloat16 if dt == _lib.SPEC_BF16 else torch.float32
        cfg = _lib.SpecModelCfg(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                                shape.ffn_dim, shape.vocab, shape.rope_theta, shape.rms_eps, dt)
        lim = _lib.SpecCtxLimits(max_batch, max_ctx, max_k, num_pages, prefill_chunk)
        h = ctypes.c_void_p()
        _lib.check(lib.spec_create(ctypes.byref(cfg), ctypes.byref(lim), ctypes.c_void_p(self.stream.cuda_stream),
                                   ctypes.byref(h)))
        self.h = h
        self.max_batch, self.max_k = max_batch, max_k
        self._weights = {}
        names, ptrs = [], []
        for n, t in weights.items():
            if t.device.type != "cuda" or t.dtype != self.tdtype or not t.is_contiguous():
                raise ValueError(f"weight {n}: need a contiguous {self.tdtype} CUDA tensor")
            self._weights[n] = t
            names.append(n.encode())
            ptrs.append(t.data_ptr())
        carr = (ctypes.c_char_p * len(names))(*names)
        parr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        _lib.check(lib.spec_load_weights(h, carr, parr, len(names)))
        if lib.spec_weights_copied(h):
            # the library keeps its own tile-major copy of the GEMM matrices and reads only
            # the embedding and the norm gains from these tensors from now on
            self._weights = {n: t for n, t in self._weights.items() if n == "embed" or n.endswith("norm")}
        V = shape.vocab
        self.V = V

    def close(self):
        if self.h:
            self.lib.spec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, seq_id, tokens, want_logits=False):
        _need(tokens, torch.int32, (tokens.numel(),), "tokens")
        out = torch.empty(self.V, dtype=torch.float32, device=self.device) if want_logits else None
        _lib.check(self.lib.spec_prefill(self.h, int(seq_id), _ptr(tokens), tokens.numel(), _ptr(out)))
        return out

    def verify(self, seq_ids, last_tokens, draft_tokens, uniforms, temperature=0.0, top_k=20, top_p=0.95,
               draft_logits=None, draft_len=None, auto_trim=True, want_logits=False, out=None):
        B = len(seq_ids)
        K = draft_tokens.shape[1] if draft_tokens is not None else 0
        _need(last_tokens, torch.int32, (B,), "last_tokens")
        if K:
            _need(draft_tokens, torch.int32, (B, K), "draft_tokens")
        _need(uniforms, torch.float32, (B, K + 1), "uniforms")
        if draft_logits is not None:
            _need(draft_logits, torch.float32, (B, K, self.V), "draft_logits")
        if draft_len is not None:
            _need(draft_len, torch.int32, (B,), "draft_len")
        dev = self.device
        if out is None:
            out = {"accepted_len": torch.empty(B, dtype=torch.int32, device=dev),
                   "next_token": torch.empty(B, dtype=torch.int32, device=dev),
                   "out_ids": torch.empty(B, _lib.SPEC_TOPK_MAX, dtype=torch.int32, device=dev),
                   "out_probs": torch.empty(B, _lib.SPEC_TOPK_MAX, dtype=torch.float32, device=dev),
                   "status": torch.empty(B, dtype=torch.int32, device=dev)}
        if want_logits:
            out["logits"] = torch.empty(B, K + 1, self.V, dtype=torch.float32, device=dev)
        s = sampling(temperature, top_k, top_p)
        _lib.check(self.lib.spec_verify(
            self.h, B, _ids(seq_ids), K, _ptr(last_tokens), _ptr(draft_tokens if K else None), _ptr(draft_len),
            _ptr(draft_logits), _ptr(uniforms), ctypes.byref(s), _ptr(out["accepted_len"]), _ptr(out["next_token"]),
            _ptr(out["out_ids"]), _ptr(out["out_probs"]), _ptr(out["status"]), _ptr(out.get("logits")),
            1 if auto_trim else 0))
        return out

    def decode(self, seq_ids, tokens, uniforms=None, temperature=0.0, top_k=20, top_p=0.95, want_logits=False,
               out=None):
        B = len(seq_ids)
        _need(tokens, torch.int32, (B,), "tokens")
        if uniforms is None:
            uniforms = torch.full((B,), 0.5, dtype=torch.float32, device=self.device)
        _need(uniforms, torch.float32, (B,), "uniforms")
        nxt = out if out is not None else torch.empty(B, dtype=torch.int32, device=self.device)
        logits = torch.empty(B, self.V, dtype=torch.float32, device=self.device) if want_logits else None
        s = sampling(temperature, top_k, top_p)
        _lib.check(self.lib.spec_decode(self.h, B, _ids(seq_ids), _ptr(tokens), ctypes.byref(s), _ptr(uniforms),
                                        _ptr(nxt), _ptr(logits)))
        return (nxt, logits) if want_logits else nxt

    def draft(self, seq_ids, tokens, K, uniforms, temperature=0.0, top_k=20, top_p=0.95, want_logits=False):
        """K draft tokens per sequence from this model in one device-resident loop (no host
        round trip between them); returns (drafts [B, K] int32, logits [B, K, V] or None)."""
        B = len(seq_ids)
        _need(tokens, torch.int32, (B,), "tokens")
        _need(uniforms, torch.float32, (B, K), "uniforms")
        out = torch.empty(B, K, dtype=torch.int32, device=self.device)
        logits = torch.empty(B, K, self.V, dtype=torch.float32, device=self.device) if want_logits else None
        s = sampling(temperature, top_k, top_p)
        _lib.check(self.lib.spec_draft(self.h, B, _ids(seq_ids), int(K), _ptr(tokens), ctypes.byref(s), _ptr(uniforms),
                                       _ptr(out), _ptr(logits)))
        return out, logits

    def gate_config(self, cost, decay=0.9):
        """Configure the device draft-length gate: cost[n] = timed cost of a verify pass with n
        drafts (n = 0 .. len(cost) - 1); resets every slot's acceptance record."""
        c = np.ascontiguousarray(np.asarray(cost, dtype=np.float64))
        _lib.check(self.lib.spec_ngram_gate_device_config(self.h, int(c.size - 1),
                                                          c.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                                          float(decay)))

    def gate_update(self, seq_ids, drafted, accepted):
        B = len(seq_ids)
        _need(drafted, torch.int32, (B,), "drafted")
        _need(accepted, torch.int32, (B,), "accepted")
        _lib.check(self.lib.spec_ngram_gate_device_update(self.h, B, _ids(seq_ids), _ptr(drafted), _ptr(accepted)))

    def gate_choose(self, seq_ids, available, out=None):
        B = len(seq_ids)
        _need(available, torch.int32, (B,), "available")
        out = out if out is not None else torch.empty(B, dtype=torch.int32, device=self.device)
        _lib.check(self.lib.spec_ngram_gate_device_choose(self.h, B, _ids(seq_ids), _ptr(available), _ptr(out)))
        return out

    def ngram_draft(self, seq_ids, pending, n_draft=8, min_match=3, max_match=8, cap=None, out=None, gated=False):
        """N-gram drafts on the device from each slot's committed tokens + pending [B]; returns
        (drafts [B, n_draft] int32, draft_len [B] int32), both on the device; gated: the
        device gate picks each draft's length from the available continuation."""
        B = len(seq_ids)
        _need(pending, torch.int32, (B,), "pending")
        if cap is not None:
            _need(cap, torch.int32, (B,), "cap")
        if out is None:
            out = (torch.empty(B, n_draft, dtype=torch.int32, device=self.device),
                   torch.empty(B, dtype=torch.int32, device=self.device))
        _lib.check(self.lib.spec_ngram_draft_device(self.h, B, _ids(seq_ids), _ptr(pending), int(n_draft),
                                                    int(min_match), int(max_match), _ptr(cap), 1 if gated else 0,
                                                    _ptr(out[0]), _ptr(out[1])))
        return out

    def kv_trim(self, seq_ids, K, accepted_len):
        _lib.check(self.lib.spec_kv_trim(self.h, len(seq_ids), _ids(seq_ids), int(K), _ptr(accepted_len)))

    def seq_len(self, seq_id):
        v = ctypes.c_int32()
        _lib.check(self.lib.spec_seq_len(self.h, int(seq_id), ctypes.byref(v)))
        return v.value

    def reset(self, seq_id):
        _lib.check(self.lib.spec_seq_reset(self.h, int(seq_id)))

    def sync(self):
        """Wait for the context's stream; raises SpecError (SPEC_E_TIMEOUT) if a device-side
        wait gave up since the context was created."""
        _lib.check(self.lib.spec_sync(self.h))

    def check_wait_timeout(self, budget_ms=50):
        """Run one bounded device wait that runs out (see spec_check_wait_timeout); the next
        sync() raises SpecError(SPEC_E_TIMEOUT) and the context is spent."""
        _lib.check(self.lib.spec_check_wait_timeout(self.h, int(budget_ms)))

    def launches(self):
        return int(self.lib.spec_kernel_launches(self.h))

    def set_option(self, option, value):
        _lib.check(self.lib.spec_set_option(self.h, int(option), int(value)))

    def profile(self, enable=True):
        _lib.check(self.lib.spec_profile(self.h, 1 if enable else 0))

    def profile_read(self):
        n = _lib.SPEC_PROF_CLASSES
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_longlong * n)()
        by = (ctypes.c_double * n)()
        _lib.check(self.lib.spec_profile_read(self.h, ms, cnt, by))
        return {name: {"ms": ms[i], "launches": cnt[i], "bytes": by[i]}
                for i, name in enumerate(_lib.PROF_CLASS_NAMES)}

"""Host-side n-gram drafter (binding of spec_ngram_* in the C ABI).

"Speculative decoding on Apple Silicon" (mlx-optiq docs), section "N-gram lookup: any
model": when the last tokens of a sequence occurred earlier in it, draft the tokens that
followed the most recent earlier occurrence (longest match first, min_match..max_match
tokens).  The index lives in the library; this module only marshals arguments.
"""
import ctypes

import numpy as np

from . import _lib


class NgramDrafter:
    """Committed tokens of one sequence and their m-gram index."""

    def __init__(self, min_match=3, max_match=8):
        self.lib = _lib.load()
        h = ctypes.c_void_p()
        _lib.check(self.lib.spec_ngram_create(int(min_match), int(max_match), ctypes.byref(h)))
        self.h = h

    def append(self, tokens):
        a = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        _lib.check(self.lib.spec_ngram_append(self.h, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), a.size))

    def draft(self, n_draft):
        out = np.zeros(max(int(n_draft), 1), dtype=np.int32)
        n = self.lib.spec_ngram_draft(self.h, int(n_draft), out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        if n < 0:
            _lib.check(n)
        return out[:n]

    def __len__(self):
        return int(self.lib.spec_ngram_length(self.h))

    def close(self):
        if self.h:
            self.lib.spec_ngram_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def draft_batch(drafters, K):
    """Drafts of several sequences at once: (tokens int32 [B, K] zero-padded, lengths int32 [B])."""
    B = len(drafters)
    toks = np.zeros((B, K), dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    arr = (ctypes.c_void_p * B)(*[d.h.value for d in drafters])
    lib = _lib.load()
    _lib.check(lib.spec_ngram_draft_batch(arr, B, int(K), toks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return toks, lens


class DraftGate:
    """Draft-length gate of one sequence (spec_ngram_gate_*): `cost[n]` is the timed cost of
    a verify pass with n drafted tokens (n = 0 .. n_max)."""

    def __init__(self, cost, decay=0.9):
        self.lib = _lib.load()
        c = np.ascontiguousarray(np.asarray(cost, dtype=np.float64))
        h = ctypes.c_void_p()
        _lib.check(self.lib.spec_ngram_gate_create(int(c.size - 1), c.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                                   float(decay), ctypes.byref(h)))
        self.h = h

    def choose(self, available):
        n = self.lib.spec_ngram_gate_choose(self.h, int(available))
        if n < 0:
            _lib.check(n)
        return n

    def update(self, drafted, accepted):
        _lib.check(self.lib.spec_ngram_gate_update(self.h, int(drafted), int(accepted)))

    def acceptance(self):
        return float(self.lib.spec_ngram_gate_acceptance(self.h))

    def close(self):
        if self.h:
            self.lib.spec_ngram_gate_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

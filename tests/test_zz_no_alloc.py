"""The allocation-free verify entry point (for callers that cannot allocate device memory,
e.g. while a CUDA graph is being captured) gives the same results as the regular entry
point with a caller workspace, on two calls in a row that share its built-in scratch.
Kept in a file collected last."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import verify as ov

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import _lib
    from speculative_decoding_verify_token_gb300 import verify as sv
    lib = _lib.load()
    B, K, V = 16, 4, 40009
    assert lib.spec_verify_logits_workspace_bytes(B, K, V) <= lib.spec_verify_logits_noalloc_max_bytes()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    s = _lib.SpecSampling(1.0, 20, 0.95)
    for seed in (21, 22):           # two calls in a row on the shared scratch
        case = synth.verify_logits_case(seed, B, K, V)
        drafts = np.array([[ov.sample_token(case["draft"][b, i], case["u_draft"][b, i], 1.0, 20, 0.95)[0]
                            for i in range(K)] for b in range(B)], dtype=np.int32)
        tgt = torch.from_numpy(case["target"]).cuda()
        dft = torch.from_numpy(case["draft"]).cuda()
        d = torch.from_numpy(drafts).cuda()
        u = torch.from_numpy(case["u"]).cuda()
        ref = sv.verify_logits(tgt, dft, d, u, 1.0, 20, 0.95)
        out = {k: torch.full_like(v, -9) for k, v in ref.items()}
        rc = lib.spec_verify_logits_noalloc(B, K, V, _ptr(tgt), _ptr(dft), _ptr(d), None, _ptr(u), ctypes.byref(s),
                                            _ptr(out["accepted_len"]), _ptr(out["next_token"]), _ptr(out["out_ids"]),
                                            _ptr(out["out_probs"]), _ptr(out["status"]), stream)
        assert rc == _lib.SPEC_OK, lib.spec_last_error()
        torch.cuda.synchronize()
        for k in ("accepted_len", "next_token", "out_ids", "status"):
            assert torch.equal(out[k], ref[k]), k
        assert torch.max(torch.abs(out["out_probs"] - ref["out_probs"])).item() <= 1e-5


def test_noalloc_rejects_sizes_above_its_scratch():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import _lib
    lib = _lib.load()
    s = _lib.SpecSampling(1.0, 20, 0.95)
    fake = ctypes.c_void_p(256)
    rc = lib.spec_verify_logits_noalloc(4096, 16, 151936, fake, fake, fake, None, fake, ctypes.byref(s), fake, fake,
                                        None, None, None, None)
    assert rc == _lib.SPEC_E_RANGE and b"scratch" in lib.spec_last_error()

"""The C-ABI library loads, exports every function include/*.h declares, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_token_gb300 import _lib
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "spec_verify_logits" in names and len(names) >= 6
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_binding_covers_declarations():
    from speculative_decoding_verify_token_gb300 import _lib
    assert declared_functions() <= set(_lib.SIGNATURES), declared_functions() - set(_lib.SIGNATURES)


def test_host_argument_validation(lib):
    from speculative_decoding_verify_token_gb300 import _lib
    s = _lib.SpecSampling(1.0, 20, 0.95)
    fake = ctypes.c_void_p(256)    # never dereferenced: validation fails first
    null = None
    # bad sizes
    assert lib.spec_verify_logits(0, 4, 100, fake, fake, fake, null, fake, ctypes.byref(s), fake, fake,
                                  null, null, null, fake, 1 << 20, null) == _lib.SPEC_E_INVAL
    assert b"bad sizes" in lib.spec_last_error()
    # top_k out of range with temperature > 0
    bad = _lib.SpecSampling(1.0, 0, 0.95)
    assert lib.spec_verify_logits(2, 4, 100, fake, fake, fake, null, fake, ctypes.byref(bad), fake, fake,
                                  null, null, null, fake, 1 << 20, null) == _lib.SPEC_E_INVAL
    bad = _lib.SpecSampling(1.0, 33, 0.95)
    assert lib.spec_sample_logits(2, 100, fake, fake, ctypes.byref(bad), fake, fake, 1 << 20, null) == _lib.SPEC_E_INVAL
    # negative temperature, NaN temperature
    for t in (-1.0, float("nan")):
        bad = _lib.SpecSampling(t, 20, 0.95)
        assert lib.spec_sample_logits(2, 100, fake, fake, ctypes.byref(bad), fake, fake, 1 << 20, null) == _lib.SPEC_E_INVAL
    # workspace too small
    need = lib.spec_verify_logits_workspace_bytes(2, 4, 100)
    assert need > 0
    assert lib.spec_verify_logits(2, 4, 100, fake, fake, fake, null, fake, ctypes.byref(s), fake, fake,
                                  null, null, null, fake, need - 1, null) == _lib.SPEC_E_NOMEM
    # misaligned workspace
    assert lib.spec_verify_logits(2, 4, 100, fake, fake, fake, null, fake, ctypes.byref(s), fake, fake,
                                  null, null, null, ctypes.c_void_p(260), need, null) == _lib.SPEC_E_INVAL
    # NULL outputs
    assert lib.spec_verify_logits(2, 4, 100, fake, fake, fake, null, fake, ctypes.byref(s), null, fake,
                                  null, null, null, fake, need, null) == _lib.SPEC_E_INVAL
    # K above the maximum
    assert lib.spec_verify_logits_workspace_bytes(1, 65, 100) == 0


def test_workspace_sizes_monotone(lib):
    a = lib.spec_verify_logits_workspace_bytes(64, 4, 151936)
    b = lib.spec_verify_logits_workspace_bytes(64, 8, 151936)
    assert 0 < a < b < 64 << 20
    assert lib.spec_sample_logits_workspace_bytes(8, 1000) > 0


def test_row_count_limits(lib):
    """Sizes whose row count or logits overflow the library's 32-bit row and 40-bit element
    counts are rejected (SPEC_E_RANGE) before anything is launched; the workspace query
    returns 0 for them."""
    from speculative_decoding_verify_token_gb300 import _lib
    s = _lib.SpecSampling(0.0, 1, 1.0)
    fake = ctypes.c_void_p(256)
    for B, K, V in ((1 << 29, 1, 2), (2**31 - 1, 64, 2), (1 << 20, 4, 1 << 20)):
        assert lib.spec_verify_logits_workspace_bytes(B, K, V) == 0
        rc = lib.spec_verify_logits(B, K, V, fake, None, fake, None, fake, ctypes.byref(s), fake, fake,
                                    None, None, None, fake, 1 << 62, None)
        assert rc == _lib.SPEC_E_RANGE and b"too large" in lib.spec_last_error()
        rc = lib.spec_verify_logits_noalloc(B, K, V, fake, None, fake, None, fake, ctypes.byref(s), fake, fake,
                                            None, None, None, None)
        assert rc == _lib.SPEC_E_RANGE
    assert lib.spec_verify_logits_workspace_bytes((1 << 30) // 3 - 1, 1, 2) > 0


def test_context_argument_validation(lib):
    """spec_create rejects shapes and limits the kernels do not support before it allocates
    anything; calls on a NULL context fail with SPEC_E_INVAL."""
    from speculative_decoding_verify_token_gb300 import _lib
    good = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=768, vocab=1024,
                rope_theta=1e6, rms_eps=1e-6, dtype=_lib.SPEC_F32)
    lim = _lib.SpecCtxLimits(1, 128, 4, 0, 0)
    h = ctypes.c_void_p()
    for change in (dict(d_model=260), dict(n_kv_heads=3), dict(head_dim=48), dict(head_dim=512),
                   dict(vocab=1023), dict(vocab=1), dict(d_model=16384), dict(rope_theta=0.0),
                   dict(rms_eps=-1.0), dict(dtype=7), dict(n_layers=0), dict(ffn_dim=100)):
        cfg = _lib.SpecModelCfg(**dict(good, **change))
        assert lib.spec_create(ctypes.byref(cfg), ctypes.byref(lim), None, ctypes.byref(h)) == _lib.SPEC_E_INVAL, change
        assert b"bad model shape" in lib.spec_last_error()
    cfg = _lib.SpecModelCfg(**good)
    for bad in (_lib.SpecCtxLimits(0, 128, 4, 0, 0), _lib.SpecCtxLimits(1, 1, 4, 0, 0),
                _lib.SpecCtxLimits(1, 128, 65, 0, 0), _lib.SpecCtxLimits(1, 128, -1, 0, 0)):
        assert lib.spec_create(ctypes.byref(cfg), ctypes.byref(bad), None, ctypes.byref(h)) == _lib.SPEC_E_INVAL
        assert b"bad limits" in lib.spec_last_error()
    assert lib.spec_create(None, ctypes.byref(lim), None, ctypes.byref(h)) == _lib.SPEC_E_INVAL
    ids = (ctypes.c_int32 * 1)(0)
    s = _lib.SpecSampling(0.0, 1, 1.0)
    fake = ctypes.c_void_p(256)
    assert lib.spec_prefill(None, 0, fake, 4, None) == _lib.SPEC_E_INVAL
    assert lib.spec_verify(None, 1, ids, 4, fake, fake, None, None, fake, ctypes.byref(s), fake, fake,
                           None, None, None, None, 1) == _lib.SPEC_E_INVAL
    assert lib.spec_kv_trim(None, 1, ids, 4, fake) == _lib.SPEC_E_INVAL
    assert lib.spec_set_option(None, _lib.SPEC_OPT_GRAPHS, 1) == _lib.SPEC_E_INVAL
    assert lib.spec_load_weights(None, None, None, 0) == _lib.SPEC_E_INVAL
    assert lib.spec_sync(None) == _lib.SPEC_E_INVAL
    assert lib.spec_check_wait_timeout(None, 50) == _lib.SPEC_E_INVAL
    assert lib.spec_weights_copied(None) == 0
    assert lib.spec_kernel_launches(None) == 0
    lib.spec_destroy(None)


def test_workspace_layout_matches_its_description(lib):
    """The verify workspace is a 4-byte work counter, then per row and 256-element fine block
    a (largest, id) pair of 8 bytes and a second-largest float, each region 256-byte aligned:
    7,152 bytes per row of 151,936 logits (149 blocks of 1,024, four fine blocks each)."""
    a = lambda x: (x + 255) // 256 * 256
    for B, K, V in ((64, 4, 151936), (1, 0, 2), (3, 7, 1025), (16, 15, 4096)):
        rows = B * (2 * K + 1)
        nfb = 4 * ((V + 1023) // 1024)
        assert lib.spec_verify_logits_workspace_bytes(B, K, V) == a(4) + a(rows * nfb * 8) + a(rows * nfb * 4)
    assert 4 * ((151936 + 1023) // 1024) * 12 == 7152
    for R, V in ((1, 2), (8, 151936)):
        assert lib.spec_sample_logits_workspace_bytes(R, V) == a(4) + a(R * 4 * ((V + 1023) // 1024) * 8) \
            + a(R * 4 * ((V + 1023) // 1024) * 4)

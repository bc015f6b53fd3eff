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

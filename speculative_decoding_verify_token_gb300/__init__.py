"""specverify: the verify step of speculative decoding on one GB300 (sm_103a).

The compute path is the CUDA library libspecverify.so (C ABI in include/specverify.h);
this package is its thin Python binding.  Importing a submodule that calls the library
fails loudly when the library has not been built.
"""
from . import _lib

__all__ = ["_lib"]

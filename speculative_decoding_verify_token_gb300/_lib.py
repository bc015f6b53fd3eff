"""ctypes loader of libspecverify.so (the C ABI declared in include/specverify.h).

The library is built in place by ``build.py``; importing the binding without it raises,
so nothing can silently run without the CUDA path.
"""
import ctypes
import os

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_DIR, "libspecverify.so")

c_int = ctypes.c_int
c_i32p = ctypes.c_void_p      # device pointers are passed as plain addresses
c_size = ctypes.c_size_t
c_vp = ctypes.c_void_p

SPEC_OK = 0
SPEC_E_INVAL = -1
SPEC_E_NOMEM = -2
SPEC_E_RANGE = -3
SPEC_E_STATE = -4
SPEC_E_TIMEOUT = -5
SPEC_E_CUDA = -6
SPEC_E_DRAFT = -7
SPEC_TOPK_MAX = 32
SPEC_NGRAM_MAX_MATCH = 8

STATUS_NAMES = {0: "SPEC_OK", -1: "SPEC_E_INVAL", -2: "SPEC_E_NOMEM", -3: "SPEC_E_RANGE",
                -4: "SPEC_E_STATE", -5: "SPEC_E_TIMEOUT", -6: "SPEC_E_CUDA", -7: "SPEC_E_DRAFT"}


class SpecSampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


class SpecError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class SpecModelCfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


class SpecCtxLimits(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int32), ("max_ctx", ctypes.c_int32), ("max_k", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("prefill_chunk", ctypes.c_int32)]


SPEC_OPT_ATTN_L2_AHEAD = 7
SPEC_OPT_GRAPHS = 1
SPEC_OPT_PDL = 2
SPEC_OPT_L2_PREFETCH = 3
SPEC_OPT_GEMM_MIN_FILL = 8
SPEC_OPT_GEMM_MAX_SPLIT = 9
SPEC_PROF_CLASSES = 8
PROF_CLASS_NAMES = ["gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_lm_head", "attention",
                    "verify", "other"]
SPEC_F32 = 0
SPEC_BF16 = 1

# name -> (restype, argtypes)
SIGNATURES = {
    "spec_last_error": (ctypes.c_char_p, []),
    "spec_version": (ctypes.c_char_p, []),
    "spec_verify_logits_workspace_bytes": (c_size, [c_int, c_int, c_int]),
    "spec_verify_logits": (c_int, [c_int, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp,
                                   ctypes.POINTER(SpecSampling), c_vp, c_vp, c_vp, c_vp, c_vp,
                                   c_vp, c_size, c_vp]),
    "spec_verify_logits_noalloc_max_bytes": (c_size, []),
    "spec_verify_logits_noalloc": (c_int, [c_int, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp,
                                           ctypes.POINTER(SpecSampling), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "spec_sample_logits_workspace_bytes": (c_size, [c_int, c_int]),
    "spec_sample_logits": (c_int, [c_int, c_int, c_vp, c_vp, ctypes.POINTER(SpecSampling), c_vp,
                                   c_vp, c_size, c_vp]),
    "spec_create": (c_int, [ctypes.POINTER(SpecModelCfg), ctypes.POINTER(SpecCtxLimits), c_vp,
                            ctypes.POINTER(c_vp)]),
    "spec_load_weights": (c_int, [c_vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(c_vp), c_int]),
    "spec_weights_copied": (c_int, [c_vp]),
    "spec_prefill": (c_int, [c_vp, c_int, c_vp, c_int, c_vp]),
    "spec_verify": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_int, c_vp, c_vp, c_vp, c_vp, c_vp,
                            ctypes.POINTER(SpecSampling), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int]),
    "spec_decode": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_vp, ctypes.POINTER(SpecSampling), c_vp,
                            c_vp, c_vp]),
    "spec_kv_trim": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_int, c_vp]),
    "spec_ngram_draft_device": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_vp, c_int, c_int, c_int, c_vp,
                                        c_int, c_vp, c_vp]),
    "spec_ngram_gate_device_config": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_double), ctypes.c_double]),
    "spec_ngram_gate_device_update": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_vp, c_vp]),
    "spec_ngram_gate_device_choose": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_vp, c_vp]),
    "spec_draft": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32), c_int, c_vp, ctypes.POINTER(SpecSampling), c_vp,
                           c_vp, c_vp]),
    "spec_seq_len": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32)]),
    "spec_seq_reset": (c_int, [c_vp, c_int]),
    "spec_sync": (c_int, [c_vp]),
    "spec_check_wait_timeout": (c_int, [c_vp, c_int]),
    "spec_kernel_launches": (ctypes.c_longlong, [c_vp]),
    "spec_profile": (c_int, [c_vp, c_int]),
    "spec_set_option": (c_int, [c_vp, c_int, c_int]),
    "spec_profile_read": (c_int, [c_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong),
                                  ctypes.POINTER(ctypes.c_double)]),
    "spec_destroy": (None, [c_vp]),
    "spec_ngram_create": (c_int, [c_int, c_int, ctypes.POINTER(c_vp)]),
    "spec_ngram_append": (c_int, [c_vp, ctypes.POINTER(ctypes.c_int32), c_int]),
    "spec_ngram_draft": (c_int, [c_vp, c_int, ctypes.POINTER(ctypes.c_int32)]),
    "spec_ngram_draft_batch": (c_int, [ctypes.POINTER(c_vp), c_int, c_int, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32)]),
    "spec_ngram_length": (c_int, [c_vp]),
    "spec_ngram_destroy": (None, [c_vp]),
    "spec_ngram_gate_create": (c_int, [c_int, ctypes.POINTER(ctypes.c_double), ctypes.c_double, ctypes.POINTER(c_vp)]),
    "spec_ngram_gate_choose": (c_int, [c_vp, c_int]),
    "spec_ngram_gate_update": (c_int, [c_vp, c_int, c_int]),
    "spec_ngram_gate_acceptance": (ctypes.c_double, [c_vp]),
    "spec_ngram_gate_destroy": (None, [c_vp]),
}

_lib = None


def load():
    """Load the shared library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(python speculative_decoding_verify_token_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(code):
    if code != SPEC_OK:
        raise SpecError(code, load().spec_last_error().decode())
    return code

"""The weight generator of gen.normal_tensor in C, for float64 CPU copies of large models.

Same (seed, tensor name, element index) -> value map as gen.normal_tensor, bit for bit
(tests/test_synth.py compares them), about 100x faster than the torch integer ops on the
CPU.  The library is compiled with gcc on first use (or by __graft_entry__.build()) into
synth/_normal_gen.so.  No arithmetic of the verify method lives here.
"""
import concurrent.futures as cf
import ctypes
import os
import subprocess

import numpy as np

from .gen import tensor_key
from .shapes import ModelShape, weight_shape

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "csrc", "normal_gen.c")
_SO = os.path.join(_DIR, "_normal_gen.so")
_lib = None


def build():
    """Compile csrc/normal_gen.c into _normal_gen.so (when missing or older than the source)."""
    if os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O3", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_f64.restype = None
        lib.synth_normal_f64.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                         ctypes.c_int, ctypes.c_void_p]
        _lib = lib
    return _lib


def normal_f64(key: int, shape, std: float, bf16: bool = True, threads: int = None, out=None) -> np.ndarray:
    """float64 copy of gen.normal_tensor(key, shape, std, bf16 or fp32); `out` (a float64
    array of at least that many elements) is filled and reused when given."""
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64) if out is None else out.reshape(-1)[:n]
    scale = float(np.float32(std / 131072.0))
    ukey = key & 0xFFFFFFFFFFFFFFFF
    threads = threads or len(os.sched_getaffinity(0))
    step = max(1 << 20, (n + threads - 1) // threads)
    base = out.ctypes.data

    def run(s0):
        m = min(step, n - s0)
        lib.synth_normal_f64(ukey, s0, m, scale, 1 if bf16 else 0, base + 8 * s0)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(run, range(0, n, step)))
    return out.reshape(shape)


def model_weight_f64(shape: ModelShape, name: str, seed: int = 0, std: float = 0.02, out=None) -> np.ndarray:
    """float64 copy of gen.model_weight(shape, name, seed) (norm gains are ones)."""
    shp = weight_shape(shape, name)
    if name.endswith("norm"):
        return np.ones(shp, dtype=np.float64)
    return normal_f64(tensor_key(seed, shape.name, name), shp, std, bf16=shape.dtype != "f32", out=out)


class EmbedRowsF64:
    """The embedding table of `shape` as float64 rows generated on demand (only the rows an
    index asks for), for the oracle decoder's x = embed[tokens]."""

    def __init__(self, shape: ModelShape, seed: int = 0, std: float = 0.02):
        self.key = tensor_key(seed, shape.name, "embed")
        self.d = shape.d_model
        self.scale = float(np.float32(std / 131072.0))
        self.bf16 = shape.dtype != "f32"

    def __getitem__(self, idx):
        idx = np.asarray(idx, dtype=np.int64)
        uniq, inv = np.unique(idx.reshape(-1), return_inverse=True)
        rows = np.empty((uniq.size, self.d), dtype=np.float64)
        lib = _load()
        for i, r in enumerate(uniq):
            lib.synth_normal_f64(self.key & 0xFFFFFFFFFFFFFFFF, int(r) * self.d, self.d, self.scale,
                                 1 if self.bf16 else 0, rows[i].ctypes.data)
        return rows[inv].reshape(idx.shape + (self.d,))


class WeightsF64:
    """weights(name) -> float64 copy of gen.model_weight(shape, name, seed), generated on the
    CPU one tensor at a time for the oracle decoder (which reads each tensor once, right
    away).  Arrays of one shape share a buffer: a returned array stays valid only until the
    next call for a tensor of the same shape."""

    def __init__(self, shape: ModelShape, seed: int = 0):
        self.shape, self.seed = shape, seed
        self.embed = EmbedRowsF64(shape, seed)
        self.bufs = {}

    def __call__(self, name):
        if name == "embed":
            return self.embed
        shp = weight_shape(self.shape, name)
        if name.endswith("norm"):
            return np.ones(shp, dtype=np.float64)
        buf = self.bufs.get(shp)
        if buf is None:
            buf = self.bufs[shp] = np.empty(int(np.prod(shp)), dtype=np.float64)
        return model_weight_f64(self.shape, name, self.seed, out=buf)

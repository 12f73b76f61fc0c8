"""Seeded synthetic inputs (splitmix64 + Box-Muller), shared by tests and bench.

This module holds none of the quantized-matmul arithmetic; it only draws
numbers.  Seeds follow one scheme so that every workload is reproducible:
weights ``0x5EED0000 + config*16 + matrix``, activations
``0xAC700000 + config*16 + M`` (see ``weight_seed`` / ``act_seed``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libq4synth.so")
_lib = None

# Qwen2.5-7B linear shapes, (N, K) with W[N,K] and y = x @ W^T.
QWEN7B_LINEARS = {
    "q_proj": (3584, 3584),
    "k_proj": (512, 3584),
    "v_proj": (512, 3584),
    "o_proj": (3584, 3584),
    "gate_proj": (18944, 3584),
    "up_proj": (18944, 3584),
    "down_proj": (3584, 18944),
}
QWEN7B_LAYERS = 28
LM_HEAD = (152064, 3584)
WEIGHT_SIGMA = 0.02


def _foreign_binary(path: str) -> bool:
    """True if `path` is an ELF file built for another CPU architecture."""
    import platform
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF" or want is None:
        return False
    return int.from_bytes(head[18:20], "little") != want


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC) or _foreign_binary(_LIB):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_uniform_f64.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_void_p]
        lib.synth_uniform_f64.restype = None
        lib.synth_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_splitmix64.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def weight_seed(config: int, matrix: int) -> int:
    return 0x5EED0000 + config * 16 + matrix


def act_seed(config: int, m: int) -> int:
    return 0xAC700000 + config * 16 + m


def normal(seed: int, shape, sigma: float = 1.0, mean: float = 0.0, offset: int = 0,
           out: np.ndarray | None = None) -> np.ndarray:
    """fp32 array of N(mean, sigma^2) deviates from stream ``seed``."""
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = int(np.prod(shape)) if shape else 1
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_f32(seed & (2**64 - 1), offset, n, mean, sigma,
                             out.ctypes.data_as(ctypes.c_void_p))
    return out


def uniform(seed: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    _load().synth_uniform_f64(seed & (2**64 - 1), offset, int(n), out.ctypes.data_as(ctypes.c_void_p))
    return out


def splitmix64(seed: int, i: int) -> int:
    return int(_load().synth_splitmix64(seed & (2**64 - 1), i))

"""CPU oracle for the Q4_0 block-quantized matmul — test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never reaches it; the two share no code.

The arithmetic lives in ``q4_oracle.c`` (plain C, fp64 accumulation); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB = os.path.join(_HERE, "libq4oracle.so")

BLOCK = 32
BLOCK_BYTES = 18
OK, ERR_SHAPE, ERR_NONFINITE, ERR_RANGE = 0, 2, 4, 5

_lib = None


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
    """Compile the oracle into ``libq4oracle.so`` next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC) or _foreign_binary(_LIB):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.q4o_f32_to_f16.argtypes = [ctypes.c_float]
        lib.q4o_f32_to_f16.restype = ctypes.c_uint16
        lib.q4o_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q4o_f16_to_f32.restype = ctypes.c_float
        lib.q4o_quantize.argtypes = [p, i64, i64, p]
        lib.q4o_dequantize.argtypes = [p, i64, i64, p]
        lib.q4o_matmul.argtypes = [p, i64, i64, p, i64, p, p, p]
        lib.q4o_matmul_pairs.argtypes = [p, i64, i64, p, i64, p, i64, p, p, p]
        lib.q4o_argmax.argtypes = [p, i64, i64, p]
        lib.q4o_num_threads.argtypes = []
        lib.q4o_set_threads.argtypes = [ctypes.c_int]
        for f in ("q4o_quantize", "q4o_dequantize", "q4o_matmul", "q4o_matmul_pairs",
                  "q4o_argmax", "q4o_num_threads", "q4o_set_threads"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, status):
        super().__init__("oracle status %d" % status)
        self.status = status


def f32_to_f16_bits(v: float) -> int:
    return int(_load().q4o_f32_to_f16(ctypes.c_float(v)))


def f16_bits_to_f32(h: int) -> float:
    return float(_load().q4o_f16_to_f32(ctypes.c_uint16(h)))


def quantize(w: np.ndarray) -> np.ndarray:
    """fp32 W[N,K] -> canonical blocks, uint8 [N, K/32, 18]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.zeros((N, max(K // BLOCK, 0), BLOCK_BYTES), dtype=np.uint8)
    s = _load().q4o_quantize(_ptr(w), N, K, _ptr(out))
    if s != OK:
        raise OracleError(s)
    return out


def dequantize(blocks: np.ndarray) -> np.ndarray:
    """canonical blocks [N, K/32, 18] -> fp32 W[N,K] = (q-8)*d16."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    N, nb, _ = blocks.shape
    w = np.empty((N, nb * BLOCK), dtype=np.float32)
    s = _load().q4o_dequantize(_ptr(blocks), N, nb * BLOCK, _ptr(w))
    if s != OK:
        raise OracleError(s)
    return w


def matmul(blocks: np.ndarray, x: np.ndarray):
    """y = x @ W^T with fp64 accumulation.  Returns (y fp32, y fp64, bound)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N, nb, _ = blocks.shape
    M, K = x.shape
    assert K == nb * BLOCK
    y = np.empty((M, N), dtype=np.float32)
    y64 = np.empty((M, N), dtype=np.float64)
    bound = np.empty((M, N), dtype=np.float64)
    s = _load().q4o_matmul(_ptr(blocks), N, K, _ptr(x), M, _ptr(y), _ptr(y64), _ptr(bound))
    if s != OK:
        raise OracleError(s)
    return y, y64, bound


def matmul_pairs(blocks: np.ndarray, x: np.ndarray, pairs: np.ndarray):
    """The same for chosen (m, n) pairs, int64 [P, 2]."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    pairs = np.ascontiguousarray(pairs, dtype=np.int64)
    N, nb, _ = blocks.shape
    M, K = x.shape
    P = pairs.shape[0]
    y = np.empty(P, dtype=np.float32)
    y64 = np.empty(P, dtype=np.float64)
    bound = np.empty(P, dtype=np.float64)
    s = _load().q4o_matmul_pairs(_ptr(blocks), N, K, _ptr(x), M, _ptr(pairs), P,
                                 _ptr(y), _ptr(y64), _ptr(bound))
    if s != OK:
        raise OracleError(s)
    return y, y64, bound


def argmax(y: np.ndarray) -> np.ndarray:
    """Per-row greedy pick over fp32 logits: lowest index on ties, NaN never wins."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    M, N = y.shape
    idx = np.empty(M, dtype=np.int32)
    s = _load().q4o_argmax(_ptr(y), M, N, _ptr(idx))
    if s != OK:
        raise OracleError(s)
    return idx


def num_threads() -> int:
    return int(_load().q4o_num_threads())


def set_threads(n: int) -> int:
    """Use n threads in the oracle's loops from now on; returns the previous count."""
    return int(_load().q4o_set_threads(int(n)))

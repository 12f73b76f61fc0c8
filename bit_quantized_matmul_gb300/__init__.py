"""Thin Python binding over the C ABI of ``libq4mm.so`` (``include/q4mm.h``).

Argument marshalling only: tensors are passed as raw device pointers with the
current PyTorch CUDA stream, and every step of the computation runs in the
library's CUDA kernels.  There is no CPU or PyTorch fallback: if the library
is missing, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch  # device memory and streams; loads the CUDA runtime first

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq4mm.so")

Q4_OK = 0
Q4_ERR_INVALID_ARG = 1
Q4_ERR_SHAPE = 2
Q4_ERR_ALIGN = 3
Q4_ERR_NONFINITE = 4
Q4_ERR_RANGE = 5
Q4_ERR_CUDA = 6
Q4_ERR_TIMEOUT = 7
Q4_ERR_NOMEM = 8
Q4_ERR_UNSUPPORTED = 9

Q4MM_BATCH_INVARIANT = 0x1
Q4MM_FORCE_SIMT = 0x2
Q4MM_FORCE_TC = 0x4
Q4MM_ROW_BY_ROW = 0x8
Q4MM_FORCE_MMA = 0x10
Q4MM_M_MAX = 4096
Q4MM_GROUP_MAX = 4
Q4MM_NOALLOC_PARTIAL_BYTES = 2457600
Q4MM_PATH_SIMT = 1
Q4MM_PATH_TC = 2
Q4MM_PATH_ROW_BY_ROW = 3
Q4MM_PATH_MMA = 4

BLOCK = 32
BLOCK_BYTES = 18

# Every symbol the header declares; the CPU test checks the library exports them.
EXPORTS = (
    "q4_quantize", "q4_import_blocks", "q4_export_blocks", "q4_weight_free", "q4_weight_shape",
    "q4_weight_device_bytes", "q4mm_forward", "q4mm_forward_ex", "q4mm_argmax", "q4mm_argmax_ex",
    "q4mm_forward_noalloc", "q4mm_forward_group", "q4mm_forward_gated", "q4mm_argmax_rows", "q4_verify_greedy",
    "q4mm_select_path", "q4mm_plan_info", "q4mm_set_m_threshold", "q4mm_get_m_threshold", "q4mm_set_group_m_threshold",
    "q4mm_get_group_m_threshold", "q4_device_status", "q4mm_set_wait_limit_ns", "q4mm_set_stall_for_test",
    "q4_status_string", "q4_scratch_bytes",
    "q4_kv_append",
)

if not os.path.exists(LIB_PATH):
    raise ImportError("libq4mm.so is not built (%s); run __graft_entry__.build() or "
                      "python bit_quantized_matmul_gb300/build.py" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_sig = {
    "q4_quantize": [_p, _i64, _i64, ctypes.POINTER(_p), _p],
    "q4_import_blocks": [_p, _i64, _i64, ctypes.POINTER(_p), _p],
    "q4_export_blocks": [_p, _p, ctypes.c_size_t],
    "q4_weight_free": [_p],
    "q4_weight_shape": [_p, ctypes.POINTER(_i64), ctypes.POINTER(_i64)],
    "q4_weight_device_bytes": [_p, ctypes.POINTER(ctypes.c_size_t)],
    "q4mm_forward": [_p, _p, _p, _i64, _p],
    "q4mm_forward_ex": [_p, _p, _p, _i64, _u32, _p],
    "q4mm_argmax": [_p, _p, _p, _p, _i64, _p],
    "q4mm_argmax_ex": [_p, _p, _p, _p, _i64, _u32, _p],
    "q4mm_forward_noalloc": [_p, _p, _p, _i64, _p],
    "q4mm_forward_group": [_p, ctypes.c_int, _p, _p, _i64, _u32, _p],
    "q4mm_forward_gated": [_p, _p, _p, _p, _i64, _u32, _p],
    "q4mm_argmax_rows": [_p, _p, _i64, _p, _i64, _p, _p, _p],
    "q4_verify_greedy": [_p, _p, _i64, _p, _i64, _p, _p],
    "q4_kv_append": [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(_i64),
                     ctypes.POINTER(_i64), _p, _p, _p, _i64, _i64, _p],
    "q4mm_select_path": [_p, _i64, _u32],
    "q4mm_plan_info": [_p, _i64, _u32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                       ctypes.POINTER(ctypes.c_int)],
    "q4mm_set_m_threshold": [_i64],
    "q4mm_get_m_threshold": [],
    "q4mm_set_group_m_threshold": [_i64],
    "q4mm_get_group_m_threshold": [],
    "q4_device_status": [],
    "q4mm_set_wait_limit_ns": [ctypes.c_uint64],
    "q4mm_set_stall_for_test": [ctypes.c_int],
    "q4_status_string": [ctypes.c_int],
    "q4_scratch_bytes": [ctypes.POINTER(ctypes.c_size_t)] * 4,
}
for _name, _args in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.q4mm_get_m_threshold.restype = ctypes.c_int64
_lib.q4mm_get_group_m_threshold.restype = ctypes.c_int64
_lib.q4_status_string.restype = ctypes.c_char_p


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        msg = "%s: %s (status %d)" % (what, q4_status_string(status), status)
        super().__init__(msg)
        self.status = status


def _check(status: int, what: str):
    if status != Q4_OK:
        raise Q4Error(status, what)


def q4_status_string(status: int) -> str:
    return _lib.q4_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev_f32(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise ValueError("%s must be a contiguous float32 CUDA tensor" % name)
    return t


class Q4Weight:
    """Owning wrapper of a ``q4_weight*`` handle (freed on ``free()`` / GC)."""

    def __init__(self, handle: int, N: int, K: int, device: torch.device):
        self._h = ctypes.c_void_p(handle)
        self.N, self.K, self.device = N, K, device

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("Q4Weight already freed")
        return self._h

    def free(self):
        if self._h:
            torch.cuda.synchronize(self.device)
            _check(_lib.q4_weight_free(self._h), "q4_weight_free")
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            if self._h:
                _lib.q4_weight_free(self._h)
        except Exception:
            pass

    def device_bytes(self) -> int:
        b = ctypes.c_size_t(0)
        _check(_lib.q4_weight_device_bytes(self.handle, ctypes.byref(b)), "q4_weight_device_bytes")
        return int(b.value)

    @property
    def packed_bytes(self) -> int:
        """Algorithmic size of the Q4_0 weights: N*K/32 blocks of 18 bytes."""
        return self.N * (self.K // BLOCK) * BLOCK_BYTES


def q4_quantize(w: torch.Tensor, stream=None) -> Q4Weight:
    """Quantize an fp32 [N, K] CUDA tensor into a library-owned Q4_0 weight."""
    _dev_f32(w, "w")
    N, K = w.shape
    h = ctypes.c_void_p(0)
    with torch.cuda.device(w.device):
        _check(_lib.q4_quantize(w.data_ptr(), N, K, ctypes.byref(h), _stream(stream)), "q4_quantize")
    return Q4Weight(h.value, N, K, w.device)


def q4_import_blocks(blocks, N: int, K: int, device=None, stream=None) -> Q4Weight:
    """Create a weight from canonical blocks (uint8 numpy array / bytes, N*K/32*18 bytes)."""
    import numpy as np

    arr = np.ascontiguousarray(np.frombuffer(bytes(blocks), np.uint8) if isinstance(blocks, (bytes, bytearray))
                               else blocks, dtype=np.uint8)
    if arr.size != N * (K // BLOCK) * BLOCK_BYTES:
        raise ValueError("blocks size does not match N, K")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    h = ctypes.c_void_p(0)
    with torch.cuda.device(device):
        _check(_lib.q4_import_blocks(arr.ctypes.data_as(ctypes.c_void_p), N, K, ctypes.byref(h),
                                     _stream(stream)), "q4_import_blocks")
    return Q4Weight(h.value, N, K, device)


def q4_export_blocks(W: Q4Weight):
    """Canonical blocks of W as a uint8 numpy array [N, K/32, 18]."""
    import numpy as np

    out = np.empty((W.N, W.K // BLOCK, BLOCK_BYTES), np.uint8)
    with torch.cuda.device(W.device):
        _check(_lib.q4_export_blocks(W.handle, out.ctypes.data_as(ctypes.c_void_p), out.nbytes),
               "q4_export_blocks")
    return out


def q4_weight_free(W: Q4Weight):
    W.free()


def q4mm_forward_ex(W: Q4Weight, x: torch.Tensor, flags: int = 0, y: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ W^T (fp32) with Q4MM_* flags."""
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [M, %d]" % W.K)
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.float32, device=x.device)
    _dev_f32(y, "y")
    if tuple(y.shape) != (M, W.N):
        raise ValueError("y must be [M, %d]" % W.N)
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_forward_ex(W.handle, x.data_ptr(), y.data_ptr(), M, int(flags), _stream(stream)),
               "q4mm_forward_ex")
    return y


def q4mm_forward(W: Q4Weight, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [M, %d]" % W.K)
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.float32, device=x.device)
    _dev_f32(y, "y")
    if tuple(y.shape) != (M, W.N):
        raise ValueError("y must be [M, %d]" % W.N)
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_forward(W.handle, x.data_ptr(), y.data_ptr(), M, _stream(stream)), "q4mm_forward")
    return y


def q4mm_forward_noalloc(W: Q4Weight, x: torch.Tensor, y: torch.Tensor, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ W^T into the caller's y, allocating no device memory.

    For callers that must not allocate mid-step (their memory is all in their
    own pool, or a device-wide wait is unacceptable).  The first call on a
    device sets up the fixed scratch and synchronizes once; calls whose kernels
    overlap on the GPU race on that scratch.  Raises Q4Error(Q4_ERR_SHAPE) when
    the split-K partial sums exceed Q4MM_NOALLOC_PARTIAL_BYTES.
    """
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [M, %d]" % W.K)
    _dev_f32(y, "y")
    if tuple(y.shape) != (M, W.N):
        raise ValueError("y must be [M, %d]" % W.N)
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_forward_noalloc(W.handle, x.data_ptr(), y.data_ptr(), M, _stream(stream)),
               "q4mm_forward_noalloc")
    return y


def q4mm_forward_group(Ws, x: torch.Tensor, ys=None, flags: int = 0, stream=None):
    """[x @ W_i^T for W_i in Ws] in one launch per 16 token rows (weights sharing K)."""
    _dev_f32(x, "x")
    M = x.shape[0]
    if not 1 <= len(Ws) <= Q4MM_GROUP_MAX:
        raise ValueError("1 to %d weights" % Q4MM_GROUP_MAX)
    if x.dim() != 2 or any(W.K != x.shape[1] for W in Ws):
        raise ValueError("x must be [M, K] with the K of every weight")
    if ys is None:
        ys = [torch.empty((M, W.N), dtype=torch.float32, device=x.device) for W in Ws]
    if len(ys) != len(Ws):
        raise ValueError("one output per weight")
    for W, y in zip(Ws, ys):
        _dev_f32(y, "y")
        if tuple(y.shape) != (M, W.N):
            raise ValueError("y must be [M, %d]" % W.N)
    hw = (ctypes.c_void_p * len(Ws))(*[W.handle for W in Ws])
    hy = (ctypes.c_void_p * len(ys))(*[y.data_ptr() for y in ys])
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_forward_group(hw, len(Ws), x.data_ptr(), hy, M, int(flags), _stream(stream)),
               "q4mm_forward_group")
    return ys


def q4mm_forward_gated(Wg: Q4Weight, Wu: Q4Weight, x: torch.Tensor, h: torch.Tensor | None = None,
                       flags: int = 0, stream=None) -> torch.Tensor:
    """h = SiLU(x @ Wg^T) * (x @ Wu^T) (the gated MLP step; q4mm_forward_gated)."""
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != Wg.K:
        raise ValueError("x must be [M, %d]" % Wg.K)
    if (Wu.N, Wu.K) != (Wg.N, Wg.K):
        raise ValueError("gate and up projections must have one shape")
    if h is None:
        h = torch.empty((M, Wg.N), dtype=torch.float32, device=x.device)
    _dev_f32(h, "h")
    if tuple(h.shape) != (M, Wg.N):
        raise ValueError("h must be [M, %d]" % Wg.N)
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_forward_gated(Wg.handle, Wu.handle, x.data_ptr(), h.data_ptr(), M, int(flags),
                                       _stream(stream)), "q4mm_forward_gated")
    return h


def q4mm_argmax_rows(W: Q4Weight, x: torch.Tensor, rows: torch.Tensor, want_max: bool = True,
                     stream=None):
    """Greedy pick (idx int32 [R], max fp32 [R] or None) for the x rows listed in `rows`."""
    _dev_f32(x, "x")
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [rows, %d]" % W.K)
    if rows.dtype != torch.int32 or not rows.is_cuda or not rows.is_contiguous():
        raise ValueError("rows must be a contiguous int32 CUDA tensor")
    R = rows.numel()
    idx = torch.empty((R,), dtype=torch.int32, device=x.device)
    mx = torch.empty((R,), dtype=torch.float32, device=x.device) if want_max else None
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_argmax_rows(W.handle, x.data_ptr(), x.shape[0], rows.data_ptr(), R, idx.data_ptr(),
                                     mx.data_ptr() if mx is not None else None, _stream(stream)),
               "q4mm_argmax_rows")
    return idx, mx


def q4_verify_greedy(idx: torch.Tensor, draft: torch.Tensor, offsets: torch.Tensor, stream=None):
    """accepted[s]: leading positions of segment s where idx == draft (-1: malformed segment)."""
    for t, n in ((idx, "idx"), (draft, "draft"), (offsets, "offsets")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous int32 CUDA tensor" % n)
    if idx.numel() != draft.numel():
        raise ValueError("idx and draft differ in length")
    S = offsets.numel() - 1
    acc = torch.empty((max(S, 0),), dtype=torch.int32, device=idx.device)
    with torch.cuda.device(idx.device):
        _check(_lib.q4_verify_greedy(idx.data_ptr(), draft.data_ptr(), idx.numel(), offsets.data_ptr(), max(S, 0),
                                     acc.data_ptr(), _stream(stream)), "q4_verify_greedy")
    return acc


def q4_kv_append(k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                 offsets: torch.Tensor, slot: torch.Tensor, pos: torch.Tensor, stream=None):
    """Write the step's new K/V rows into a preallocated cache, in place.

    k_cache, v_cache: contiguous [layers, slots, heads, capacity, head_dim];
    k_new, v_new: [layers, total, heads, head_dim] views (head_dim contiguous,
    any other strides) of the same dtype (2- or 4-byte elements);
    offsets int32 [S + 1], slot and pos int32 [S], all on the cache's device.
    """
    if k_cache.dim() != 5 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() or \
            not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [layers, slots, heads, capacity, head_dim] of one shape")
    if k_new.dim() != 4 or v_new.shape != k_new.shape:
        raise ValueError("new rows must be [layers, total, heads, head_dim] views of one shape")
    L, slots, H, cap, D = k_cache.shape
    if k_new.shape[0] != L or k_new.shape[2] != H or k_new.shape[3] != D or k_new.stride(3) != 1 or \
            v_new.stride(3) != 1:
        raise ValueError("new rows do not match the cache shape (or head_dim is not contiguous)")
    for t in (v_cache, k_new, v_new):
        if t.dtype != k_cache.dtype or t.device != k_cache.device:
            raise ValueError("caches and new rows must share dtype and device")
    for t, n in ((offsets, "offsets"), (slot, "slot"), (pos, "pos")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.device != k_cache.device:
            raise ValueError("%s must be a contiguous int32 tensor on the cache's device" % n)
    S = slot.numel()
    if offsets.numel() != S + 1 or pos.numel() != S:
        raise ValueError("offsets must have S + 1 entries and pos S")
    with torch.cuda.device(k_cache.device):
        ks = (_i64 * 3)(*k_new.stride()[:3])
        vs = (_i64 * 3)(*v_new.stride()[:3])
        _check(_lib.q4_kv_append(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                 L, slots, H, D, cap, k_cache.element_size(), ks, vs, offsets.data_ptr(),
                                 slot.data_ptr(), pos.data_ptr(), S, k_new.shape[1], _stream(stream)),
               "q4_kv_append")


def q4mm_argmax_ex(W: Q4Weight, x: torch.Tensor, flags: int = 0, want_max: bool = True, stream=None):
    """Fused greedy pick: (idx int32 [M], maxval fp32 [M] or None)."""
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [M, %d]" % W.K)
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    mx = torch.empty(M, dtype=torch.float32, device=x.device) if want_max else None
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_argmax_ex(W.handle, x.data_ptr(), idx.data_ptr(), mx.data_ptr() if mx is not None else None,
                                   M, int(flags), _stream(stream)), "q4mm_argmax_ex")
    return idx, mx


def q4mm_argmax(W: Q4Weight, x: torch.Tensor, want_max: bool = True, stream=None):
    _dev_f32(x, "x")
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("x must be [M, %d]" % W.K)
    idx = torch.empty(M, dtype=torch.int32, device=x.device)
    mx = torch.empty(M, dtype=torch.float32, device=x.device) if want_max else None
    with torch.cuda.device(x.device):
        _check(_lib.q4mm_argmax(W.handle, x.data_ptr(), idx.data_ptr(), mx.data_ptr() if mx is not None else None,
                                M, _stream(stream)), "q4mm_argmax")
    return idx, mx


def q4mm_select_path(W: Q4Weight, M: int, flags: int = 0) -> int:
    with torch.cuda.device(W.device):
        r = _lib.q4mm_select_path(W.handle, M, int(flags))
    if r < 0:
        raise Q4Error(-r, "q4mm_select_path")
    return r


def q4mm_plan_info(W: Q4Weight, M: int, flags: int = 0):
    """(path, kernel launches, K splits) that a call would use."""
    p, l, s = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    with torch.cuda.device(W.device):
        _check(_lib.q4mm_plan_info(W.handle, M, int(flags), ctypes.byref(p), ctypes.byref(l), ctypes.byref(s)),
               "q4mm_plan_info")
    return p.value, l.value, s.value


def q4mm_set_m_threshold(m: int):
    _check(_lib.q4mm_set_m_threshold(int(m)), "q4mm_set_m_threshold")


def q4mm_get_m_threshold() -> int:
    return int(_lib.q4mm_get_m_threshold())


def q4mm_set_group_m_threshold(m: int):
    _check(_lib.q4mm_set_group_m_threshold(int(m)), "q4mm_set_group_m_threshold")


def q4mm_get_group_m_threshold() -> int:
    return int(_lib.q4mm_get_group_m_threshold())


def q4mm_set_wait_limit_ns(ns: int):
    """Bound of the kernels' waits in ns for later launches (0: the default, 1 s)."""
    _check(_lib.q4mm_set_wait_limit_ns(int(ns)), "q4mm_set_wait_limit_ns")


def q4mm_set_stall_for_test(on: bool):
    """Test setting: later launches withhold their first hand-off so that waits run out."""
    _check(_lib.q4mm_set_stall_for_test(1 if on else 0), "q4mm_set_stall_for_test")


def q4_device_status() -> int:
    return int(_lib.q4_device_status())


def q4_scratch_bytes() -> tuple:
    """(partial, xop, gu, xpre): bytes of the library's scratch now held on the current device."""
    v = [ctypes.c_size_t(0) for _ in range(4)]
    _check(_lib.q4_scratch_bytes(*[ctypes.byref(a) for a in v]), "q4_scratch_bytes")
    return tuple(int(a.value) for a in v)


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library (for callers that marshal pointers themselves)."""
    return _lib

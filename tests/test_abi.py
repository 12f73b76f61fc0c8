"""Host-side checks of the C ABI that need no GPU: the shared library builds
and loads, exports every symbol ``include/q4mm.h`` declares, and rejects bad
arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    return q4


def _declared():
    text = open(os.path.join(ROOT, "include", "q4mm.h")).read()
    return sorted(set(re.findall(r"^Q4_API\s+[\w\s\*]+?\b(q4\w*)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("q4_quantize", "q4mm_forward", "q4mm_argmax", "q4_import_blocks", "q4_export_blocks"):
        assert want in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(q4):
    lib = ctypes.CDLL(q4.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(q4.EXPORTS) == _declared()


def test_status_strings_and_threshold(q4):
    assert q4.q4_status_string(q4.Q4_OK) == "ok"
    assert "aligned" in q4.q4_status_string(q4.Q4_ERR_ALIGN)
    assert q4.q4_status_string(12345) == "unknown status"
    old = q4.q4mm_get_m_threshold()
    assert old >= 1
    q4.q4mm_set_m_threshold(7)
    assert q4.q4mm_get_m_threshold() == 7
    q4.q4mm_set_m_threshold(old)
    with pytest.raises(q4.Q4Error) as e:
        q4.q4mm_set_m_threshold(0)
    assert e.value.status == q4.Q4_ERR_INVALID_ARG
    old_g = q4.q4mm_get_group_m_threshold()
    assert old_g >= 1
    q4.q4mm_set_group_m_threshold(9)
    assert q4.q4mm_get_group_m_threshold() == 9
    q4.q4mm_set_group_m_threshold(old_g)
    with pytest.raises(q4.Q4Error) as e:
        q4.q4mm_set_group_m_threshold(q4.Q4MM_M_MAX + 2)
    assert e.value.status == q4.Q4_ERR_INVALID_ARG


def test_null_arguments_rejected_on_host(q4):
    lib = q4.raw_library()
    assert lib.q4mm_forward(None, None, None, 4, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_ex(None, None, None, 4, 0, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_argmax(None, None, None, None, 4, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4_quantize(None, 4, 32, None, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4_weight_free(None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4_export_blocks(None, None, 0) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_select_path(None, 1, 0) == -q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_noalloc(None, None, None, 4, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_group(None, 1, None, None, 4, 0, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_argmax_rows(None, None, 1, None, 1, None, None, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4_verify_greedy(None, None, 0, None, 1, None, None) == q4.Q4_ERR_INVALID_ARG


def test_kv_append_arguments_checked_on_host(q4):
    lib = q4.raw_library()
    a16 = 4096  # aligned stand-in addresses: these calls return before any CUDA call

    I3 = ctypes.c_int64 * 3

    def call(p=a16, layers=2, slots=2, heads=2, head_dim=64, cap=16, eb=2, st=128, S=1, total=1, off=a16,
             strides=True):
        ks, vs = I3(0, st, 64), I3(0, 64, 128)
        return lib.q4_kv_append(p, p, p, p, layers, slots, heads, head_dim, cap, eb, ks if strides else None,
                                vs, off, off, off, S, total, None)

    assert call(layers=0) == q4.Q4_ERR_INVALID_ARG
    assert call(eb=3) == q4.Q4_ERR_INVALID_ARG
    assert call(st=-1) == q4.Q4_ERR_INVALID_ARG
    assert call(strides=False) == q4.Q4_ERR_INVALID_ARG
    assert call(S=-1) == q4.Q4_ERR_INVALID_ARG
    assert call(S=0) == q4.Q4_OK and call(total=0) == q4.Q4_OK  # nothing to write
    assert call(p=None) == q4.Q4_ERR_INVALID_ARG
    assert call(off=None) == q4.Q4_ERR_INVALID_ARG
    assert call(head_dim=12) == q4.Q4_ERR_ALIGN     # 24-byte rows
    assert call(st=100) == q4.Q4_ERR_ALIGN          # 200-byte token stride
    assert call(p=a16 + 8) == q4.Q4_ERR_ALIGN
    assert call(total=2 ** 30) == q4.Q4_ERR_INVALID_ARG  # 8 vectors per row: past the 32-bit item index


def test_binding_constants_match_the_header(q4):
    # every numeric #define of the header (status codes, flags, limits, paths)
    # has the same value in the Python binding
    text = open(os.path.join(ROOT, "include", "q4mm.h")).read()
    defs = dict(re.findall(r"^#define\s+(Q4\w*)\s+(0x[0-9A-Fa-f]+|\d+)u?\b", text, re.M))
    assert len(defs) >= 20
    for name, value in defs.items():
        assert hasattr(q4, name), name
        assert getattr(q4, name) == int(value, 0), (name, value, getattr(q4, name))

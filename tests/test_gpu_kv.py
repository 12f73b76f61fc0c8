"""KV-cache append on the GPU (q4_kv_append) against the oracle, bit for bit.

The new K rows are a plain [layers, total, heads, head_dim] tensor; the new V
rows are a transposed view of a [layers, heads, total, head_dim] tensor, the
non-contiguous source that "A non-contiguous KV cache cuts Qwen2 decode speed
by 59 % at 2k context in Candle on Metal" (§"Cause and workaround") traces the
slow appends to.  Steps mix a prefill, decode rows and verify rows of several
requests, as a continuous-batching step does."""
import numpy as np
import pytest
import torch

from oracle import kv as kv_oracle
import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    return q4


def _bits(t):
    """Exact bit pattern as a numpy array (int16 for 2-byte, int32 for 4-byte elements)."""
    return t.cpu().view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def _new_rows(seed, layers, total, heads, D, dtype):
    k = torch.from_numpy(synthetic.normal(seed, (layers, total, heads, D))).to(dtype)
    vt = torch.from_numpy(synthetic.normal(seed + 1, (layers, heads, total, D))).to(dtype)
    return k.cuda(), vt.cuda().transpose(1, 2)  # v: a strided [layers, total, heads, D] view


def _run_steps(q4, dtype, layers, heads, D, slots, cap, plan, seed):
    kc = torch.full((layers, slots, heads, cap, D), -3.5, dtype=dtype, device="cuda")
    vc = kc.clone()
    kc_ref, vc_ref = _bits(kc), _bits(vc)
    lengths = np.zeros(slots, np.int32)
    for i, step in enumerate(plan):
        lead = step[0]  # packed rows before the first request are not cached
        reqs = step[1:]
        total = lead + sum(n for _, n in reqs)
        k_new, v_new = _new_rows(seed + 10 * i, layers, total, heads, D, dtype)
        offsets = np.concatenate([[lead], lead + np.cumsum([n for _, n in reqs])]).astype(np.int32)
        slot = np.array([s for s, _ in reqs], np.int32)
        pos = lengths[slot].copy()
        q4.q4_kv_append(kc, vc, k_new, v_new, torch.from_numpy(offsets).cuda(), torch.from_numpy(slot).cuda(),
                        torch.from_numpy(pos).cuda())
        kc_ref, vc_ref, rej = kv_oracle.kv_append(kc_ref, vc_ref, _bits(k_new), _bits(v_new), offsets, slot, pos)
        assert rej == []
        lengths[slot] += np.diff(offsets).astype(np.int32)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == q4.Q4_OK
    assert np.array_equal(_bits(kc), kc_ref)
    assert np.array_equal(_bits(vc), vc_ref)


# each step: (rows before the first request, then (slot, rows) per request)
PLAN = [
    (0, (0, 37), (2, 1), (5, 4)),            # a prefill, a decode row, 4 verify rows
    (3, (0, 1), (2, 1), (5, 1), (1, 0)),     # decode rows, an empty request
    (0, (1, 13), (0, 4), (2, 1), (5, 2), (3, 1)),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("layers,heads,D", [(3, 2, 64), (1, 5, 16)])
def test_kv_append_matches_oracle(q4, dtype, layers, heads, D):
    _run_steps(q4, dtype, layers, heads, D, slots=6, cap=64, plan=PLAN, seed=0x4B560000 + D)


def test_kv_append_qwen05b_prefill_then_decode(q4):
    # Qwen2.5-0.5B-shaped cache (24 layers, 2 KV heads, head_dim 64, bf16): a
    # 2,049-row prefill into one slot, then a decode step of 64 requests
    plan = [(0, (0, 2049)), tuple([0] + [(s, 1) for s in range(64)])]
    _run_steps(q4, torch.bfloat16, 24, 2, 64, slots=64, cap=2112, plan=plan, seed=0x4B570000)


def test_kv_append_out_of_range_requests_left_unwritten(q4):
    layers, heads, D, slots, cap = 2, 2, 16, 3, 8
    kc = torch.zeros((layers, slots, heads, cap, D), dtype=torch.float32, device="cuda")
    vc = torch.zeros_like(kc)
    k_new, v_new = _new_rows(77, layers, 9, heads, D, torch.float32)
    offsets = np.array([0, 3, 6, 8, 9], np.int32)
    slot = np.array([0, 1, 5, 2], np.int32)   # request 2: no such slot
    pos = np.array([6, 0, 0, -1], np.int32)   # request 0 passes capacity, request 3 is negative
    q4.q4_kv_append(kc, vc, k_new, v_new, *(torch.from_numpy(a).cuda() for a in (offsets, slot, pos)))
    torch.cuda.synchronize()
    assert q4.q4_device_status() == q4.Q4_ERR_INVALID_ARG
    assert q4.q4_device_status() == q4.Q4_OK  # read and cleared
    k_ref, v_ref, rej = kv_oracle.kv_append(_bits(torch.zeros_like(kc)), _bits(torch.zeros_like(vc)),
                                            _bits(k_new), _bits(v_new), offsets, slot, pos)
    assert rej == [0, 2, 3]
    assert np.array_equal(_bits(kc), k_ref) and np.array_equal(_bits(vc), v_ref)


def test_kv_append_binding_rejects_bad_views(q4):
    kc = torch.zeros((1, 2, 1, 4, 16), dtype=torch.float32, device="cuda")
    rows = torch.zeros((1, 2, 1, 16), dtype=torch.float32, device="cuda")
    i32 = lambda *v: torch.tensor(v, dtype=torch.int32, device="cuda")  # noqa: E731
    with pytest.raises(ValueError):  # head_dim not contiguous
        q4.q4_kv_append(kc, kc.clone(), rows.transpose(2, 3), rows.transpose(2, 3), i32(0, 2), i32(0), i32(0))
    with pytest.raises(ValueError):  # offsets too short
        q4.q4_kv_append(kc, kc.clone(), rows, rows, i32(0), i32(0), i32(0))


def test_kv_append_as_first_call_of_a_process():
    # a fresh process whose first library call is the append (device set-up
    # happens inside it)
    import subprocess
    import sys

    code = ("import torch, sys; sys.path.insert(0, %r); import bit_quantized_matmul_gb300 as q4;"
            "kc = torch.zeros((1, 1, 1, 4, 16), device='cuda'); vc = torch.zeros_like(kc);"
            "rows = torch.ones((1, 2, 1, 16), device='cuda');"
            "i32 = lambda *v: torch.tensor(v, dtype=torch.int32, device='cuda');"
            "q4.q4_kv_append(kc, vc, rows, rows * 2, i32(0, 2), i32(0), i32(1)); torch.cuda.synchronize();"
            "assert q4.q4_device_status() == q4.Q4_OK;"
            "assert kc[0, 0, 0, 1:3].eq(1).all() and vc[0, 0, 0, 1:3].eq(2).all() and kc[0, 0, 0, 0].eq(0).all()"
            % __import__("conftest").ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]

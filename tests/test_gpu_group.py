"""GPU checks of q4mm_forward_group: several weights that share K and the
activations (a decoder layer's q/k/v or gate/up projections) in one launch.
Each output is compared element by element with the oracle's bound."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, weights

pytestmark = pytest.mark.gpu

q4 = pytest.importorskip("bit_quantized_matmul_gb300")


def _group(shapes, config):
    ws = [weights(config, i, N, K) for i, (N, K) in enumerate(shapes)]
    Ws = [q4.q4_quantize(torch.from_numpy(w).cuda()) for w in ws]
    blocks = [oracle.quantize(w) for w in ws]
    return Ws, blocks


@pytest.mark.parametrize("shapes,Ms", [
    ([(3584, 3584), (512, 3584), (512, 3584)], (1, 5, 8, 13)),   # q, k, v
    ([(300, 1024), (130, 1024)], (1, 3, 17)),                     # ragged tiles
    ([(18944, 3584), (18944, 3584)], (2,)),                       # gate, up
])
def test_group_matches_oracle(shapes, Ms):
    Ws, blocks = _group(shapes, 95)
    K = shapes[0][1]
    for M in Ms:
        x_np = acts(95, M, K)
        ys = q4.q4mm_forward_group(Ws, torch.from_numpy(x_np).cuda())
        torch.cuda.synchronize()
        assert q4.q4_device_status() == q4.Q4_OK
        for i, (y, b) in enumerate(zip(ys, blocks)):
            _, y64, bound = oracle.matmul(b, x_np)
            assert_within_bound(y.cpu().numpy(), y64, bound, "group weight %d M=%d" % (i, M))
    for W in Ws:
        W.free()


def test_group_of_one_equals_single_call():
    Ws, _ = _group([(896, 896)], 96)
    x = torch.from_numpy(acts(96, 6, 896)).cuda()
    (yg,) = q4.q4mm_forward_group(Ws, x, flags=q4.Q4MM_FORCE_MMA)
    ys = q4.q4mm_forward_ex(Ws[0], x, q4.Q4MM_FORCE_MMA)
    assert torch.equal(yg.view(torch.int32), ys.view(torch.int32))
    Ws[0].free()


@pytest.mark.parametrize("force_tc", [False, True])
def test_group_batch_invariant_rows(force_tc):
    Ws, blocks = _group([(3584, 3584), (512, 3584), (512, 3584)], 97)
    inv = q4.Q4MM_BATCH_INVARIANT | (q4.Q4MM_FORCE_TC if force_tc else 0)
    x_np = acts(97, 40, 3584)
    big = torch.from_numpy(x_np).cuda()
    y40 = q4.q4mm_forward_group(Ws, big, flags=inv)
    y7 = q4.q4mm_forward_group(Ws, big[:7].contiguous(), flags=inv)
    for r in (0, 3, 6, 33, 39):
        y1 = q4.q4mm_forward_group(Ws, big[r:r + 1].contiguous(), flags=inv)
        for a, b in zip(y40, y1):
            assert torch.equal(a[r].view(torch.int32), b[0].view(torch.int32)), r
    for a, b in zip(y40, y7):
        assert torch.equal(a[:7].view(torch.int32), b.view(torch.int32))
    for y, b in zip(y40, blocks):
        _, y64, bound = oracle.matmul(b, x_np)
        assert_within_bound(y.cpu().numpy(), y64, bound, "group invariant tc=%s" % force_tc)
    for W in Ws:
        W.free()


@pytest.mark.parametrize("shapes,Ms", [
    ([(300, 1024), (256, 1024)], (3, 40)),                    # ragged first weight
    ([(1000, 3584), (130, 3584), (130, 3584)], (1, 17, 64)),  # q/k/v-like: 8 + 2 + 2 tiles, ragged
    ([(2000, 2048), (2000, 2048)], (33, 300)),                # gate/up-like; two launch pairs at 300
])
def test_group_above_threshold_one_tensor_core_launch(shapes, Ms):
    # at or above the group threshold one tcgen05 launch covers every tile of
    # the group: each tile's weight, output and partial-sum slots come from
    # the global tile index
    Ws, blocks = _group(shapes, 98)
    thr = q4.q4mm_get_group_m_threshold()
    try:
        q4.q4mm_set_group_m_threshold(1)  # every M below on the grouped tensor-core path
        for M in Ms:
            x_np = acts(98, M, shapes[0][1])
            ys = q4.q4mm_forward_group(Ws, torch.from_numpy(x_np).cuda())
            for i, (y, b) in enumerate(zip(ys, blocks)):
                _, y64, bound = oracle.matmul(b, x_np)
                assert_within_bound(y.cpu().numpy(), y64, bound, "group weight %d M=%d" % (i, M))
    finally:
        q4.q4mm_set_group_m_threshold(thr)
    assert q4.q4_device_status() == q4.Q4_OK
    for W in Ws:
        W.free()


def test_group_argument_errors():
    Ws, _ = _group([(300, 1024), (256, 1024)], 99)
    other = q4.q4_quantize(torch.from_numpy(weights(99, 7, 128, 512)).cuda())
    lib = q4.raw_library()
    x = torch.zeros((4, 1024), device="cuda")
    ys = [torch.zeros((4, W.N), device="cuda") for W in Ws]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(handles, outs, M=4, flags=0, xp=None):
        hw = (ctypes.c_void_p * max(1, len(handles)))(*handles)
        hy = (ctypes.c_void_p * max(1, len(outs)))(*outs)
        return lib.q4mm_forward_group(hw, len(handles), ctypes.c_void_p(xp or x.data_ptr()), hy, M,
                                      flags, stream)

    hs = [W.handle for W in Ws]
    ps = [y.data_ptr() for y in ys]
    assert call(hs, ps) == q4.Q4_OK
    assert call([], []) == q4.Q4_ERR_INVALID_ARG
    assert call(hs * 3, ps * 3) == q4.Q4_ERR_INVALID_ARG                    # 6 > Q4MM_GROUP_MAX
    assert call([hs[0], other.handle], ps) == q4.Q4_ERR_INVALID_ARG         # K differs
    assert call(hs, [ps[0], None]) == q4.Q4_ERR_INVALID_ARG                 # null output
    assert call(hs, [ps[0], ps[1] + 4]) == q4.Q4_ERR_ALIGN
    assert call(hs, ps, flags=q4.Q4MM_FORCE_SIMT) == q4.Q4_ERR_INVALID_ARG
    assert call(hs, ps, flags=q4.Q4MM_FORCE_TC | q4.Q4MM_FORCE_MMA) == q4.Q4_ERR_INVALID_ARG
    assert call(hs, ps, M=q4.Q4MM_M_MAX + 1) == q4.Q4_ERR_SHAPE
    assert call(hs, ps, M=0) == q4.Q4_OK
    torch.cuda.synchronize()
    for W in Ws + [other]:
        W.free()

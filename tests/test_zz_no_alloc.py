"""GPU checks of q4mm_forward_noalloc, the compute call that allocates no
device memory (its scratch is a fixed array inside the library).

The file name makes pytest collect it last, so in a full run it also runs
after every other test has used the ordinary entry points in this process;
it must pass alone in a fresh process as well.  Every call goes through the C
ABI (the raw ctypes library), and each output is checked against the oracle's
bound, against the ordinary entry point q4mm_forward within twice that bound,
and bit for bit against q4mm_forward_ex(..., Q4MM_FORCE_MMA), which runs the
same kernel with the ordinary scratch.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, weights

pytestmark = pytest.mark.gpu

q4 = pytest.importorskip("bit_quantized_matmul_gb300")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(W, x, y, M=None):
    M = x.shape[0] if M is None else M
    return q4.raw_library().q4mm_forward_noalloc(W.handle, ctypes.c_void_p(x.data_ptr()),
                                                 ctypes.c_void_p(y.data_ptr()), M, _stream())


def _setup(N, K, c, m):
    w = weights(c, m, N, K)
    W = q4.q4_quantize(torch.from_numpy(w).cuda())
    return W, oracle.quantize(w)


def _partial_need(W, M):
    _, _, splits = q4.q4mm_plan_info(W, M, q4.Q4MM_FORCE_MMA)
    n_pad = (W.N + 127) // 128 * 128
    return 0 if splits <= 1 else splits * min(M, 16) * n_pad * 8


# (N, K, token-row counts): ragged tiles, a many-way K split with launches
# of 16 + ... rows, the largest scratch of a 7B layer (q_proj at M >= 16), a
# one-split shape and a 7B down projection (five K splits).  The ordinary
# entry point converts the activations of row-group launches of 4 to 8 rows
# in a separate pre-conversion pass; this entry point converts them inside
# the kernel, so the bit-for-bit check below also pins that the pass writes
# the same bytes.
CASES = [
    (300, 1024, (1, 5, 17)),
    (512, 3584, (1, 4, 8, 16, 40)),
    (3584, 3584, (16,)),
    (18944, 3584, (3,)),
    (3584, 18944, (5, 8)),
    (384, 2080, (4, 7)),      # 65 blocks: an odd count and a partial last chunk of the pass
]


@pytest.mark.parametrize("N,K,Ms", CASES)
def test_noalloc_matches_existing_entry_point_twice(N, K, Ms):
    W, blocks = _setup(N, K, 90, N % 97)
    for M in Ms:
        assert _partial_need(W, M) <= q4.Q4MM_NOALLOC_PARTIAL_BYTES
        x_np = acts(90, M, K, salt=N % 13)
        _, y64, bound = oracle.matmul(blocks, x_np)
        x = torch.from_numpy(x_np).cuda()
        y_fwd = q4.q4mm_forward(W, x)
        y_mma = q4.q4mm_forward_ex(W, x, q4.Q4MM_FORCE_MMA)
        outs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        for y in outs:  # two calls in a row on one stream
            assert _noalloc(W, x, y) == q4.Q4_OK
        torch.cuda.synchronize()
        assert q4.q4_device_status() == q4.Q4_OK
        ref_fwd = y_fwd.cpu().numpy()
        ref_mma = y_mma.cpu().numpy()
        for i, y in enumerate(outs):
            got = y.cpu().numpy()
            what = "noalloc N=%d K=%d M=%d call %d" % (N, K, M, i)
            assert_within_bound(got, y64, bound, what)
            assert np.all(np.abs(got.astype(np.float64) - ref_fwd) <= 2 * bound), what
            assert np.array_equal(got.view(np.uint32), ref_mma.view(np.uint32)), what
    W.free()


def test_pre_conversion_pass_is_launched():
    # a 152-SM device: 512 x 3584 and 384 x 2080 run as row-group CTAs up to 8
    # rows (the pass from 4 rows adds one launch per main launch), 3584 x 18944
    # as five K splits (no pass), 300 x 1024 as row-group CTAs with a K too
    # short for the pass
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("launch plan measured for 152 SMs")
    for (N, K), with_pass, without in (((512, 3584), (4, 8), (1, 3)), ((3584, 18944), (), (1, 5, 8)),
                                       ((384, 2080), (4, 7), (3,)), ((300, 1024), (), (4, 8))):
        W, _ = _setup(N, K, 94, 0)
        for M in with_pass:
            assert q4.q4mm_plan_info(W, M, q4.Q4MM_FORCE_MMA)[1] == 2, (N, K, M)
        for M in without:
            assert q4.q4mm_plan_info(W, M, q4.Q4MM_FORCE_MMA)[1] == 1, (N, K, M)
        W.free()


def test_noalloc_allocates_no_device_memory():
    N, K, M = 512, 3584, 24
    W, _ = _setup(N, K, 91, 0)
    x = torch.from_numpy(acts(91, M, K)).cuda()
    ys = [torch.empty((M, N), device="cuda") for _ in range(3)]
    assert _noalloc(W, x, ys[0]) == q4.Q4_OK  # set-up and first kernel launches
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for y in ys[1:]:
        assert _noalloc(W, x, y) == q4.Q4_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.equal(ys[1], ys[0]) and torch.equal(ys[2], ys[0])
    W.free()


def test_noalloc_rejects_oversized_calls_before_launch():
    # 1024 x 18944: 8 tiles, so a 152-SM device splits K 19 ways and 16 rows
    # need 19 * 16 * 1024 * 8 bytes of partial sums, more than the capacity.
    N, K = 1024, 18944
    W, blocks = _setup(N, K, 92, 0)
    checked_reject = False
    for M in (6, 7, 8, 33):
        x_np = acts(92, M, K)
        x = torch.from_numpy(x_np).cuda()
        y = torch.full((M, N), float("nan"), device="cuda")
        torch.cuda.synchronize()
        st = _noalloc(W, x, y)
        torch.cuda.synchronize()
        if _partial_need(W, M) > q4.Q4MM_NOALLOC_PARTIAL_BYTES:
            assert st == q4.Q4_ERR_SHAPE, M
            assert torch.isnan(y).all(), "a rejected call wrote y"
            checked_reject = True
        else:
            assert st == q4.Q4_OK, M
            _, y64, bound = oracle.matmul(blocks, x_np)
            assert_within_bound(y.cpu().numpy(), y64, bound, "noalloc M=%d" % M)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert checked_reject
    # the ordinary entry point has no such limit
    x = torch.from_numpy(acts(92, 8, K)).cuda()
    y = q4.q4mm_forward(W, x)
    _, y64, bound = oracle.matmul(blocks, acts(92, 8, K))
    assert_within_bound(y.cpu().numpy(), y64, bound, "q4mm_forward M=8")
    W.free()


def test_noalloc_argument_errors():
    N, K = 300, 1024
    W, _ = _setup(N, K, 93, 0)
    x = torch.zeros((8, K), device="cuda")
    y = torch.zeros((8, N), device="cuda")
    lib = q4.raw_library()
    assert _noalloc(W, x, y, M=q4.Q4MM_M_MAX + 1) == q4.Q4_ERR_SHAPE
    assert _noalloc(W, x, y, M=-1) == q4.Q4_ERR_INVALID_ARG
    assert _noalloc(W, x, y, M=0) == q4.Q4_OK
    st = lib.q4mm_forward_noalloc(W.handle, ctypes.c_void_p(x.data_ptr() + 4),
                                  ctypes.c_void_p(y.data_ptr()), 4, _stream())
    assert st == q4.Q4_ERR_ALIGN
    st = lib.q4mm_forward_noalloc(W.handle, ctypes.c_void_p(x.data_ptr()), None, 4, _stream())
    assert st == q4.Q4_ERR_INVALID_ARG
    W.free()

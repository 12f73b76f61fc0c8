"""GPU checks that the single-weight calls never grow the library's scratch.

Creating a weight reserves the largest scratch any q4mm_forward_ex /
q4mm_argmax_ex call on it can need, so those calls, at every M and with
every flag, run without cudaMalloc, cudaFree or a device synchronize (the
steps that would break a CUDA-graph capture or stall other streams).  The
test reads the scratch sizes through q4_scratch_bytes before and after a
sweep of calls and checks that they did not move, and that the reserved
partial-sum area covers each call's split-K need as q4mm_plan_info reports
it.  The outputs themselves are checked against the oracle elsewhere; here
a call on the largest shape is compared with the oracle on a few sampled
rows so that a call that silently skipped work would fail.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, weights

pytestmark = pytest.mark.gpu

q4 = pytest.importorskip("bit_quantized_matmul_gb300")

FLAGS = (0, q4.Q4MM_BATCH_INVARIANT, q4.Q4MM_FORCE_MMA, q4.Q4MM_FORCE_SIMT, q4.Q4MM_FORCE_TC,
         q4.Q4MM_ROW_BY_ROW)
MS = (1, 7, 8, 9, 16, 17, 31, 64, 255, 256, 257, 520)


def _partial_need(W, M, flags):
    path, _, splits = q4.q4mm_plan_info(W, M, flags)
    n_pad = (W.N + 127) // 128 * 128
    # token rows per launch of each path
    rows = {q4.Q4MM_PATH_TC: 256, q4.Q4MM_PATH_MMA: 16, q4.Q4MM_PATH_SIMT: 8}.get(path, 1)
    return 0 if splits <= 1 else splits * min(M, rows) * n_pad * 8


# (N, K): a narrow matrix with a long K (the most split-K partial sums per
# output), and a 7B decoder's down projection.
@pytest.mark.parametrize("N,K", [(640, 16384), (3584, 18944)])
def test_single_weight_calls_do_not_grow_scratch(N, K):
    w = weights(95, N % 89, N, K)
    W = q4.q4_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    before = q4.q4_scratch_bytes()
    xs = {M: torch.from_numpy(acts(95, M, K, salt=N % 11)).cuda() for M in MS}
    need = 0
    last = None
    for flags in FLAGS:
        for M in MS:
            need = max(need, _partial_need(W, M, flags))
            y = q4.q4mm_forward_ex(W, xs[M], flags)
            idx, _ = q4.q4mm_argmax_ex(W, xs[M], flags)
            if flags == 0 and M == MS[-1]:
                last = y
            assert q4.q4_scratch_bytes() == before, "flags %d M %d grew the scratch" % (flags, M)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == q4.Q4_OK
    assert q4.q4_scratch_bytes() == before
    assert before[0] >= need, "reserved partial sums %d < need %d" % (before[0], need)
    assert torch.isfinite(y).all() and int(idx.min()) >= 0 and int(idx.max()) < N
    # a few rows of the largest default call against the oracle
    rows = np.array([0, 1, MS[-1] // 2, MS[-1] - 1])
    blocks = oracle.quantize(w)
    _, y64, bound = oracle.matmul(blocks, xs[MS[-1]].cpu().numpy()[rows])
    assert_within_bound(last.cpu().numpy()[rows], y64, bound, "N=%d K=%d M=%d" % (N, K, MS[-1]))

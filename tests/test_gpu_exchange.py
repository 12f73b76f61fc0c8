"""GPU parity of the split-K exchanges, against the CPU oracle.

The streaming kernel adds the K splits of a tile either inside a thread-block
cluster (at most 4 splits, all clusters resident at once) or through flagged
64-bit words in global memory; the tensor-core kernel either reduce-scatters
among the splits (a launch of one wave) or lets the last CTA of a tile add them
up.  The shapes here are chosen to land on each of those paths on a 152-SM
GB300 (the plan is read back through q4mm_plan_info), and every result is
compared element by element with the oracle's bound.  A second test alternates
shapes that share the counter slots, so that each call depends on the previous
one having reset them."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, plant_near_ties, weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
K = 3584


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    torch.cuda.set_device(0)
    return q4


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _setup(q4, N, config):
    w = weights(config, N % 11, N, K)
    return q4.q4_quantize(torch.from_numpy(w).to(DEV)), oracle.quantize(w)


# (N, K) -> K splits of the streaming kernel on 152 SMs: 32 tiles -> 4, 40 ->
# 3, 63 -> 2 (all three within the GPU's cluster capacity: cluster path); 28
# -> 5 (global-memory path).  The 4- and 5-split shapes use K = 4608: at K up
# to 4096 those tile counts run as row-group CTAs without a K split (below).
STREAM_CASES = [(4000, 4608, 4), (5000, K, 3), (8000, K, 2), (3584, 4608, 5)]


@pytest.mark.parametrize("N,KK,splits", STREAM_CASES)
def test_streaming_split_exchange_matches_oracle(q4, N, KK, splits):
    w = weights(70, N % 11, N, KK)
    W, blocks = q4.q4_quantize(torch.from_numpy(w).to(DEV)), oracle.quantize(w)
    _, _, s = q4.q4mm_plan_info(W, 1, q4.Q4MM_FORCE_MMA)
    if _sms() == 152:
        assert s == splits
    for M in (1, 3, 8, 11):  # one, one, two and three column groups
        x = acts(70, M, KK, salt=N)
        y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), q4.Q4MM_FORCE_MMA).cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert_within_bound(y, y64, bound, "mma N=%d K=%d M=%d" % (N, KK, M))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


@pytest.mark.parametrize("N", [4000, 3584, 640])
def test_streaming_row_group_ctas_match_oracle(q4, N):
    # K = 3584 with 32, 28 and 5 tiles: four CTAs per tile fit on the SMs, so
    # each CTA takes one 32-row group pair over the whole K (no K split)
    W, blocks = _setup(q4, N, 72)
    _, _, s = q4.q4mm_plan_info(W, 1, q4.Q4MM_FORCE_MMA)
    assert s == 1
    for M in (1, 2, 3, 5, 8, 9, 16):
        x = acts(72, M, K, salt=N)
        y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), q4.Q4MM_FORCE_MMA).cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert_within_bound(y, y64, bound, "row groups N=%d M=%d" % (N, M))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_streaming_cluster_greedy_pick_matches_oracle(q4):
    # the greedy pick always takes the global-memory exchange, also on a
    # shape whose plain calls use clusters
    N = 4000
    W, blocks = _setup(q4, N, 71)
    M = 6
    x = acts(71, M, K)
    idx, mx = q4.q4mm_argmax(W, torch.from_numpy(x).to(DEV))
    _, y64, bound = oracle.matmul(blocks, x)
    idx = idx.cpu().numpy()
    for m in range(M):
        order = np.argsort(-y64[m], kind="stable")
        if y64[m, order[0]] - y64[m, order[1]] > bound[m, order[0]]:
            assert idx[m] == order[0], m
        assert abs(float(mx.cpu().numpy()[m]) - y64[m, idx[m]]) <= bound[m, idx[m]]
    W.free()


# tensor-core path: 3584 rows = 28 tiles split 5 ways at these M (one wave:
# reduce-scatter); batch-invariant mode plans for one token tile, so M = 100
# there runs several waves (last-CTA exchange)
@pytest.mark.parametrize("M,flags", [(16, "tc"), (48, "tc"), (64, "tc"), (100, "tc"), (100, "inv_tc")])
def test_tensor_core_split_exchange_matches_oracle(q4, M, flags):
    N = 3584
    W, blocks = _setup(q4, N, 72)
    f = q4.Q4MM_FORCE_TC if flags == "tc" else (q4.Q4MM_FORCE_TC | q4.Q4MM_BATCH_INVARIANT)
    x = acts(72, M, K, salt=M)
    y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), f).cpu().numpy()
    _, y64, bound = oracle.matmul(blocks, x)
    assert_within_bound(y, y64, bound, "tc %s M=%d" % (flags, M))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_alternating_shapes_share_counter_slots(q4):
    # calls of different split counts and exchanges use the same counter slots
    # and partial-sum words one after the other (row-group CTAs with none in
    # between); every result stays right.  Batch-invariant mode keeps the K
    # split: clusters of 4 for 4000 rows, global words for 3584.
    mma, inv = q4.Q4MM_FORCE_MMA, q4.Q4MM_BATCH_INVARIANT
    cases = [(4000, 8, mma), (4000, 3, mma | inv), (300, 3, mma), (3584, 5, mma | inv),
             (3584, 32, q4.Q4MM_FORCE_TC), (3584, 5, mma), (8000, 1, mma), (512, 20, q4.Q4MM_FORCE_TC)]
    prepared = []
    for i, (N, M, f) in enumerate(cases):
        W, blocks = _setup(q4, N, 73 + i)
        x = acts(73, M, K, salt=i)
        _, y64, bound = oracle.matmul(blocks, x)
        prepared.append((W, torch.from_numpy(x).to(DEV), f, y64, bound, N, M))
    for rep in range(3):
        for W, xd, f, y64, bound, N, M in prepared:
            y = q4.q4mm_forward_ex(W, xd, f).cpu().numpy()
            assert_within_bound(y, y64, bound, "rep %d N=%d M=%d" % (rep, N, M))
    assert q4.q4_device_status() == q4.Q4_OK
    for p in prepared:
        p[0].free()


@pytest.mark.parametrize("shapes", [
    [(155 * 128 - 37, 1024)],                 # 155 tiles (odd), ragged last tile
    [(153 * 128 - 5, 1024), (300, 1024)],     # a CTA's two tiles in different weights
])
def test_two_tile_ctas_match_oracle(q4, shapes):
    # more tiles than SMs and one K split: each CTA streams two tiles over the
    # whole K (one or two column groups); three groups keep one tile per CTA
    Ws, blocks = [], []
    for i, (N, KK) in enumerate(shapes):
        w = weights(74, i, N, KK)
        Ws.append(q4.q4_quantize(torch.from_numpy(w).to(DEV)))
        blocks.append(oracle.quantize(w))
    _, _, s = q4.q4mm_plan_info(Ws[0], 1, q4.Q4MM_FORCE_MMA)
    assert s == 1
    for M in (1, 2, 3, 5, 8, 11):
        x = acts(74, M, shapes[0][1], salt=len(shapes))
        xd = torch.from_numpy(x).to(DEV)
        if len(Ws) == 1:
            ys = [q4.q4mm_forward_ex(Ws[0], xd, q4.Q4MM_FORCE_MMA)]
        else:
            ys = q4.q4mm_forward_group(Ws, xd, flags=q4.Q4MM_FORCE_MMA)
        for i, (y, b) in enumerate(zip(ys, blocks)):
            _, y64, bound = oracle.matmul(b, x)
            assert_within_bound(y.cpu().numpy(), y64, bound, "two tiles weight %d M=%d" % (i, M))
    assert q4.q4_device_status() == q4.Q4_OK
    for W in Ws:
        W.free()


def test_two_tile_ctas_greedy_pick_matches_oracle(q4):
    # the greedy pick on two-tile CTAs: 155 tiles on 78 CTAs (the last with
    # one tile), each tile folded into the per-row maximum on its own.  Rows
    # 70 and 200 (two tiles of the first CTA) and 19750 (the lone last tile)
    # hold the same weights, so an exact tie across tiles picks row 70.
    N, KK = 155 * 128 - 37, 1024
    w = weights(75, 0, N, KK)
    w[200] = w[70]
    w[19750] = w[70]
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    _, _, s = q4.q4mm_plan_info(W, 1, q4.Q4MM_FORCE_MMA)
    assert s == 1
    rng = np.random.default_rng(75)
    for M in (1, 2, 5, 8, 11):
        x = acts(75, M, KK)
        x, planted = plant_near_ties(blocks, x, list(range(1, M, 2)), rng)
        wd = oracle.dequantize(blocks[[70]]).astype(np.float64)[0]
        x[0] = (wd / np.linalg.norm(wd) * 40).astype(np.float32)  # row 0: the exact tie
        xd = torch.from_numpy(x).to(DEV)
        idx, mx = q4.q4mm_argmax_ex(W, xd, q4.Q4MM_FORCE_MMA)
        idx, mx = idx.cpu().numpy(), mx.cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert idx[0] == 70, M
        for m in range(M):
            top = np.argsort(-y64[m], kind="stable")
            margin = y64[m, top[0]] - y64[m, top[1]]
            if m in planted:
                assert margin > bound[m, top[0]] + bound[m, top[1]], "planted gap below the bound"
            # exact wherever the oracle's top-2 margin exceeds the bound at the top index
            if margin > bound[m, top[0]]:
                assert idx[m] == top[0], (M, m)
            assert abs(float(mx[m]) - y64[m, idx[m]]) <= bound[m, idx[m]]
        # the same sums as the call that writes y (both on two-tile CTAs)
        yf = q4.q4mm_forward_ex(W, xd, q4.Q4MM_FORCE_MMA).cpu().numpy()
        assert np.array_equal(np.argmax(yf, axis=1), idx)
        assert np.array_equal(yf.max(axis=1).view(np.uint32), mx.view(np.uint32))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


SIXTEEN_ROW_CASES = [(4000, 4608), (3584, 3584), (155 * 128 - 37, 1024), (300, 1024)]


@pytest.mark.parametrize("N,KK", SIXTEEN_ROW_CASES)
def test_sixteen_row_launches_match_oracle(q4, N, KK):
    # 9 to 16 token rows in one streaming launch (three or four column groups,
    # one row group per warp, two K slices per CTA) over each exchange on a
    # 152-SM device: clusters (32 tiles x 4 splits), flagged global words
    # (28 tiles x 5 splits; a ragged 3-tile weight x 8) and one K split (155
    # tiles); 20 and 23 rows add a launch of 4 or 7 rows
    w = weights(76, 0, N, KK)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    if (N, KK) == (3584, 3584) and torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert q4.q4mm_plan_info(W, 1, q4.Q4MM_FORCE_MMA)[2] == 1    # row-group CTAs
        assert q4.q4mm_plan_info(W, 16, q4.Q4MM_FORCE_MMA)[1:] == (1, 5)  # one launch, 5 splits
    for M in (9, 12, 14, 16, 20, 23):
        x = acts(76, M, KK)
        y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), q4.Q4MM_FORCE_MMA).cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert_within_bound(y, y64, bound, "N=%d K=%d M=%d" % (N, KK, M))
    # the greedy pick at 16 rows adds the splits in the order of the call that
    # writes y, so it picks the same indices and values
    xd = torch.from_numpy(acts(77, 16, KK)).to(DEV)
    idx, mx = q4.q4mm_argmax_ex(W, xd, q4.Q4MM_FORCE_MMA)
    yf = q4.q4mm_forward_ex(W, xd, q4.Q4MM_FORCE_MMA).cpu().numpy()
    assert np.array_equal(idx.cpu().numpy(), np.argmax(yf, axis=1))
    assert np.array_equal(mx.cpu().numpy().view(np.uint32), yf.max(axis=1).view(np.uint32))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()

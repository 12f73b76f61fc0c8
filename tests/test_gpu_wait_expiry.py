"""GPU test of the bounded waits: every wait a kernel makes on another of its
roles or CTAs gives up after a bound, records Q4_ERR_TIMEOUT and returns, so
that a hand-off that never comes costs the call, not the GPU.

The test shortens the bound to 2 ms (``q4mm_set_wait_limit_ns``) and makes the
launches withhold their first hand-off (``q4mm_set_stall_for_test``), which
makes each kind of wait run out:

  ring        converter warps that hand over no chunk; the compute warps'
              wait on the ring runs out (9 to 16 rows, one row group a warp)
  two-tile    the same ring in CTAs that stream two tiles over the whole K,
              for the fused greedy pick (keys and completion count left
              mid-launch)
  split poll  CTAs of a K split that store no partial sum; the last CTA's
              poll of its peers' words runs out
  tensor core a producer that issues no copy; the MMA issuer's, the
              converters' and the epilogue's waits run out, and TMEM must
              still be released

Each stalled call must end within seconds and ``q4_device_status`` must
report Q4_ERR_TIMEOUT.  With the settings back to their defaults the same
calls must then match the oracle: the scratch words were reset and the
tensor-core CTAs released their TMEM (a leaked allocation would leave the
next tensor-core launch unable to run)."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LIMIT_NS = 2_000_000


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    torch.cuda.set_device(0)
    yield q4
    q4.q4mm_set_stall_for_test(False)
    q4.q4mm_set_wait_limit_ns(0)


def _quant(q4, config, N, K):
    w = weights(config, 0, N, K)
    return q4.q4_quantize(torch.from_numpy(w).to(DEV)), oracle.quantize(w)


# (name, N, K, M, flags, greedy pick, expected path, K splits: None = any, ">4" = flagged-word exchange)
CASES = [
    ("ring", 1024, 8192, 12, "mma", False, "mma", None),
    ("two_tile_greedy", 20480, 8192, 1, 0, True, "mma", 1),
    ("split_poll", 1024, 18944, 1, 0, False, "mma", ">4"),
    ("tensor_core", 1024, 4096, 32, "tc", False, "tc", None),
]


def _flags(q4, f):
    return {0: 0, "mma": q4.Q4MM_FORCE_MMA, "tc": q4.Q4MM_FORCE_TC}[f]


def _path(q4, name):
    return {"mma": q4.Q4MM_PATH_MMA, "tc": q4.Q4MM_PATH_TC}[name]


def _run(q4, W, xd, flags, greedy):
    if greedy:
        return q4.q4mm_argmax_ex(W, xd, flags)
    return q4.q4mm_forward_ex(W, xd, flags)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_stalled_waits_time_out_then_calls_recover(q4, case):
    name, N, K, M, f, greedy, path, splits = case
    flags = _flags(q4, f)
    W, blocks = _quant(q4, 90 + CASES.index(case), N, K)
    p, _, s = q4.q4mm_plan_info(W, M, flags)
    assert p == _path(q4, path), (name, p)
    if splits == ">4":
        assert s > 4, (name, s)
    elif splits is not None:
        assert s == splits, (name, s)
    x = acts(90, M, K, salt=N)
    xd = torch.from_numpy(x).to(DEV)
    assert q4.q4_device_status() == q4.Q4_OK

    q4.q4mm_set_wait_limit_ns(LIMIT_NS)
    q4.q4mm_set_stall_for_test(True)
    try:
        t0 = time.perf_counter()
        _run(q4, W, xd, flags, greedy)
        torch.cuda.synchronize()
        took = time.perf_counter() - t0
        status = q4.q4_device_status()
    finally:
        q4.q4mm_set_stall_for_test(False)
        q4.q4mm_set_wait_limit_ns(0)
    assert status == q4.Q4_ERR_TIMEOUT, (name, status)
    assert took < 5.0, (name, took)
    assert q4.q4_device_status() == q4.Q4_OK  # read once, then cleared

    # defaults again: the same call, twice (the second one sees whatever the
    # first left in the scratch words), against the oracle
    _, y64, bound = oracle.matmul(blocks, x)
    for _ in range(2):
        out = _run(q4, W, xd, flags, greedy)
        if greedy:
            idx = out[0].cpu().numpy()
            mx = out[1].cpu().numpy()
            for m in range(M):
                top = np.argsort(-y64[m], kind="stable")
                if y64[m, top[0]] - y64[m, top[1]] > bound[m, top[0]]:
                    assert idx[m] == top[0], (name, m)
                assert abs(float(mx[m]) - y64[m, idx[m]]) <= bound[m, idx[m]]
        else:
            assert_within_bound(out.cpu().numpy(), y64, bound, name)
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_limit_setting_round_trip(q4):
    # the default bound is restored by 0, and a normal call under a short bound
    # does not time out (the bound only cuts waits that would not end)
    W, blocks = _quant(q4, 99, 1024, 8192)
    x = acts(99, 12, 8192)
    xd = torch.from_numpy(x).to(DEV)
    q4.q4mm_set_wait_limit_ns(LIMIT_NS)
    try:
        y = q4.q4mm_forward_ex(W, xd, q4.Q4MM_FORCE_MMA).cpu().numpy()
    finally:
        q4.q4mm_set_wait_limit_ns(0)
    assert q4.q4_device_status() == q4.Q4_OK
    _, y64, bound = oracle.matmul(blocks, x)
    assert_within_bound(y, y64, bound, "short bound, no stall")
    W.free()

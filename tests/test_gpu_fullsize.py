"""GPU parity at the full workload sizes (Qwen2.5-7B decode linears, the
M=124 mixed continuous-batching step, the 152064 x 3584 LM head, the M sweep
to 256), on sampled outputs the oracle computes one by one, plus bit-exact
quantizer output and bitwise batch invariance at full size."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_helpers import acts, assert_within_bound, plant_near_ties, weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LIN = synthetic.QWEN7B_LINEARS
MATRIX_ID = {name: i for i, name in enumerate(LIN)}


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    torch.cuda.set_device(0)
    return q4


_cache = {}


def _weight(q4, config, name, N=None, K=None):
    key = (config, name)
    if key not in _cache:
        if N is None:
            N, K = LIN[name]
        w = weights(config, MATRIX_ID.get(name, 15), N, K)
        blocks = oracle.quantize(w)
        W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
        assert np.array_equal(q4.q4_export_blocks(W), blocks), "quantizer differs at %s" % name
        _cache.clear()
        _cache[key] = (W, blocks)
    return _cache[key]


def _sampled_check(q4, W, blocks, x, flags, rng, n_per_row=1024, what=""):
    M, K = x.shape
    N = blocks.shape[0]
    y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), flags).cpu().numpy()
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(n_per_row, N), replace=False)]))
    pairs = np.array([(m, n) for m in range(M) for n in cols], np.int64)
    _, y64, bound = oracle.matmul_pairs(blocks, x, pairs)
    got = y[pairs[:, 0], pairs[:, 1]]
    return assert_within_bound(got, y64, bound, what)


@pytest.mark.parametrize("name", ["q_proj", "k_proj", "o_proj", "gate_proj", "down_proj"])
def test_qwen7b_linear_decode_parity(q4, name):
    W, blocks = _weight(q4, 2, name)
    rng = np.random.default_rng(MATRIX_ID[name])
    for M in (1, 2, 3, 4, 5, 8):
        x = acts(2, M, W.K)
        _sampled_check(q4, W, blocks, x, 0, rng, what="%s M=%d" % (name, M))
    x = acts(2, 8, W.K, salt=1)
    for flags in (q4.Q4MM_FORCE_SIMT, q4.Q4MM_FORCE_TC, q4.Q4MM_BATCH_INVARIANT):
        _sampled_check(q4, W, blocks, x, flags, rng, n_per_row=512, what="%s flags=%d" % (name, flags))
    assert q4.q4_device_status() == q4.Q4_OK


@pytest.mark.parametrize("group", [("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj")])
def test_qwen7b_grouped_calls_as_benchmarked(q4, group):
    """The grouped calls of the benchmark step (q/k/v: row-group CTAs, with the
    activation pre-conversion pass from M = 4; gate/up: two-tile CTAs) at the
    7B shapes and the step's M, on sampled outputs of every weight."""
    cache = {}
    for i, name in enumerate(group):
        N, K = LIN[name]
        w = weights(6, MATRIX_ID[name], N, K)
        cache[name] = (q4.q4_quantize(torch.from_numpy(w).to(DEV)), oracle.quantize(w))
        del w
    Ws = [cache[n][0] for n in group]
    rng = np.random.default_rng(len(group))
    K = Ws[0].K
    for M in (1, 2, 3, 4, 5, 8):
        x = acts(6, M, K, salt=M)
        ys = q4.q4mm_forward_group(Ws, torch.from_numpy(x).to(DEV))
        for name, y in zip(group, ys):
            blocks = cache[name][1]
            N = blocks.shape[0]
            cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(512, N), replace=False)]))
            pairs = np.array([(m, n) for m in range(M) for n in cols], np.int64)
            _, y64, bound = oracle.matmul_pairs(blocks, x, pairs)
            got = y.cpu().numpy()[pairs[:, 0], pairs[:, 1]]
            assert_within_bound(got, y64, bound, "group %s M=%d" % (name, M))
    assert q4.q4_device_status() == q4.Q4_OK
    for W in Ws:
        W.free()


def test_qwen7b_kv_full_elementwise(q4):
    W, blocks = _weight(q4, 2, "v_proj")
    for M in (1, 5, 8):
        x = acts(2, M, W.K, salt=2)
        y = q4.q4mm_forward(W, torch.from_numpy(x).to(DEV)).cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert_within_bound(y, y64, bound, "v_proj M=%d" % M)


@pytest.mark.parametrize("name", ["gate_proj", "down_proj"])
def test_qwen7b_gate_down_full_elementwise_m8(q4, name):
    # every element of the output at M = 8, default path and batch-invariant mode
    W, blocks = _weight(q4, 2, name)
    x = acts(2, 8, W.K, salt=4)
    _, y64, bound = oracle.matmul(blocks, x)
    for flags in (0, q4.Q4MM_BATCH_INVARIANT):
        y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), flags).cpu().numpy()
        assert_within_bound(y, y64, bound, "%s M=8 flags=%d" % (name, flags))


def test_896_config_full_elementwise(q4):
    W, blocks = _weight(q4, 0, "square896", 896, 896)
    for M in (1, 2, 4):
        x = acts(0, M, 896)
        for flags in (0, q4.Q4MM_BATCH_INVARIANT, q4.Q4MM_FORCE_SIMT):
            y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), flags).cpu().numpy()
            _, y64, bound = oracle.matmul(blocks, x)
            assert_within_bound(y, y64, bound, "896 M=%d" % M)


@pytest.mark.parametrize("mode", ["streaming", "tensor_core"])
@pytest.mark.parametrize("name", ["gate_proj", "up_proj", "down_proj"])
def test_mixed_step_m124_parity_and_invariance(q4, name, mode):
    """120 prefill rows + 4 verify rows in one call (continuous batching), in
    the batch-invariant mode of the streaming kernel or of the tensor cores."""
    W, blocks = _weight(q4, 3, name)
    rng = np.random.default_rng(124)
    K = W.K
    prefill = acts(3, 120, K)
    verify = acts(3, 4, K, salt=1)
    x = np.concatenate([prefill, verify])
    if mode == "streaming":  # the default mode once, on the same batch
        _sampled_check(q4, W, blocks, x, 0, rng, n_per_row=256, what="%s M=124" % name)
    inv = q4.Q4MM_BATCH_INVARIANT | (q4.Q4MM_FORCE_TC if mode == "tensor_core" else 0)
    xd = torch.from_numpy(x).to(DEV)
    y124 = q4.q4mm_forward_ex(W, xd, inv).cpu().numpy()
    y4 = q4.q4mm_forward_ex(W, xd[120:].contiguous(), inv).cpu().numpy()
    assert np.array_equal(y124[120:].view(np.uint32), y4.view(np.uint32))
    for r in rng.choice(124, size=16, replace=False):
        y1 = q4.q4mm_forward_ex(W, xd[r:r + 1].contiguous(), inv).cpu().numpy()
        assert np.array_equal(y124[r].view(np.uint32), y1[0].view(np.uint32)), r
    redrawn = acts(3, 124, K, salt=7)
    redrawn[120:] = verify
    y_re = q4.q4mm_forward_ex(W, torch.from_numpy(redrawn).to(DEV), inv).cpu().numpy()
    assert np.array_equal(y_re[120:].view(np.uint32), y124[120:].view(np.uint32))
    cols = rng.choice(W.N, size=256, replace=False)
    pairs = np.array([(m, n) for m in (0, 119, 120, 123) for n in cols], np.int64)
    _, y64, bound = oracle.matmul_pairs(blocks, x, pairs)
    assert_within_bound(y124[pairs[:, 0], pairs[:, 1]], y64, bound, "%s %s invariant M=124" % (name, mode))


def test_gate_m_sweep_parity(q4):
    W, blocks = _weight(q4, 4, "gate_proj")
    rng = np.random.default_rng(77)
    for M in (6, 16, 17, 32, 64, 128, 256):
        x = acts(4, M, W.K)
        _sampled_check(q4, W, blocks, x, 0, rng, n_per_row=64, what="gate M=%d" % M)
        _sampled_check(q4, W, blocks, x, q4.Q4MM_FORCE_MMA, rng, n_per_row=32, what="gate mma M=%d" % M)


def test_lm_head_argmax_planted_near_ties(q4):
    N, K = synthetic.LM_HEAD
    W, blocks = _weight(q4, 3, "lm_head", N, K)
    rng = np.random.default_rng(2024)
    for M in (1, 4, 16):
        x = acts(3, M, K, salt=3)
        x, planted = plant_near_ties(blocks, x, list(range(0, M, 2)), rng)
        for flags in (0, q4.Q4MM_BATCH_INVARIANT):
            idx, mx = q4.q4mm_argmax_ex(W, torch.from_numpy(x).to(DEV), flags)
            idx, mx = idx.cpu().numpy(), mx.cpu().numpy()
            y, y64, bound = oracle.matmul(blocks, x)
            ref = oracle.argmax(y)
            for m in range(M):
                top = np.argsort(-y64[m], kind="stable")
                margin = y64[m, top[0]] - y64[m, top[1]]
                if m in planted:
                    assert margin > bound[m, top[0]] + bound[m, top[1]], "planted gap below the bound"
                # exact wherever the oracle's top-2 margin exceeds the bound at the top index
                if margin > bound[m, top[0]]:
                    assert idx[m] == ref[m], (M, m, flags, planted.get(m))
                else:
                    assert y64[m, ref[m]] - y64[m, idx[m]] <= bound[m, ref[m]] + bound[m, idx[m]]
                assert abs(float(mx[m]) - y64[m, idx[m]]) <= bound[m, idx[m]]
    assert q4.q4_device_status() == q4.Q4_OK

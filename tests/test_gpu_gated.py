"""GPU parity of the gated MLP step, h = SiLU(x Wg^T) * (x Wu^T) (the hidden
state between the gate/up and down projections of the Qwen2.5-7B decoder
layer), against the CPU oracle: the oracle's fp64 gate and up outputs through
``oracle.mlp.silu_mul``, within the tolerance propagated from their bounds
(``oracle.mlp.silu_mul_bound``).  The down projection of the GPU's h is
checked against the oracle's matmul of that same h.  Where the grouped call
adds up g and u the same way (whole-K two-tile CTAs for the 7B gate/up at up
to 8 rows, the tensor-core path, batch-invariant mode), h is also checked
against SiLU(g) * u formed on the host from that call's own g and u."""
import numpy as np
import pytest
import torch

import oracle
from oracle import mlp
import synthetic
from gpu_helpers import acts, assert_within_bound, weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    torch.cuda.set_device(0)
    return q4


def _quant(q4, config, matrix, N, K):
    w = weights(config, matrix, N, K)
    return q4.q4_quantize(torch.from_numpy(w).to(DEV)), oracle.quantize(w)


def _check_h(h, g64, bg, u64, bu, what):
    ref = mlp.silu_mul(g64, u64)
    bound = mlp.silu_mul_bound(g64, u64, bg, bu)
    err = np.abs(h.astype(np.float64) - ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), "%s: err/bound %.3g at %s" % (what, float((err / bound)[worst]), worst)


def _check_against_group(q4, Wg, Wu, xd, h, flags):
    # h against SiLU(g) * u from the grouped call's own outputs (fp64 on the host)
    g, u = q4.q4mm_forward_group([Wg, Wu], xd, flags=flags)
    g = g.cpu().numpy().astype(np.float64)
    u = u.cpu().numpy().astype(np.float64)
    ref = mlp.silu(g) * u
    assert np.all(np.abs(h - ref) <= 2.0 ** -20 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("N,K,Ms", [(300, 1024, (1, 5, 8, 11)), (1000, 3584, (1, 3, 16, 40))])
def test_gated_small_shapes_full_elementwise(q4, N, K, Ms):
    Wg, bg_blocks = _quant(q4, 80, 0, N, K)
    Wu, bu_blocks = _quant(q4, 80, 1, N, K)
    for M in Ms:
        x = acts(80, M, K, salt=N)
        xd = torch.from_numpy(x).to(DEV)
        _, g64, bg = oracle.matmul(bg_blocks, x)
        _, u64, bu = oracle.matmul(bu_blocks, x)
        inv_tc = q4.Q4MM_BATCH_INVARIANT | q4.Q4MM_FORCE_TC
        for flags in (0, q4.Q4MM_BATCH_INVARIANT, q4.Q4MM_FORCE_MMA, inv_tc):
            h = q4.q4mm_forward_gated(Wg, Wu, xd, flags=flags).cpu().numpy()
            _check_h(h, g64, bg, u64, bu, "N=%d M=%d flags=%d" % (N, M, flags))
            if flags in (q4.Q4MM_BATCH_INVARIANT, inv_tc):  # the same grouped call, then SiLU * up
                _check_against_group(q4, Wg, Wu, xd, h, flags)
                if M > 1:  # and row 1 alone gives the same bits
                    h1 = q4.q4mm_forward_gated(Wg, Wu, xd[1:2].contiguous(), flags=flags).cpu().numpy()
                    assert np.array_equal(h1[0].view(np.uint32), h[1].view(np.uint32)), (M, flags)
    assert q4.q4_device_status() == q4.Q4_OK
    Wg.free()
    Wu.free()


def test_gated_qwen7b_then_down(q4):
    N, K = synthetic.QWEN7B_LINEARS["gate_proj"]
    Wg, bg_blocks = _quant(q4, 81, 0, N, K)
    Wu, bu_blocks = _quant(q4, 81, 1, N, K)
    Nd, Kd = synthetic.QWEN7B_LINEARS["down_proj"]
    Wd, bd_blocks = _quant(q4, 81, 2, Nd, Kd)
    rng = np.random.default_rng(81)
    for M, flags in ((1, 0), (8, 0), (8, q4.Q4MM_BATCH_INVARIANT), (124, 0)):
        x = acts(81, M, K)
        xd = torch.from_numpy(x).to(DEV)
        hd = q4.q4mm_forward_gated(Wg, Wu, xd, flags=flags)
        h = hd.cpu().numpy()
        if M <= 8:
            _, g64, bg = oracle.matmul(bg_blocks, x)
            _, u64, bu = oracle.matmul(bu_blocks, x)
            _check_h(h, g64, bg, u64, bu, "7B M=%d flags=%d" % (M, flags))
        else:
            cols = rng.choice(N, size=256, replace=False)
            pairs = np.array([(m, n) for m in range(M) for n in cols], np.int64)
            _, g64, bg = oracle.matmul_pairs(bg_blocks, x, pairs)
            _, u64, bu = oracle.matmul_pairs(bu_blocks, x, pairs)
            _check_h(h[pairs[:, 0], pairs[:, 1]], g64, bg, u64, bu, "7B M=%d" % M)
        _check_against_group(q4, Wg, Wu, xd, h, flags)
        # the down projection of this h, against the oracle on the same h
        y = q4.q4mm_forward_ex(Wd, hd, flags).cpu().numpy()
        if M <= 8:
            _, y64, bound = oracle.matmul(bd_blocks, h)
            assert_within_bound(y, y64, bound, "down(h) M=%d" % M)
        else:
            cols = rng.choice(Nd, size=256, replace=False)
            pairs = np.array([(m, n) for m in range(M) for n in cols], np.int64)
            _, y64, bound = oracle.matmul_pairs(bd_blocks, h, pairs)
            assert_within_bound(y[pairs[:, 0], pairs[:, 1]], y64, bound, "down(h) M=%d" % M)
    assert q4.q4_device_status() == q4.Q4_OK
    for W in (Wg, Wu, Wd):
        W.free()


def test_gated_argument_errors(q4):
    Wg, _ = _quant(q4, 82, 0, 300, 1024)
    Wu, _ = _quant(q4, 82, 1, 300, 1024)
    Wo, _ = _quant(q4, 82, 2, 256, 1024)
    x = torch.zeros((4, 1024), device=DEV)
    h = torch.zeros((4, 300), device=DEV)
    lib = q4.raw_library()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.q4mm_forward_gated(Wg.handle, Wo.handle, x.data_ptr(), h.data_ptr(), 4, 0, s) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_gated(Wg.handle, Wu.handle, x.data_ptr(), h.data_ptr(), 4, q4.Q4MM_FORCE_SIMT, s) == \
        q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_gated(Wg.handle, Wu.handle, x.data_ptr(), h.data_ptr(), 4,
                                  q4.Q4MM_FORCE_TC | q4.Q4MM_FORCE_MMA, s) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_gated(Wg.handle, Wu.handle, x.data_ptr() + 4, h.data_ptr(), 4, 0, s) == q4.Q4_ERR_ALIGN
    assert lib.q4mm_forward_gated(Wg.handle, Wu.handle, x.data_ptr(), h.data_ptr(), 0, 0, s) == q4.Q4_OK
    for W in (Wg, Wu, Wo):
        W.free()

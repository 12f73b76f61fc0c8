"""Pins for the CPU oracle, each against something other than the oracle itself.

- a hand-worked block (tests/golden/q4_worked_block.txt);
- the IEEE binary16 conversion against numpy's float16 cast;
- the quantizer against a brute-force nearest-level search;
- the round-trip error bound of the block rule;
- exact rational arithmetic (fractions) for the fp64 matmul on dyadic inputs;
- linearity in x, a closed form on constructed blocks, numpy's fp64 matmul;
- the greedy pick against the scores the continuous-batching investigation
  prints (tests/golden/greedy_top2_logits.txt) and numpy's argmax.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _worked():
    kv, _ = read_golden("q4_worked_block.txt")
    x = np.array([float(v) for v in kv["x"].split()], dtype=np.float32)
    q = [int(v) for v in kv["q"].split()]
    return kv, x, q


def _q_of(blocks):
    """Unpack canonical blocks [N, nb, 18] -> q [N, nb*32] (format definition)."""
    lo = blocks[..., 2:] & 0x0F
    hi = blocks[..., 2:] >> 4
    q = np.concatenate([lo, hi], axis=-1)
    return q.reshape(blocks.shape[0], -1).astype(np.int64)


def _d_of(blocks):
    return (blocks[..., 0].astype(np.uint16) | (blocks[..., 1].astype(np.uint16) << 8)).view(np.float16)


# ---------------------------------------------------------------- worked block

def test_worked_block_q_and_bytes():
    kv, x, q = _worked()
    blk = oracle.quantize(x.reshape(1, 32))
    assert blk.shape == (1, 1, 18)
    assert blk.tobytes().hex() == kv["bytes"]
    assert _q_of(blk)[0].tolist() == q
    assert "%04x" % (int(blk[0, 0, 0]) | int(blk[0, 0, 1]) << 8) == kv["d16"]


def test_worked_block_dequant_errors_and_dots():
    kv, x, q = _worked()
    blk = oracle.quantize(x.reshape(1, 32))
    w = oracle.dequantize(blk)[0]
    err = np.abs(x.astype(np.float64) - w.astype(np.float64))
    assert err[1] == float(kv["err_1"])
    assert err[11] == float(kv["err_11"])
    assert err[2] == float(kv["err_2"]) and err[3] == float(kv["err_2"])
    assert abs(err[6] - float(kv["err_6"])) < 1e-7 and abs(err[7] - float(kv["err_6"])) < 1e-7
    a1 = np.ones((1, 32), np.float32)
    a5 = ((np.arange(32) % 5) - 2).astype(np.float32).reshape(1, 32)
    y1, _, _ = oracle.matmul(blk, a1)
    y5, _, _ = oracle.matmul(blk, a5)
    assert y1[0, 0] == float(kv["y_ones"])
    assert y5[0, 0] == float(kv["y_mod5"])


def test_round_half_away_from_zero_pinned():
    # element 2 is x/d = -0.5 exactly: half-away gives -1 -> q=7; half-even would give 0 -> q=8
    _, x, q = _worked()
    assert q[2] == 7 and q[3] == 9
    assert _q_of(oracle.quantize(x.reshape(1, 32)))[0, 2] == 7


def test_first_of_equal_absmax_sets_the_sign():
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = -2.0
    x[0, 7] = 2.0  # equal |x|, later index
    blk = oracle.quantize(x)
    d = float(_d_of(blk)[0, 0])
    assert d == 0.25  # m = -2 (first), d = -2/-8
    assert _q_of(blk)[0, 3] == 0 and _q_of(blk)[0, 7] == 15  # the opposite sign clamps


# ---------------------------------------------------------------- binary16

def test_f16_conversion_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.01),
        rng.standard_normal(20000).astype(np.float32) * np.float32(1000.0),
        (rng.standard_normal(20000) * 1e-5).astype(np.float32),   # binary16 subnormal range
        (rng.standard_normal(5000) * 1e-8).astype(np.float32),    # underflow to zero
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0**-14, 2.0**-24,
                  2.0**-25, 3 * 2.0**-26, 2.0**-25 * 1.0000001, np.inf, -np.inf, 1.0 + 2.0**-11,
                  1.0 + 3 * 2.0**-11, 2049.0, 2051.0, 6.103515625e-05], dtype=np.float32),
    ])
    # halfway cases between adjacent binary16 values (round to nearest even)
    h = np.arange(0, 0x7C00, 97, dtype=np.uint16).view(np.float16).astype(np.float32)
    h2 = (np.arange(1, 0x7C00, 97, dtype=np.uint16)).view(np.float16).astype(np.float32)
    mids = ((h[: len(h2)].astype(np.float64) + h2.astype(np.float64)) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_f16_widening_matches_numpy():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_bits_to_f32(int(b)) for b in bits[::7]], dtype=np.float32)
    r = ref[::7]
    finite = np.isfinite(r)
    assert np.array_equal(got[finite], r[finite])
    assert np.all(np.isnan(got[np.isnan(r)]))


# ---------------------------------------------------------------- quantizer

def test_quantizer_is_nearest_level_brute_force():
    """q is the level (q-8)*d nearest to x among q in 0..15 (ties excepted)."""
    w = synthetic.normal(synthetic.weight_seed(99, 0), (64, 256), sigma=0.02)
    blocks = oracle.quantize(w)
    q = _q_of(blocks)
    for n in range(w.shape[0]):
        for b in range(w.shape[1] // 32):
            xb = w[n, 32 * b: 32 * b + 32].astype(np.float64)
            m = xb[np.argmax(np.abs(xb))]  # numpy argmax: first of equal values
            d = np.float32(np.float32(m) / np.float32(-8.0))
            levels = (np.arange(16) - 8) * np.float64(d)
            dist = np.abs(xb[:, None] - levels[None, :])
            best = np.argmin(dist, axis=1)
            srt = np.sort(dist, axis=1)
            clear = srt[:, 1] - srt[:, 0] > 1e-12 * abs(float(d))
            assert np.array_equal(q[n, 32 * b: 32 * b + 32][clear], best[clear])


def test_round_trip_bound():
    """|x - deq(q(x))| <= |d32|/2 + 8|d32-d16| unclamped, <= |d32| + 8|d32-d16| clamped."""
    w = synthetic.normal(synthetic.weight_seed(98, 0), (256, 512), sigma=0.02)
    blocks = oracle.quantize(w)
    deq = oracle.dequantize(blocks).astype(np.float64)
    xb = w.reshape(256, -1, 32).astype(np.float64)
    idx = np.argmax(np.abs(xb), axis=2)
    m = np.take_along_axis(xb, idx[..., None], axis=2)[..., 0].astype(np.float32)
    d32 = (m / np.float32(-8.0)).astype(np.float64)[..., None]
    d16 = _d_of(blocks).astype(np.float64)[..., None]
    err = np.abs(xb - deq.reshape(xb.shape))
    clamped = (xb / d32) >= 7.5
    slack = 8 * np.abs(d32 - d16)
    assert np.all(err[~clamped] <= np.abs(d32 / 2 + 0 * xb)[~clamped] + slack.repeat(32, 2)[~clamped] + 1e-12)
    assert np.all(err[clamped] <= np.abs(d32 + 0 * xb)[clamped] + slack.repeat(32, 2)[clamped] + 1e-12)
    assert clamped.any()  # the clamped tail exists with N(0, 0.02) weights


def test_all_zero_block_and_status_codes():
    z = np.zeros((2, 64), np.float32)
    blk = oracle.quantize(z)
    assert np.all(_q_of(blk) == 8) and np.all(_d_of(blk) == 0)
    bad = np.zeros((1, 32), np.float32)
    bad[0, 5] = np.nan
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize(bad)
    assert e.value.status == oracle.ERR_NONFINITE
    big = np.full((1, 32), 1e6, np.float32)  # d = -125000 overflows binary16
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize(big)
    assert e.value.status == oracle.ERR_RANGE
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize(np.zeros((1, 48), np.float32))
    assert e.value.status == oracle.ERR_SHAPE


# ---------------------------------------------------------------- matmul

def _dyadic(seed, shape, scale=16):
    rng = np.random.default_rng(seed)
    return (rng.integers(-64, 65, size=shape) / scale).astype(np.float32)


@pytest.mark.parametrize("N,K,M", [(1, 32, 1), (3, 64, 2), (4, 32, 3), (2, 96, 3)])
def test_matmul_equals_exact_rational_dequant_then_dot(N, K, M):
    w = synthetic.normal(synthetic.weight_seed(97, N * K + M), (N, K), sigma=0.02)
    x = _dyadic(N + K + M, (M, K))
    blocks = oracle.quantize(w)
    q = _q_of(blocks)
    d = _d_of(blocks)
    y, y64, bound = oracle.matmul(blocks, x)
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            a = Fraction(0)
            for k in range(K):
                wk = (int(q[n, k]) - 8) * Fraction(float(d[n, k // 32]))
                p = wk * Fraction(float(x[m, k]))
                s += p
                a += abs(p)
            assert Fraction(float(y64[m, n])) == s        # exact: all sums are dyadic
            assert float(y[m, n]) == float(np.float32(float(s)))
            assert abs(bound[m, n] - (1e-5 * float(a) + 1e-6)) <= 1e-15 * (1 + float(a))


def test_linearity_in_x():
    w = synthetic.normal(synthetic.weight_seed(96, 0), (8, 128), sigma=0.02)
    blocks = oracle.quantize(w)
    x1 = _dyadic(1, (3, 128))
    x2 = _dyadic(2, (3, 128))
    a, b = np.float32(0.5), np.float32(-2.0)
    _, y1, _ = oracle.matmul(blocks, x1)
    _, y2, _ = oracle.matmul(blocks, x2)
    _, y12, _ = oracle.matmul(blocks, a * x1 + b * x2)
    assert np.array_equal(y12, 0.5 * y1 - 2.0 * y2)


def test_closed_form_constant_levels():
    """All q = c and x = 1 give y_n = 32 (c - 8) sum_b d16[n, b]."""
    rng = np.random.default_rng(5)
    N, nb = 5, 7
    for c in (0, 3, 8, 15):
        blocks = np.zeros((N, nb, 18), np.uint8)
        dvals = (rng.standard_normal((N, nb)) * 0.01).astype(np.float16)
        blocks[..., 0:2] = dvals.view(np.uint8).reshape(N, nb, 2)
        blocks[..., 2:] = c | (c << 4)
        x = np.ones((2, nb * 32), np.float32)
        _, y64, _ = oracle.matmul(blocks, x)
        expect = 32.0 * (c - 8) * dvals.astype(np.float64).sum(axis=1)
        assert np.allclose(y64[0], expect, rtol=0, atol=1e-15) and np.array_equal(y64[0], y64[1])


def test_matches_numpy_fp64_matmul_of_dequantized():
    w = synthetic.normal(synthetic.weight_seed(95, 0), (96, 896), sigma=0.02)
    x = synthetic.normal(synthetic.act_seed(95, 4), (4, 896))
    blocks = oracle.quantize(w)
    wd = oracle.dequantize(blocks).astype(np.float64)
    ref = x.astype(np.float64) @ wd.T
    y, y64, bound = oracle.matmul(blocks, x)
    assert np.allclose(y64, ref, rtol=1e-13, atol=1e-15)
    assert np.array_equal(y, y64.astype(np.float32))
    assert np.allclose(bound, 1e-5 * (np.abs(x.astype(np.float64)) @ np.abs(wd).T) + 1e-6, rtol=1e-12)


def test_matmul_pairs_agrees_with_full():
    w = synthetic.normal(synthetic.weight_seed(94, 0), (40, 256), sigma=0.02)
    x = synthetic.normal(synthetic.act_seed(94, 3), (3, 256))
    blocks = oracle.quantize(w)
    y, y64, bound = oracle.matmul(blocks, x)
    pairs = np.array([[0, 0], [2, 39], [1, 17], [2, 5]], np.int64)
    py, py64, pb = oracle.matmul_pairs(blocks, x, pairs)
    assert np.array_equal(py, y[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(py64, y64[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(pb, bound[pairs[:, 0], pairs[:, 1]])


# ---------------------------------------------------------------- argmax

def test_greedy_pick_from_printed_scores():
    _, rows = read_golden("greedy_top2_logits.txt")
    assert len(rows) == 2
    for mode, s476, s323, sel in rows:
        logits = np.full((1, 600), -1.0, np.float32)
        logits[0, 476] = np.float32(s476)
        logits[0, 323] = np.float32(s323)
        assert int(oracle.argmax(logits)[0]) == int(sel), mode


def test_argmax_ties_nan_and_numpy():
    rng = np.random.default_rng(7)
    y = rng.standard_normal((6, 1000)).astype(np.float32)
    assert np.array_equal(oracle.argmax(y), np.argmax(y, axis=1))
    t = np.zeros((1, 10), np.float32)
    t[0, [3, 6]] = 5.0
    assert oracle.argmax(t)[0] == 3
    n = np.array([[np.nan, 1.0, 2.0, np.nan, 2.0]], np.float32)
    assert oracle.argmax(n)[0] == 2

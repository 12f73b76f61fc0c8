"""GPU parity: the CUDA library against the CPU oracle, element by element,
at sizes that span several 128-row tiles, several K splits and a ragged tail.

Every call goes through the C ABI (libq4mm.so) via the thin binding."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, assert_within_bound, plant_near_ties, weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_matmul_gb300 as q4

    torch.cuda.set_device(0)
    return q4


def _flags(q4):
    return {"auto": 0, "simt": q4.Q4MM_FORCE_SIMT, "mma": q4.Q4MM_FORCE_MMA,
            "tc": q4.Q4MM_FORCE_TC, "invariant": q4.Q4MM_BATCH_INVARIANT,
            "invariant_tc": q4.Q4MM_BATCH_INVARIANT | q4.Q4MM_FORCE_TC,
            "row_by_row": q4.Q4MM_ROW_BY_ROW}


# ------------------------------------------------------------------ quantizer

@pytest.mark.parametrize("N,K", [(1, 32), (17, 64), (129, 96), (300, 1024), (896, 896), (512, 3584)])
def test_quantize_byte_identical_to_oracle(q4, N, K):
    w = weights(50, N % 16, N, K)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    assert np.array_equal(q4.q4_export_blocks(W), oracle.quantize(w))
    W.free()


def test_quantize_edge_blocks(q4):
    from conftest import read_golden

    kv, _ = read_golden("q4_worked_block.txt")
    rows = [np.array([float(v) for v in kv["x"].split()], np.float32)]
    rows.append(np.zeros(32, np.float32))                          # all-zero block
    r = np.zeros(32, np.float32); r[3], r[7] = -2.0, 2.0; rows.append(r)   # equal +-absmax
    rows.append((np.arange(32) - 16).astype(np.float32) * np.float32(1e-41))  # fp32 subnormals
    rows.append(np.full(32, 3.0, np.float32))                      # constant block
    rows.append((np.arange(32, dtype=np.float32) - 15.5) * np.float32(1 / 8))  # exact halves
    w = np.stack(rows)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    got = q4.q4_export_blocks(W)
    assert np.array_equal(got, oracle.quantize(w))
    assert got[0, 0].tobytes().hex() == kv["bytes"]


def test_import_export_round_trip(q4):
    rng = np.random.default_rng(3)
    N, K = 257, 128
    blocks = rng.integers(0, 256, size=(N, K // 32, 18), dtype=np.uint8)
    d = (rng.standard_normal((N, K // 32)) * 0.01).astype(np.float16)
    blocks[..., 0:2] = d.view(np.uint8).reshape(N, K // 32, 2)
    W = q4.q4_import_blocks(blocks, N, K)
    assert np.array_equal(q4.q4_export_blocks(W), blocks)
    x = acts(60, 3, K)
    y = q4.q4mm_forward(W, torch.from_numpy(x).to(DEV)).cpu().numpy()
    _, y64, bound = oracle.matmul(blocks, x)
    assert_within_bound(y, y64, bound, "imported")


def test_status_codes(q4):
    bad = np.zeros((2, 64), np.float32)
    bad[1, 40] = np.nan
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_quantize(torch.from_numpy(bad).to(DEV))
    assert e.value.status == q4.Q4_ERR_NONFINITE
    big = np.full((1, 32), 1e6, np.float32)
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_quantize(torch.from_numpy(big).to(DEV))
    assert e.value.status == q4.Q4_ERR_RANGE
    blocks = np.zeros((1, 1, 18), np.uint8)
    blocks[0, 0, 0:2] = [0x00, 0x7C]  # +inf scale
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_import_blocks(blocks, 1, 32)
    assert e.value.status == q4.Q4_ERR_NONFINITE

    w = weights(61, 0, 40, 64)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    lib = q4.raw_library()
    buf = torch.zeros(4 * 64 + 4, device=DEV)
    y = torch.zeros(4 * 40 + 4, device=DEV)
    # x misaligned by 4 bytes
    assert lib.q4mm_forward(W.handle, buf.data_ptr() + 4, y.data_ptr(), 4, None) == q4.Q4_ERR_ALIGN
    assert lib.q4mm_forward(W.handle, buf.data_ptr(), y.data_ptr(), q4.Q4MM_M_MAX + 1, None) == q4.Q4_ERR_SHAPE
    assert lib.q4mm_forward(W.handle, buf.data_ptr(), y.data_ptr(), -1, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_ex(W.handle, buf.data_ptr(), y.data_ptr(), 2, 0x100, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_ex(W.handle, buf.data_ptr(), y.data_ptr(), 2,
                               q4.Q4MM_FORCE_SIMT | q4.Q4MM_FORCE_TC, None) == q4.Q4_ERR_INVALID_ARG
    assert lib.q4mm_forward_ex(W.handle, buf.data_ptr(), y.data_ptr(), 2,
                               q4.Q4MM_FORCE_MMA | q4.Q4MM_ROW_BY_ROW, None) == q4.Q4_ERR_INVALID_ARG
    y.fill_(7.0)
    assert lib.q4mm_forward(W.handle, buf.data_ptr(), y.data_ptr(), 0, None) == q4.Q4_OK  # no-op
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


# ------------------------------------------------------------------ forward

CASES = [
    (300, 1024, (1, 2, 3, 5, 8, 9, 17, 64, 70)),   # 3 tiles + ragged tail, several K splits
    (896, 896, (1, 2, 4)),                          # the 896 x 896 config
    (130, 3584, (1, 4, 33)),                        # 2 tiles, one of 2 rows
    (33, 18944, (1, 3)),                            # the long-K down_proj K, one ragged tile
    (200, 224, (1, 3, 9, 16, 30)),                  # 7 blocks: the last pair half padding
    (257, 1440, (2, 8, 12, 24)),                    # 45 blocks, 3 tiles, one of 1 row
]


@pytest.mark.parametrize("N,K,Ms", CASES)
@pytest.mark.parametrize("mode", ["auto", "simt", "mma", "tc", "invariant", "row_by_row"])
def test_forward_matches_oracle(q4, N, K, Ms, mode):
    w = weights(51, N % 16, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    flags = _flags(q4)[mode]
    for M in Ms:
        if mode == "row_by_row" and M > 9:
            continue
        x = acts(51, M, K, salt=N)
        y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), flags).cpu().numpy()
        _, y64, bound = oracle.matmul(blocks, x)
        assert_within_bound(y, y64, bound, "%s N=%d K=%d M=%d" % (mode, N, K, M))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_forward_default_entry_and_preallocated_output(q4):
    N, K, M = 200, 512, 6
    w = weights(52, 0, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    x = acts(52, M, K)
    y = torch.full((M, N), float("nan"), device=DEV)
    q4.q4mm_forward(W, torch.from_numpy(x).to(DEV), y=y)
    _, y64, bound = oracle.matmul(blocks, x)
    assert_within_bound(y.cpu().numpy(), y64, bound, "q4mm_forward")
    W.free()


def test_special_inputs(q4):
    """Zero activations, zero weights, a single nonzero column and huge/tiny x."""
    N, K = 150, 256
    w = weights(53, 0, N, K)
    w[5] = 0.0
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    xs = [np.zeros((2, K), np.float32)]
    one = np.zeros((1, K), np.float32); one[0, 77] = 1.0; xs.append(one)
    xs.append(acts(53, 3, K) * np.float32(1e30))
    xs.append(acts(53, 3, K) * np.float32(1e-30))
    for x in xs:
        for mode in ("auto", "simt", "mma", "tc", "invariant"):
            y = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), _flags(q4)[mode]).cpu().numpy()
            _, y64, bound = oracle.matmul(blocks, x)
            assert_within_bound(y, y64, bound, mode)
    W.free()


# ------------------------------------------------------------------ batch invariance

# streaming: Q4MM_BATCH_INVARIANT alone; tensor_core: with Q4MM_FORCE_TC (one
# instruction shape and K partition for every M, 64 token rows per tile, so
# the 124 rows run as two tiles and a single row as one)
@pytest.mark.parametrize("mode", ["streaming", "tensor_core"])
@pytest.mark.parametrize("N,K", [(300, 1024), (260, 3584)])
def test_batch_invariant_rows_bit_identical(q4, N, K, mode):
    w = weights(54, 0, N, K)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    inv = q4.Q4MM_BATCH_INVARIANT | (q4.Q4MM_FORCE_TC if mode == "tensor_core" else 0)
    big = acts(54, 124, K)
    xb = torch.from_numpy(big).to(DEV)
    y124 = q4.q4mm_forward_ex(W, xb, inv).cpu().numpy()
    y4 = q4.q4mm_forward_ex(W, xb[120:124].contiguous(), inv).cpu().numpy()
    assert np.array_equal(y124[120:124].view(np.uint32), y4.view(np.uint32))
    rng = np.random.default_rng(5)
    for r in rng.choice(124, size=16, replace=False):
        y1 = q4.q4mm_forward_ex(W, xb[r:r + 1].contiguous(), inv).cpu().numpy()
        assert np.array_equal(y124[r].view(np.uint32), y1[0].view(np.uint32)), r
    other = acts(54, 124, K, salt=9)
    other[17] = big[17]
    y_other = q4.q4mm_forward_ex(W, torch.from_numpy(other).to(DEV), inv).cpu().numpy()
    assert np.array_equal(y_other[17].view(np.uint32), y124[17].view(np.uint32))
    # every row is also within the oracle's bound
    _, y64, bound = oracle.matmul(oracle.quantize(w), big)
    assert_within_bound(y124, y64, bound, "%s invariant M=124" % mode)
    W.free()


# ------------------------------------------------------------------ argmax

@pytest.mark.parametrize("mode", ["auto", "simt", "mma", "tc", "invariant", "invariant_tc"])
def test_argmax_matches_oracle(q4, mode):
    N, K = 1000, 512
    w = weights(55, 0, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    rng = np.random.default_rng(11)
    for M in (1, 4, 16, 70):
        x = acts(55, M, K)
        x, planted = plant_near_ties(blocks, x, list(range(0, M, 2)), rng)
        idx, mx = q4.q4mm_argmax_ex(W, torch.from_numpy(x).to(DEV), _flags(q4)[mode])
        idx, mx = idx.cpu().numpy(), mx.cpu().numpy()
        y, y64, bound = oracle.matmul(blocks, x)
        ref = oracle.argmax(y)
        for m in range(M):
            top = np.argsort(-y64[m], kind="stable")
            margin = y64[m, top[0]] - y64[m, top[1]]
            # exact wherever the oracle's top-2 margin exceeds the bound at the top index
            if margin > bound[m, top[0]]:
                assert idx[m] == ref[m], (mode, M, m, planted.get(m))
            else:
                assert y64[m, ref[m]] - y64[m, idx[m]] <= bound[m, ref[m]] + bound[m, idx[m]]
            assert abs(float(mx[m]) - y64[m, idx[m]]) <= bound[m, idx[m]]
        # argmax agrees with the library's own forward output
        yf = q4.q4mm_forward_ex(W, torch.from_numpy(x).to(DEV), _flags(q4)[mode]).cpu().numpy()
        assert np.array_equal(np.argmax(yf, axis=1), idx)
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_argmax_exact_ties_pick_lowest_index(q4):
    # two identical weight rows give identical logits: the lower index must win
    N, K = 400, 256
    w = weights(56, 0, N, K)
    w[310] = w[57] * 3.0
    w[371] = w[310]
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    wd = oracle.dequantize(blocks[[310]]).astype(np.float64)[0]
    x = (wd / np.linalg.norm(wd) * 40).astype(np.float32)[None, :]
    idx, mx = q4.q4mm_argmax(W, torch.from_numpy(x).to(DEV))
    assert int(idx.item()) == 310
    W.free()


def test_forward_at_the_largest_m(q4):
    # M = Q4MM_M_MAX in one call (tensor-core path, several token tiles), every
    # output of a seeded sample of rows against the oracle; the streaming path
    # (16 rows per launch) on the same rows
    N, K = 300, 1024
    w = weights(52, 3, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).to(DEV))
    M = q4.Q4MM_M_MAX
    x = acts(52, M, K)
    xd = torch.from_numpy(x).to(DEV)
    rows = np.sort(np.random.default_rng(52).choice(M, 96, replace=False))
    rows[-1] = M - 1
    _, y64, bound = oracle.matmul(blocks, x[rows])
    for flags in (0, q4.Q4MM_FORCE_MMA):
        y = q4.q4mm_forward_ex(W, xd, flags).cpu().numpy()
        assert_within_bound(y[rows], y64, bound, "M=%d flags=%d" % (M, flags))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()

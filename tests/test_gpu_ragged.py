"""GPU checks of the ragged continuous-batching helpers: the greedy pick for a
subset of a step's rows (q4mm_argmax_rows) and greedy verification of draft
tokens per request (q4_verify_greedy)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import acts, weights

pytestmark = pytest.mark.gpu

q4 = pytest.importorskip("bit_quantized_matmul_gb300")


def _oracle_argmax(blocks, x):
    _, y64, bound = oracle.matmul(blocks, x)
    return np.asarray(oracle.argmax(y64)), y64, bound


def test_argmax_rows_matches_oracle_and_gathered_call():
    N, K = 3000, 896
    w = weights(120, 0, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).cuda())
    x_np = acts(120, 40, K)
    x = torch.from_numpy(x_np).cuda()
    for sel in ([39], [3, 7, 7, 0], list(range(39, 0, -3)), [5] * 11):
        rows = torch.tensor(sel, dtype=torch.int32, device="cuda")
        idx, mx = q4.q4mm_argmax_rows(W, x, rows)
        ref_idx, y64, bound = _oracle_argmax(blocks, x_np[sel])
        got = idx.cpu().numpy()
        for r in range(len(sel)):
            top = np.sort(y64[r])[::-1]
            if top[0] - top[1] > bound[r].max():
                assert got[r] == ref_idx[r], (sel, r)
            else:  # near-tie: any index within the bound of the top is correct
                assert y64[r, got[r]] >= top[0] - bound[r, got[r]]
        gi, gm = q4.q4mm_argmax(W, x[sel].contiguous())
        assert torch.equal(gi, idx) and torch.equal(gm.view(torch.int32), mx.view(torch.int32))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_argmax_rows_on_two_tile_ctas():
    # a head of more tiles than SMs with one K split (155 tiles, K = 1024)
    # runs the row-list pick on CTAs that stream two tiles each
    N, K = 155 * 128 - 37, 1024
    w = weights(123, 0, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).cuda())
    _, _, splits = q4.q4mm_plan_info(W, 1, q4.Q4MM_FORCE_MMA)
    assert splits == 1
    x_np = acts(123, 30, K)
    x = torch.from_numpy(x_np).cuda()
    for sel in ([29], [3, 7, 7, 0, 12], list(range(29, 0, -3))):
        rows = torch.tensor(sel, dtype=torch.int32, device="cuda")
        idx, mx = q4.q4mm_argmax_rows(W, x, rows)
        ref_idx, y64, bound = _oracle_argmax(blocks, x_np[sel])
        got, gmx = idx.cpu().numpy(), mx.cpu().numpy()
        for r in range(len(sel)):
            top = np.sort(y64[r])[::-1]
            if top[0] - top[1] > bound[r].max():
                assert got[r] == ref_idx[r], (sel, r)
            else:
                assert y64[r, got[r]] >= top[0] - bound[r, got[r]]
            assert abs(float(gmx[r]) - y64[r, got[r]]) <= bound[r, got[r]]
        gi, gm = q4.q4mm_argmax(W, x[sel].contiguous())
        assert torch.equal(gi, idx) and torch.equal(gm.view(torch.int32), mx.view(torch.int32))
    assert q4.q4_device_status() == q4.Q4_OK
    W.free()


def test_argmax_rows_out_of_range_index_is_reported_not_read():
    N, K = 300, 256
    W = q4.q4_quantize(torch.from_numpy(weights(121, 0, N, K)).cuda())
    x = torch.from_numpy(acts(121, 4, K)).cuda()
    for bad in (4, -1, 1 << 30):
        rows = torch.tensor([0, bad, 2], dtype=torch.int32, device="cuda")
        q4.q4mm_argmax_rows(W, x, rows)
        assert q4.q4_device_status() == q4.Q4_ERR_INVALID_ARG
    assert q4.q4_device_status() == q4.Q4_OK  # cleared
    W.free()


def _verify_ref(idx, draft, offsets, total):
    out = []
    for s in range(len(offsets) - 1):
        b, e = offsets[s], offsets[s + 1]
        if b < 0 or e < b or e > total:
            out.append(-1)
            continue
        n = 0
        while b + n < e and idx[b + n] == draft[b + n]:
            n += 1
        out.append(n)
    return out


def test_verify_greedy_against_reference():
    rng = np.random.default_rng(7)
    for S in (1, 5, 300):
        lens = rng.integers(0, 9, size=S)
        offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        total = int(offsets[-1])
        idx = rng.integers(0, 4, size=total).astype(np.int32)
        draft = np.where(rng.random(total) < 0.8, idx, (idx + 1) % 4).astype(np.int32)
        if S > 1:  # a malformed segment and one running past the end
            offsets[1] = offsets[2] + 1 if S > 2 else offsets[1]
        if S > 4:
            offsets[-2] = total + 5
        args = [torch.from_numpy(a).cuda() for a in (idx, draft, offsets)]
        got = q4.q4_verify_greedy(*args).cpu().numpy().tolist()
        assert got == _verify_ref(idx, draft, offsets.tolist(), total), S


def test_ragged_step_end_to_end():
    """A packed step: request A prefill (6 rows, only the last needs logits),
    request B verifying 3 drafts (3 rows), request C decoding (1 row)."""
    N, K = 2000, 512
    w = weights(122, 0, N, K)
    blocks = oracle.quantize(w)
    W = q4.q4_quantize(torch.from_numpy(w).cuda())
    x_np = acts(122, 10, K)
    need = [5, 6, 7, 8, 9]  # last prefill row of A, B's verify rows, C's decode row
    ref_idx, _, _ = _oracle_argmax(blocks, x_np[need])
    idx, _ = q4.q4mm_argmax_rows(W, torch.from_numpy(x_np).cuda(),
                                 torch.tensor(need, dtype=torch.int32, device="cuda"))
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    # B's drafts: first two agree with the greedy pick, third does not
    draft = idx.clone()
    draft[3] = (draft[3] + 1) % N
    offsets = torch.tensor([0, 1, 4, 5], dtype=torch.int32, device="cuda")  # A, B, C
    acc = q4.q4_verify_greedy(idx, draft, offsets).cpu().numpy().tolist()
    assert acc == [1, 2, 1]
    W.free()

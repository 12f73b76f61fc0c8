"""Pins of the KV-cache append oracle (CPU).

The preallocated append (``oracle.kv.kv_append``) is checked against the
growing cache that concatenates every step's rows (``kv_concat``), the other
cache kind of "A non-contiguous KV cache cuts Qwen2 decode speed by 59 % at 2k
context in Candle on Metal" whose values must agree with it (§"Reproduce"),
and against what must stay untouched."""
import numpy as np

from oracle import kv
import synthetic


def _steps(seed, layers, heads, D, slots, plan):
    """plan: list of steps, each a list of (slot, n_rows); yields (k_new, v_new, offsets, slot)."""
    out = []
    for i, step in enumerate(plan):
        total = sum(n for _, n in step)
        k = synthetic.normal(seed + 2 * i, (layers, total, heads, D))
        v = synthetic.normal(seed + 2 * i + 1, (layers, heads, total, D)).transpose(0, 2, 1, 3)  # strided view
        offsets = np.concatenate([[0], np.cumsum([n for _, n in step])]).astype(np.int32)
        out.append((k, v, offsets, np.array([s for s, _ in step], dtype=np.int32)))
    return out


def test_prealloc_append_equals_concatenated_cache():
    layers, heads, D, slots, cap = 3, 2, 8, 4, 40
    plan = [[(0, 7), (2, 1), (3, 0)], [(0, 1), (2, 1), (1, 5)], [(2, 4), (0, 1), (1, 1), (3, 2)]]
    sentinel = np.float32(-7.25)
    kc = np.full((layers, slots, heads, cap, D), sentinel, np.float32)
    vc = kc.copy()
    lengths = np.zeros(slots, np.int32)
    grown = {}
    for k_new, v_new, offsets, slot in _steps(0xC0FFEE, layers, heads, D, slots, plan):
        pos = lengths[slot].astype(np.int32)
        kc, vc, rejected = kv.kv_append(kc, vc, k_new, v_new, offsets, slot, pos)
        assert rejected == []
        grown = kv.kv_concat(grown, k_new, v_new, offsets, slot)
        lengths[slot] += np.diff(offsets).astype(np.int32)
    for sl in range(slots):
        n = lengths[sl]
        if sl in grown:
            assert np.array_equal(kc[:, sl, :, :n], grown[sl][0])
            assert np.array_equal(vc[:, sl, :, :n], grown[sl][1])
        assert np.all(kc[:, sl, :, n:] == sentinel) and np.all(vc[:, sl, :, n:] == sentinel)


def test_rows_go_to_the_slot_and_position_given():
    # hand-made: one layer, one head, head_dim 2; request 0 (slot 1) appends two rows at position 3
    kc = np.zeros((1, 2, 1, 6, 2), np.float32)
    k_new = np.array([[[[1, 2]], [[3, 4]]]], np.float32)  # [1, 2, 1, 2]
    out, _, rej = kv.kv_append(kc, kc, k_new, k_new, np.array([0, 2], np.int32), np.array([1], np.int32),
                               np.array([3], np.int32))
    assert rej == []
    assert out[0, 1, 0, 3].tolist() == [1, 2] and out[0, 1, 0, 4].tolist() == [3, 4]
    assert np.count_nonzero(out) == 4


def test_out_of_range_requests_are_rejected_whole():
    layers, heads, D, slots, cap = 2, 1, 4, 3, 8
    kc = np.zeros((layers, slots, heads, cap, D), np.float32)
    k_new = synthetic.normal(5, (layers, 9, heads, D))
    offsets = np.array([0, 3, 6, 8, 9], np.int32)
    slot = np.array([0, 1, 5, 2], np.int32)      # request 2: no such slot
    pos = np.array([6, 0, 0, -1], np.int32)      # request 0 overflows capacity, request 3 negative
    out, _, rej = kv.kv_append(kc, kc, k_new, k_new, offsets, slot, pos)
    assert rej == [0, 2, 3]
    assert np.array_equal(out[:, 1, :, 0:3], np.transpose(k_new[:, 3:6], (0, 2, 1, 3)))
    assert np.count_nonzero(out[:, 0]) == 0 and np.count_nonzero(out[:, 2]) == 0

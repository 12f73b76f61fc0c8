"""CPU oracle for the KV-cache append of one continuous-batching step — test
infrastructure only (only the test suite and bench.py's CPU-baseline leg may
import it; the CUDA library never reaches it and shares no code with it).

"A non-contiguous KV cache cuts Qwen2 decode speed by 59 % at 2k context in
Candle on Metal" measures three caches that must hold the same values
(§"Reproduce": its unit test asserts that every cache kind returns the same
tensors): one that grows by concatenation on every step, the same with a
contiguous copy first, and a preallocated buffer that each step writes its
new rows into (`slice_set`, §"What was measured and how").  ``kv_append`` is
the preallocated kind written out plainly: for each request, each new packed
row is copied to the next free position of the request's slot, in every layer
and head.  ``kv_concat`` is the growing kind, used to pin it.

Arrays are numpy; element type is whatever the caller passes (the append is a
copy, so results are exact).
"""
from __future__ import annotations

import numpy as np


def kv_append(k_cache, v_cache, k_new, v_new, offsets, slot, pos):
    """Preallocated-cache append.

    k_cache, v_cache: [layers, slots, heads, capacity, head_dim]
    k_new, v_new:     [layers, total, heads, head_dim] (any strides)
    offsets: [S + 1]; slot, pos: [S]
    Returns (k_out, v_out, rejected): copies of the caches with the new rows
    written, and the requests left unwritten because their slot, position or
    row range was out of range.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    layers, slots, heads, capacity, _ = k_out.shape
    total = k_new.shape[1]
    rejected = []
    for s in range(len(slot)):
        b, e = int(offsets[s]), int(offsets[s + 1])
        sl, p0 = int(slot[s]), int(pos[s])
        n = e - b
        if n <= 0:
            continue
        if sl < 0 or sl >= slots or p0 < 0 or b < 0 or e > total or p0 + n > capacity:
            rejected.append(s)
            continue
        for j in range(n):
            for layer in range(layers):
                for h in range(heads):
                    k_out[layer, sl, h, p0 + j, :] = k_new[layer, b + j, h, :]
                    v_out[layer, sl, h, p0 + j, :] = v_new[layer, b + j, h, :]
    return k_out, v_out, rejected


def kv_concat(cache_rows, k_new, v_new, offsets, slot):
    """Growing-cache append: per (slot) a list of appended [layers, heads,
    head_dim] rows for K and V, extended by concatenation; returns the new
    dict {slot: (K [layers, heads, len, head_dim], V ...)}."""
    out = {}
    for sl, (k, v) in cache_rows.items():
        out[sl] = (k, v)
    for s in range(len(slot)):
        b, e = int(offsets[s]), int(offsets[s + 1])
        if e <= b:
            continue
        sl = int(slot[s])
        kn = np.transpose(np.asarray(k_new[:, b:e]), (0, 2, 1, 3))  # [layers, heads, n, head_dim]
        vn = np.transpose(np.asarray(v_new[:, b:e]), (0, 2, 1, 3))
        if sl in out:
            k, v = out[sl]
            out[sl] = (np.concatenate([k, kn], axis=2), np.concatenate([v, vn], axis=2))
        else:
            out[sl] = (kn.copy(), vn.copy())
    return out

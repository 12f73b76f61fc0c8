"""Shared helpers for the GPU parity tests: seeded inputs, the oracle side,
and element-wise comparison against the oracle's tolerance."""
import numpy as np

import oracle
import synthetic


def weights(config, matrix, N, K, sigma=0.02):
    return synthetic.normal(synthetic.weight_seed(config, matrix), (N, K), sigma=sigma)


def acts(config, M, K, salt=0):
    return synthetic.normal(synthetic.act_seed(config, M) + (salt << 20), (M, K))


def assert_within_bound(y_gpu, y_ref64, bound, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_ref64)
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(err <= bound), "%s: max err/bound %.3g at %s (gpu %r ref %r)" % (
        what, float(ratio[worst]), worst, float(y_gpu[worst]), float(y_ref64[worst]))
    return float(ratio.max())


def plant_near_ties(blocks, x, rows, rng, gap=1e-3, lead=2.0):
    """Return x with rows[i] replaced so that two logits a, b are the top two,
    ell_a - ell_b = gap and both clear the rest by about `lead`.

    x' = x + c1 w_a + c2 w_b with (c1, c2) from the 2x2 Gram system of the
    dequantized rows; the result is re-checked with the oracle."""
    x = x.copy()
    N = blocks.shape[0]
    out = {}
    for r in rows:
        for _attempt in range(20):
            a, b = rng.choice(N, size=2, replace=False)
            wab = oracle.dequantize(blocks[[a, b]]).astype(np.float64)
            _, l0, _ = oracle.matmul(blocks, x[r:r + 1])
            l0 = l0[0]
            rest = np.delete(l0, [a, b]).max()
            target = np.array([rest + lead, rest + lead - gap])
            G = wab @ wab.T
            c = np.linalg.solve(G, target - l0[[a, b]])
            xr = (x[r].astype(np.float64) + c @ wab).astype(np.float32)
            _, l1, bnd = oracle.matmul(blocks, xr[None, :])
            l1 = l1[0]
            order = np.argsort(-l1, kind="stable")
            if {order[0], order[1]} == {a, b} and l1[order[1]] - l1[order[2]] > 0.1 and \
                    abs((l1[a] - l1[b]) - gap) < 0.05 * gap:
                x[r] = xr
                out[r] = (int(a), int(b))
                break
        else:
            raise RuntimeError("could not plant a near-tie in row %d" % r)
    return x, out

"""Pins for the multi-query decode oracle (CPU only).

``oracle.attention.sparse_attn_decode_mq`` builds one key set with a
visibility mask; each pin reaches the same numbers another way: the
single-query decode with each query's own window length, a brute-force
softmax in plain Python loops, and the causality invariants of the reading
(a query ignores later window rows and other queries' inputs).
"""
import math

import numpy as np

from oracle import attention as oatt


def _problem(seed, ql, H=4, n=300, K=40, W=12, swa_len=10):
    rng = np.random.default_rng(seed)
    latent = rng.standard_normal((n, 512))
    rope = rng.standard_normal((n, 64))
    topk = np.sort(rng.choice(n, size=K, replace=False)).astype(np.int64)
    topk[-3:] = -1
    swa = rng.standard_normal((W, 576))
    q = rng.standard_normal((ql, H, 576)) * 0.05
    return q, latent, rope, topk, swa, swa_len


def test_each_query_is_a_single_decode_with_its_own_window():
    for ql in (1, 2, 3, 4):
        q, lat, rope, topk, swa, swl = _problem(1 + ql, ql)
        o, l = oatt.sparse_attn_decode_mq(q, lat, rope, topk, swa, swl, 0.07)
        for i in range(ql):
            oi, li = oatt.sparse_attn_decode(q[i], lat, rope, topk, swa, swl - (ql - 1 - i), 0.07)
            np.testing.assert_allclose(o[i], oi, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(l[i], li, rtol=1e-12, atol=1e-12)


def test_brute_force_loops():
    """Tiny case, every logit / weight / output channel in Python loops."""
    q, lat, rope, topk, swa, swl = _problem(7, 3, H=2, n=20, K=5, W=4, swa_len=4)
    sc = 0.11
    o, l = oatt.sparse_attn_decode_mq(q, lat, rope, topk, swa, swl, sc)
    main = [int(t) for t in topk if t >= 0]
    for i in range(3):
        lim = swl - (3 - 1 - i)
        keys = [list(lat[t]) + list(rope[t]) for t in main] + [list(swa[r]) for r in range(lim)]
        vals = [list(lat[t]) for t in main] + [list(swa[r][:512]) for r in range(lim)]
        for h in range(2):
            lg = [sc * math.fsum(q[i, h, c] * k[c] for c in range(576)) for k in keys]
            m = max(lg)
            w = [math.exp(x - m) for x in lg]
            z = math.fsum(w)
            assert abs(l[i, h] - (m + math.log(z))) < 1e-12
            for d in (0, 1, 255, 511):
                ref = math.fsum(wi * v[d] for wi, v in zip(w, vals)) / z
                assert abs(o[i, h, d] - ref) < 1e-12


def test_causality_and_independence():
    q, lat, rope, topk, swa, swl = _problem(9, 4)
    o, l = oatt.sparse_attn_decode_mq(q, lat, rope, topk, swa, swl, 0.05)
    # rows the first query cannot see (its limit is swl - 3) change nothing for it
    swa2 = swa.copy()
    swa2[swl - 3:] += 5.0
    q2 = q.copy()
    q2[1:] *= -3.0                                       # the other queries' inputs
    o2, l2 = oatt.sparse_attn_decode_mq(q2, lat, rope, topk, swa2, swl, 0.05)
    np.testing.assert_array_equal(o2[0], o[0])
    np.testing.assert_array_equal(l2[0], l[0])
    # the last query sees the whole valid window: the single-query decode
    ol, ll = oatt.sparse_attn_decode(q[3], lat, rope, topk, swa, swl, 0.05)
    np.testing.assert_allclose(o[3], ol, rtol=1e-12, atol=1e-12)


def test_short_window_and_empty_sets():
    """A window shorter than the draft block: the first queries see no window
    row; with no Top-K entry either, their result is o = 0, lse = -inf."""
    q, lat, rope, topk, swa, _ = _problem(11, 4)
    o, l = oatt.sparse_attn_decode_mq(q, lat, rope, np.full(8, -1), swa, 2, 0.05)
    assert np.all(o[:2] == 0) and np.all(np.isneginf(l[:2]))
    assert np.all(np.isfinite(l[2:]))
    o1, _ = oatt.sparse_attn_decode(q[2], lat, rope, np.full(8, -1), swa, 1, 0.05)
    np.testing.assert_allclose(o[2], o1, rtol=1e-12, atol=1e-12)

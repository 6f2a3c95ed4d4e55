"""Pins for the oracle's indexer (CPU only).

Checks against exact rational dot products, brute-force sorting with
deliberate ties, closed-form special cases, and the structural statements of
the pages (pool covering the whole context reduces the hierarchical indexer
to a flat Top-K; the Full layer's Top-K equals the flat Top-K).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import indexer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_round(x):
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000      # RNE to bf16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def e4m3_values():
    from oracle.codec import e4m3_decode
    v = e4m3_decode(np.arange(256))
    return v[np.isfinite(v)]


def rand_e4m3(rng, shape, scale=1.0):
    vals = e4m3_values()
    x = rng.standard_normal(shape) * scale
    idx = np.abs(x[..., None] - vals).argmin(-1)
    return vals[idx]


def exact_dot(q, k):
    return float(sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(q, k)))


def test_head_dots_match_fraction_fp8():
    rng = np.random.default_rng(0)
    q = bf16_round(rng.standard_normal((3, 128)))
    q[1, :10] *= 2.0 ** -40               # wide exponent spread in one head
    q[2, :5] *= 2.0 ** 60                 # forces the fsum path
    K = rand_e4m3(rng, (150, 128))
    d = indexer.head_dots_exact_multi(q, K)
    for h in range(3):
        for t in range(150):
            assert d[t, h] == exact_dot(q[h], K[t])


def test_head_dots_match_fraction_fp32():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 64)).astype(np.float32).astype(np.float64)
    K = rng.standard_normal((120, 64)).astype(np.float32).astype(np.float64)
    d = indexer.head_dots_exact_multi(q, K)
    for h in range(4):
        for t in range(120):
            assert d[t, h] == exact_dot(q[h], K[t])


def test_head_dots_cancellation_exact():
    """Heavy cancellation: sum = tiny exact value, far below float64 error."""
    q = np.array([1.0, 1.0, 1.0, 0.0])
    K = np.array([[2.0 ** 30, -(2.0 ** 30), 2.0 ** -20, 5.0]])
    assert indexer.head_dots_exact_multi(q[None], K)[0, 0] == 2.0 ** -20


def test_scores_unit_query_closed_form():
    """q_h = unit vector e_c, w = 1 -> s_t = max(k_tc, 0)."""
    rng = np.random.default_rng(2)
    K = rand_e4m3(rng, (64, 16))
    for c in range(16):
        q = np.zeros((1, 16)); q[0, c] = 1.0
        s = indexer.scores(q, np.array([1.0]), K)
        assert np.array_equal(s, np.maximum(K[:, c], 0.0))


def test_scores_opposite_heads_closed_form():
    """Heads q and -q with weights a, b: s = a*d if d > 0 else -b*d."""
    rng = np.random.default_rng(3)
    K = rand_e4m3(rng, (200, 32))
    q1 = bf16_round(rng.standard_normal(32))
    q = np.stack([q1, -q1])
    a, b = 0.75, 0.25
    s = indexer.scores(q, np.array([a, b]), K)
    d = np.array([exact_dot(q1, k) for k in K])
    want = np.where(d > 0, a * d, -b * d)
    assert np.array_equal(s, want)


def test_scores_invariances():
    rng = np.random.default_rng(4)
    q = bf16_round(rng.standard_normal((4, 32)))
    w = rng.random(4).astype(np.float32).astype(np.float64)
    K = rand_e4m3(rng, (300, 32))
    s = indexer.scores(q, w, K)
    perm = rng.permutation(32)
    assert np.array_equal(indexer.scores(q[:, perm], w, K[:, perm]), s)
    assert np.array_equal(indexer.scores(q, 2.0 * w, K), 2.0 * s)   # power-of-2 scale
    assert np.all(indexer.scores(q, np.zeros(4), K) == 0.0)
    # negative weights are allowed: a head with w<0 lowers the score
    s_neg = indexer.scores(q, -w, K)
    assert np.array_equal(s_neg, -s)


def test_block_scores_brute_force():
    rng = np.random.default_rng(5)
    for n in [1, 7, 8, 9, 63, 64, 65]:
        s = rng.integers(-5, 5, n).astype(np.float64)
        bs = indexer.block_scores(s, 8)
        want = [max(s[j:j + 8]) for j in range(0, n, 8)]
        assert bs.tolist() == want


def test_top_order_brute_force_with_ties():
    rng = np.random.default_rng(6)
    for n in [1, 5, 17, 64]:
        for _ in range(20):
            v = rng.integers(0, 4, n).astype(np.float64)      # many exact ties
            for k in range(0, n + 1):
                want = sorted(range(n), key=lambda i: (-v[i], i))[:k]
                assert indexer.top_order(v, k).tolist() == want


def test_top_order_signed_zero_is_a_tie():
    v = np.array([0.0, -0.0, 0.0, -0.0])
    assert indexer.top_order(v, 2).tolist() == [0, 1]


def _brute_full(q, w, K, pool_blocks, topk, block=8):
    n = K.shape[0]
    s = [sum(float(w[h]) * max(exact_dot(q[h], K[t]), 0.0) for h in range(q.shape[0]))
         for t in range(n)]
    nb = -(-n // block)
    bs = [max(s[j * block:min(n, j * block + block)]) for j in range(nb)]
    pool = sorted(sorted(range(nb), key=lambda j: (-bs[j], j))[:min(pool_blocks, nb)])
    pos = [t for j in pool for t in range(j * block, min(n, j * block + block))]
    sel = sorted(sorted(pos, key=lambda t: (-s[t], t))[:min(topk, len(pos))])
    return pool, sel + [-1] * (topk - len(sel))


def test_full_topk_brute_force_tiny():
    rng = np.random.default_rng(7)
    for n in [5, 8, 37, 64]:
        q = bf16_round(rng.standard_normal((3, 16)))
        w = rng.random(3).astype(np.float32).astype(np.float64)
        K = rand_e4m3(rng, (n, 16))
        for P, k in [(2, 4), (3, 16), (100, 8), (1, 3)]:
            r = indexer.full_topk(q, w, K, P, k)
            pool, sel = _brute_full(q, w, K, P, k)
            assert r["pool"].tolist() == pool
            assert r["topk"].tolist() == sel


def test_full_topk_ties_go_low():
    """Integer-valued, heavily tied scores: lower positions / blocks win."""
    K = np.zeros((40, 4))
    K[:, 0] = np.tile([1.0, 2.0, 2.0, 1.0, 0.0, 2.0, 1.0, 2.0], 5)
    q = np.array([[1.0, 0, 0, 0]])
    r = indexer.full_topk(q, np.array([1.0]), K, pool_blocks=2, topk=6)
    assert r["pool"].tolist() == [0, 1]                 # all blocks tie at 2
    assert r["topk"].tolist() == [1, 2, 5, 7, 9, 10]


def test_pool_covering_context_equals_flat_topk():
    rng = np.random.default_rng(8)
    q = bf16_round(rng.standard_normal((4, 32)))
    w = rng.random(4).astype(np.float32).astype(np.float64)
    K = rand_e4m3(rng, (500, 32))
    r = indexer.full_topk(q, w, K, pool_blocks=10 ** 6, topk=37)
    s = indexer.scores(q, w, K)
    flat = np.sort(indexer.top_order(s, 37))
    assert r["pool"].tolist() == list(range(63))
    assert r["topk"].tolist() == flat.tolist()


def test_full_topk_equals_flat_topk_with_small_pool():
    """Top-K of the pool = flat Top-K whenever pool_blocks >= K."""
    rng = np.random.default_rng(9)
    for trial in range(5):
        q = bf16_round(rng.standard_normal((4, 32)))
        w = rng.random(4).astype(np.float32).astype(np.float64)
        K = rand_e4m3(rng, (3000, 32))
        r = indexer.full_topk(q, w, K, pool_blocks=40, topk=40)
        flat = np.sort(indexer.top_order(r["scores"], 40))
        assert r["topk"].tolist() == flat.tolist()
        # ... and lies in the Top-K blocks
        topblocks = set(indexer.top_order(r["block_scores"], 40).tolist())
        assert set((r["topk"] // 8).tolist()) <= topblocks


def test_short_context_pads():
    rng = np.random.default_rng(10)
    q = bf16_round(rng.standard_normal((2, 16)))
    K = rand_e4m3(rng, (5, 16))
    r = indexer.full_topk(q, np.array([0.5, 0.5]), K, pool_blocks=2048, topk=8)
    assert r["pool"].tolist() == [0]
    assert r["topk"].tolist() == [0, 1, 2, 3, 4, -1, -1, -1]


def test_reindex_same_query_equals_full():
    rng = np.random.default_rng(11)
    q = bf16_round(rng.standard_normal((4, 32)))
    w = rng.random(4).astype(np.float32).astype(np.float64)
    K = rand_e4m3(rng, (2000, 32))
    f = indexer.full_topk(q, w, K, pool_blocks=64, topk=50)
    ri = indexer.reindex_topk(q, w, K, f["pool"], topk=50)
    assert ri["topk"].tolist() == f["topk"].tolist()


def test_reindex_reads_only_the_pool():
    rng = np.random.default_rng(12)
    q = bf16_round(rng.standard_normal((4, 32)))
    q2 = bf16_round(rng.standard_normal((4, 32)))
    w = rng.random(4).astype(np.float32).astype(np.float64)
    K = rand_e4m3(rng, (2000, 32))
    f = indexer.full_topk(q, w, K, pool_blocks=64, topk=50)
    K2 = K.copy()
    outside = np.setdiff1d(np.arange(2000), indexer.pool_positions(f["pool"], 2000))
    K2[outside] = 100.0                  # would dominate if it were read
    a = indexer.reindex_topk(q2, w, K, f["pool"], topk=50)
    b = indexer.reindex_topk(q2, w, K2, f["pool"], topk=50)
    assert a["topk"].tolist() == b["topk"].tolist()
    assert set(a["topk"].tolist()) <= set(indexer.pool_positions(f["pool"], 2000).tolist())


def test_golden_pool_geometry():
    g = json.load(open(os.path.join(GOLDEN, "formats.json")))
    assert indexer.BLOCK == g["indexer_block"]
    assert g["pool_blocks"] * g["indexer_block"] == g["pool_positions"]
    # a pool of 2048 blocks over a long context covers exactly 16,384 positions
    pool = np.arange(0, 2 * g["pool_blocks"], 2)
    assert indexer.pool_positions(pool, 10 ** 7).shape[0] == g["pool_positions"]

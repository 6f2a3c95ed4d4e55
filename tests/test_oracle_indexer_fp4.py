"""Pins for the oracle of the indexer with FP4 query and key (CPU only).

The FP4 indexer has no kernel yet; its oracle is pinned first.  Checks:
the storage size the format implies; exact round trips on the E2M1 grid; the
scores against exact rational arithmetic on tiny inputs and a brute-force
Top-K; equivariance under power-of-two scaling; a quantization error bound
derived from the codec's per-element bound; and that only the quantized
inputs matter.
"""
from fractions import Fraction

import numpy as np

from oracle import codec, indexer, indexer_fp4
from tests.test_oracle_indexer import bf16_round


def _grid_rows(rng, n, C, exps):
    """Rows whose every group of 16 holds signed E2M1 levels times 2^e with
    one element at +-6 * 2^e, so that amax / 6 = 2^e is an exact E4M3 scale."""
    lv = codec.E2M1_LEVELS
    x = lv[rng.integers(0, 8, (n, C))] * np.where(rng.random((n, C)) < 0.5, -1.0, 1.0)
    g = x.reshape(n, C // 16, 16)
    g[:, :, 0] = 6.0 * np.where(rng.random((n, C // 16)) < 0.5, -1.0, 1.0)
    e = rng.choice(exps, size=(n, C // 16))
    return (g * np.exp2(e)[..., None]).reshape(n, C)


def test_key_row_bytes():
    """128 E2M1 nibbles (64 B) plus one E4M3 byte per 16 channels (8 B)."""
    rng = np.random.default_rng(1)
    k = bf16_round(rng.standard_normal((5, 128)))
    codes, scales = indexer_fp4.quantize(k)
    assert codes.shape == (5, 64) and codes.dtype == np.uint8
    assert scales.shape == (5, 8) and scales.dtype == np.uint8
    assert indexer_fp4.KEY_ROW_BYTES == 72 == codes.shape[1] + scales.shape[1]


def test_grid_values_round_trip_and_score_unchanged():
    rng = np.random.default_rng(2)
    q = _grid_rows(rng, 4, 128, np.arange(-4, 5))
    k = _grid_rows(rng, 40, 128, np.arange(-6, 7))
    w = rng.random(4)
    qc, qs = indexer_fp4.quantize(q)
    kc, ks = indexer_fp4.quantize(k)
    np.testing.assert_array_equal(indexer_fp4.dequantize(qc, qs), q)
    np.testing.assert_array_equal(indexer_fp4.dequantize(kc, ks), k)
    np.testing.assert_array_equal(indexer_fp4.scores(qc, qs, w, kc, ks), indexer.scores(q, w, k))


def test_scores_match_fraction_arithmetic():
    """Tiny case: every head dot as an exact rational, rounded once; the head
    sum in head order (the indexer's exact-score rule)."""
    rng = np.random.default_rng(3)
    q = bf16_round(rng.standard_normal((3, 32)))
    k = bf16_round(rng.standard_normal((6, 32)) * 3.0)
    w = bf16_round(rng.random(3))
    qc, qs = indexer_fp4.quantize(q)
    kc, ks = indexer_fp4.quantize(k)
    s = indexer_fp4.scores(qc, qs, w, kc, ks)
    # the dequantized values from the E4M3 and E2M1 tables, then Fractions
    def dq(codes, scales):
        out = []
        for r in range(codes.shape[0]):
            row = []
            for j in range(2 * codes.shape[1]):
                nib = (int(codes[r, j // 2]) >> (4 * (j % 2))) & 0xF
                sc = codec.e4m3_decode(np.array([scales[r, j // 16]]))[0]
                mag = [0, 0.5, 1, 1.5, 2, 3, 4, 6][nib & 7]
                row.append(Fraction(-mag if nib & 8 else mag) * Fraction(float(sc)))
            out.append(row)
        return out
    Q, K = dq(qc, qs), dq(kc, ks)
    for t in range(6):
        acc = 0.0
        for h in range(3):
            d = float(sum(a * b for a, b in zip(Q[h], K[t])))
            acc = acc + float(w[h]) * (d if d > 0 else 0.0)
        assert acc == s[t]


def test_full_topk_brute_force_tiny():
    rng = np.random.default_rng(4)
    n = 200
    q = bf16_round(rng.standard_normal((2, 32)))
    k = bf16_round(rng.standard_normal((n, 32)))
    w = bf16_round(rng.random(2))
    r = indexer_fp4.full_topk(q, w, k, pool_blocks=5, topk=12)
    s = indexer_fp4.scores(*indexer_fp4.quantize(q), w, *indexer_fp4.quantize(k))
    bs = [max(s[8 * j: 8 * j + 8]) for j in range(n // 8)]
    pool = sorted(sorted(range(len(bs)), key=lambda j: (-bs[j], j))[:5])
    np.testing.assert_array_equal(r["pool"], pool)
    pos = [8 * j + i for j in pool for i in range(8)]
    top = sorted(sorted(pos, key=lambda t: (-s[t], t))[:12])
    np.testing.assert_array_equal(r["topk"], top)


def test_power_of_two_equivariance():
    """k * 2^j quantizes to the same codes with scales times 2^j (no E4M3
    subnormals or saturation on the way), so every score scales by 2^j."""
    rng = np.random.default_rng(5)
    q = bf16_round(rng.standard_normal((4, 128)))
    k = bf16_round(rng.standard_normal((64, 128)))
    w = rng.random(4)
    qc, qs = indexer_fp4.quantize(q)
    kc, ks = indexer_fp4.quantize(k)
    base = indexer_fp4.scores(qc, qs, w, kc, ks)
    for j in (-2, -1, 1, 3):
        kc2, ks2 = indexer_fp4.quantize(k * 2.0 ** j)
        np.testing.assert_array_equal(kc2, kc)
        np.testing.assert_array_equal(codec.e4m3_decode(ks2), codec.e4m3_decode(ks) * 2.0 ** j)
        np.testing.assert_array_equal(indexer_fp4.scores(qc, qs, w, kc2, ks2), base * 2.0 ** j)


def test_quantization_error_bound():
    """|s_fp4 - s| <= sum_h |w_h| sum_c (|q||dk| + |dq||k| + |dq||dk|), with
    |x - dq(x)| <= the group's scale (the codec's per-element bound) and
    ReLU 1-Lipschitz; plus float64 rounding slack."""
    rng = np.random.default_rng(6)
    q = bf16_round(rng.standard_normal((8, 128)))
    k = bf16_round(rng.standard_normal((300, 128)) * np.exp(rng.normal(0, 0.5, 128)))
    w = rng.random(8)
    qc, qs = indexer_fp4.quantize(q)
    kc, ks = indexer_fp4.quantize(k)
    s4 = indexer_fp4.scores(qc, qs, w, kc, ks)
    s = indexer.scores(q, w, k)
    eq = np.repeat(codec.e4m3_decode(qs), 16, axis=1)      # per-element error bounds
    ek = np.repeat(codec.e4m3_decode(ks), 16, axis=1)
    bound = (np.abs(q) @ ek.T + eq @ np.abs(k).T + eq @ ek.T)   # [Hi, n]
    bound = (np.abs(w)[:, None] * bound).sum(axis=0)
    slack = 1e-12 * (np.abs(w)[:, None] * (np.abs(q) @ np.abs(k).T)).sum(axis=0)
    assert np.all(np.abs(s4 - s) <= bound + slack)
    assert np.any(s4 != s)                                  # the quantization is not a no-op


def test_depends_only_on_quantized_inputs():
    """Quantizing a dequantized row gives the same codes back, so the result
    for raw inputs equals the result for their dequantized images."""
    rng = np.random.default_rng(7)
    q = bf16_round(rng.standard_normal((4, 128)))
    k = bf16_round(rng.standard_normal((500, 128)))
    w = rng.random(4)
    qd = indexer_fp4.dequantize(*indexer_fp4.quantize(q))
    kd = indexer_fp4.dequantize(*indexer_fp4.quantize(k))
    a = indexer_fp4.full_topk(q, w, k, pool_blocks=16, topk=32)
    b = indexer_fp4.full_topk(qd, w, kd, pool_blocks=16, topk=32)
    np.testing.assert_array_equal(a["scores"], b["scores"])
    np.testing.assert_array_equal(a["topk"], b["topk"])
    pool = a["pool"]
    ra = indexer_fp4.reindex_topk(q, w, k, pool, topk=32)
    rb = indexer.reindex_topk(qd, w, kd, pool, topk=32)
    np.testing.assert_array_equal(ra["topk"], rb["topk"])

"""Pins for the oracle's FP4 codec (CPU only).

Each test checks ``oracle.codec`` against something other than itself:
exact rational arithmetic (``fractions.Fraction``), an independent
threshold formulation, hand-worked examples and round-trip identities.
"""
import bisect
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_bf16_finite():
    """Every finite bf16 value (as float64), from the bit patterns."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


def e4m3_fraction_table():
    """(code, Fraction) for every non-negative finite E4M3 code, by the OCP rule."""
    out = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else \
            (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((c, v))
    return out


def fraction_rne(x: Fraction, table):
    """Nearest table entry to x >= 0, ties to the even code, saturating."""
    vals = [v for _, v in table]
    i = bisect.bisect_left(vals, x)
    if i == 0:
        return table[0][0]
    if i == len(vals):
        return table[-1][0]
    lo, hi = table[i - 1], table[i]
    dl, dh = x - lo[1], hi[1] - x
    if dl < dh:
        return lo[0]
    if dh < dl:
        return hi[0]
    return lo[0] if lo[0] % 2 == 0 else hi[0]


def test_golden_format_constants():
    g = json.load(open(os.path.join(GOLDEN, "formats.json")))
    assert list(codec.E2M1_LEVELS) == g["e2m1_levels"]
    assert codec.E4M3_MAX == g["e4m3_max"]
    assert codec.GROUP == g["group_size"]
    assert codec.e4m3_decode(np.array([0x7E]))[0] == g["e4m3_max"]


def test_e4m3_decode_matches_ocp_definition():
    table = e4m3_fraction_table()
    got = codec.e4m3_decode(np.arange(256))
    for c, v in table:
        assert got[c] == float(v)
        assert got[c | 0x80] == -float(v) or (v == 0 and got[0x80] == 0)
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.signbit(got[0x80])


def test_scale_rounding_exhaustive_over_bf16_amax():
    """s_code(amax) for every non-negative finite bf16 amax vs exact rounding."""
    table = e4m3_fraction_table()
    a = all_bf16_finite()
    a = np.unique(np.abs(a))
    got = codec.e4m3_encode_rne_sat(a / 6.0)
    for ai, gi in zip(a, got):
        want = fraction_rne(Fraction(float(ai)) / 6, table)
        assert int(gi) == want, (ai, gi, want)


def test_element_rounding_exhaustive_threshold_form():
    """Every bf16 |x| against every positive E4M3 scale.

    Independent formulation: the magnitude code is the number of decision
    thresholds passed, thresholds T = M*s at the E2M1 midpoints M, where a
    move into an odd code needs |x| > T and into an even code |x| >= T.  Both
    sides of each comparison are exact in float64 (M*s has <= 7 bits).
    """
    x = np.unique(np.abs(all_bf16_finite()))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    scales = codec.e4m3_decode(np.arange(1, 0x7F))
    for s in scales:
        r = x / s
        got = codec.e2m1_round_magnitude(r)
        want = np.zeros(x.shape, dtype=np.int64)
        for i, M in enumerate(mids):
            target = i + 1
            T = M * s
            want += (x > T) if target % 2 == 1 else (x >= T)
        assert np.array_equal(got, want), s


def test_element_rounding_fraction_spot_checks():
    """Random (x, s) pairs and all exact midpoints against Fraction rounding."""
    levels = [(i, Fraction(v)) for i, v in enumerate(codec.E2M1_LEVELS)]
    rng = np.random.default_rng(1)
    x = np.unique(np.abs(all_bf16_finite()))
    scales = codec.e4m3_decode(np.arange(1, 0x7F))
    pairs = [(x[i], scales[j]) for i, j in zip(rng.integers(0, x.size, 4000),
                                                rng.integers(0, scales.size, 4000))]
    for M in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]:
        for s in scales[::7]:
            pairs.append((M * s, s))
    for xv, s in pairs:
        want = fraction_rne(Fraction(float(xv)) / Fraction(float(s)), levels)
        got = int(codec.e2m1_round_magnitude(np.array([xv / s]))[0])
        assert got == want, (xv, s, got, want)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "codec_worked_example.json")))
    x = np.array(g["x"])[None, :]
    codes, scales = codec.quantize_rows(x)
    assert codes[0].tolist() == g["codes"]
    assert scales[0].tolist() == g["scales"]


def test_sixteen_codes_round_trip():
    """Groups x = c_i * s with amax = 6 s recover every E2M1 code exactly."""
    rng = np.random.default_rng(2)
    signed = np.concatenate([codec.E2M1_LEVELS, -codec.E2M1_LEVELS])   # 16 codes
    for s_code in range(1, 0x7F):
        s = codec.e4m3_decode(np.array([s_code]))[0]
        if 6 * s > 3.0e38:
            continue
        perm = rng.permutation(16)
        vals = signed[perm].copy()
        vals[np.argmax(np.abs(vals))] = 6.0   # keep one +6 so amax = 6 s
        if not np.any(np.abs(vals) == 6.0):
            vals[0] = 6.0
        x = np.tile(vals * s, 2)[None, :]      # 32 channels = 2 groups
        codes, scales = codec.quantize_rows(x)
        assert scales[0].tolist() == [s_code, s_code]
        back = codec.dequantize_rows(codes, scales)
        assert np.array_equal(back, x)
        nib = np.empty(32, dtype=np.int64)
        nib[0::2], nib[1::2] = codes[0] & 15, codes[0] >> 4
        mag = codec.E2M1_LEVELS[nib & 7] * np.where(nib & 8, -1, 1)
        assert np.array_equal(mag, np.tile(vals, 2))


def test_negative_zero_keeps_sign():
    s = 1.0
    x = np.zeros((1, 32))
    x[0, 0] = 6.0 * s           # amax -> scale 1
    x[0, 1] = -0.1              # rounds to zero, negative
    x[0, 2] = -0.0
    x[0, 3] = 0.1
    codes, _ = codec.quantize_rows(x)
    assert codes[0, 0] == (0x7 | (0x8 << 4))
    assert codes[0, 1] == (0x8 | (0x0 << 4))


def test_nibble_layout_pattern():
    """Channel 2j lands in the low nibble of byte j, channel 2j+1 in the high."""
    x = np.zeros((1, 32))
    x[0, :16] = 6.0                     # group 0: scale 1, all code 7
    x[0, 16] = 6.0
    x[0, 17] = 0.5                      # group 1: channel 17 -> code 1 (high nibble)
    codes, scales = codec.quantize_rows(x)
    assert codes[0, :8].tolist() == [0x77] * 8
    assert codes[0, 8] == 0x17
    assert codes[0, 9:].tolist() == [0] * 7


def test_p1_rule_agrees_off_ties():
    """[P1]'s argmin rule equals ties-to-even wherever no tie or -0 occurs."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
    a, sa = codec.quantize_rows(x)
    b, sb = codec.quantize_rows(x, p1_mode=True)
    assert np.array_equal(sa, sb)
    s = np.repeat(codec.e4m3_decode(sa), 16, axis=1)
    r = np.abs(x) / s
    tie = np.isin(r, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    negzero = (x < 0) & (r < 0.25)
    na = np.empty(x.shape, np.int64); na[:, 0::2], na[:, 1::2] = a & 15, a >> 4
    nb = np.empty(x.shape, np.int64); nb[:, 0::2], nb[:, 1::2] = b & 15, b >> 4
    ok = ~(tie | negzero)
    assert np.array_equal(na[ok], nb[ok])
    assert np.any(na[~ok] != nb[~ok])


def test_dequant_error_bound_random():
    """|x - dq(x)| <= s (half the widest E2M1 gap times s); exact if x = level*s."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((200, 512)) * np.exp(rng.normal(0, 2, (200, 1)))
    x = x.astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
    codes, scales = codec.quantize_rows(x)
    dq = codec.dequantize_rows(codes, scales)
    s = np.repeat(codec.e4m3_decode(scales), 16, axis=1)
    sat = np.abs(x) > 6.0 * s          # saturated groups (amax/6 above 448)
    assert np.all(np.abs(x - dq)[~sat] <= s[~sat])
    assert np.all(np.abs(dq[sat]) == 6.0 * s[sat])
    # rounding goes to the nearest level: no other level is strictly closer
    lv = np.concatenate([codec.E2M1_LEVELS, -codec.E2M1_LEVELS])
    d_all = np.abs(x[..., None] - lv * s[..., None])
    assert np.all(np.abs(x - dq) <= d_all.min(-1) + 0.0)

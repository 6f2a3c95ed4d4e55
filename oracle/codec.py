"""Oracle: FP4 E2M1 main-KV codec with one E4M3 scale per 16 channels.

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix
------------------
* Main KV entries are stored as FP4 E2M1 values with one E4M3 scale for every
  16 channels, and are dequantized just before attention; there is no FP4
  arithmetic ([P3] section 3.2 "FP4 main KV"; [P1] section 4).
* The E2M1 magnitude set is {0, 0.5, 1, 1.5, 2, 3, 4, 6} with a sign bit
  ([P1] section 8, ``FP4Quantizer.e2m1_levels``; [P4] section 3, "Microscopic
  FP4 (E2M1) Cache Compression": 1 sign, 2 exponent, 1 mantissa bit).
* The per-group scale is amax / 6, limited to the E4M3 maximum 448, and there
  is no second-level (per-tensor) scale ([P1] section 8,
  ``FP4Quantizer.quantize_and_pack`` and its docstring).

Readings where the pages are silent or disagree (each also listed in the
design notes):

* Group size 16 ([P1], [P3]); [P4]'s 32-element blocks are not followed.
* The scale is *stored* as an E4M3 code: amax/6 is rounded to E4M3 with
  round-to-nearest-even and saturation to 448 (the OCP conversion default).
  [P1]'s simulation keeps an unrounded fp32 scale, which cannot be stored in
  the 890 B/token format the pages describe.
* Elements round onto the E2M1 grid with round-to-nearest, ties to the even
  code, saturating at 6, keeping the sign bit of the input (also for results
  that round to zero).  [P1]'s ``argmin`` picks the lower level on ties and
  returns +0 for small negatives; ``p1_mode=True`` reproduces that rule for a
  cross-check on non-tie inputs.
* A group whose scale rounds to zero stores magnitude code 0 for every
  element (the sign bit is kept).
* Byte ``j`` of a packed row holds element ``2j`` in its low nibble and element
  ``2j+1`` in its high nibble.

Everything is plain numpy in float64.  Inputs are bf16 or E4M3 values, which
float64 holds exactly; every rounding step below is done explicitly.
"""
from __future__ import annotations

import numpy as np

GROUP = 16                      # channels per E4M3 scale ([P3] 3.2, [P1] 4)
E2M1_LEVELS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # [P1] 8
E4M3_MAX = 448.0                # [P1] section 8, "E4M3 max range 448"


# --------------------------------------------------------------------------
# E4M3 (OCP FP8, bias 7, subnormals, no infinities, S.1111.111 = NaN)
# --------------------------------------------------------------------------
def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 byte codes as float64 (NaN codes give NaN)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** -9                              # e == 0: m/8 * 2^(1-7)
    nrm = (8 + m) * np.exp2(e.astype(np.float64) - 10.0)   # (1+m/8)*2^(e-7)
    val = np.where(e == 0, sub, nrm)
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode_rne_sat(t: np.ndarray) -> np.ndarray:
    """Round non-negative float64 values to E4M3, nearest-even, saturating.

    Returns uint8 codes.  The grid spacing at magnitude t is 2^(E-3) for
    normals (E = floor(log2 t) >= -6) and 2^-9 below 2^-6.  Dividing by a
    power of two is exact, so ``rint`` (ties to even) performs the rounding.
    """
    t = np.asarray(t, dtype=np.float64)
    if np.any(t < 0) or np.any(~np.isfinite(t)):
        raise ValueError("e4m3_encode_rne_sat takes finite non-negative values")
    _, ex = np.frexp(t)                   # t = f * 2^ex, f in [0.5, 1)
    E = ex.astype(np.int64) - 1           # floor(log2 t) for t > 0
    E = np.where(t > 0, np.maximum(E, -6), -6)
    spacing = np.exp2((E - 3).astype(np.float64))
    v = np.rint(t / spacing) * spacing
    v = np.minimum(v, E4M3_MAX)
    # encode the (now representable) value v
    _, ex2 = np.frexp(v)
    E2 = ex2.astype(np.int64) - 1
    normal = (v >= 2.0 ** -6)
    e_field = np.where(normal, E2 + 7, 0)
    m_field = np.where(normal,
                       v / np.exp2((E2 - 3).astype(np.float64)) - 8.0,
                       v / 2.0 ** -9)
    m_field = np.where(v == 0, 0.0, m_field)
    e_field = np.where(v == 0, 0, e_field)
    code = (e_field << 3) | m_field.astype(np.int64)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# E2M1
# --------------------------------------------------------------------------
def e2m1_round_magnitude(r: np.ndarray, p1_mode: bool = False) -> np.ndarray:
    """Index (0..7) into E2M1_LEVELS of the level nearest to r >= 0.

    Ties go to the even index (round-half-even on the E2M1 code).  With
    ``p1_mode`` ties go to the lower level, as ``torch.argmin`` does in [P1]'s
    simulation.  Values above 6 saturate to index 7 (6 is simply nearest).
    """
    r = np.asarray(r, dtype=np.float64)
    # Every r >= 5 rounds to 6; capping at 7 keeps that decision and keeps
    # the float64 distances below exact (huge r would make them all equal).
    r = np.minimum(r, 7.0)
    dist = np.abs(r[..., None] - E2M1_LEVELS)
    best = np.argmin(dist, axis=-1)                 # first (lower) minimum
    if not p1_mode:
        nxt = np.minimum(best + 1, 7)
        d_best = np.take_along_axis(dist, best[..., None], -1)[..., 0]
        d_next = np.take_along_axis(dist, nxt[..., None], -1)[..., 0]
        tie = (nxt != best) & (d_next == d_best)
        best = np.where(tie & (best % 2 == 1), nxt, best)
    return best.astype(np.int64)


# --------------------------------------------------------------------------
# Row codec
# --------------------------------------------------------------------------
def quantize_rows(x: np.ndarray, p1_mode: bool = False):
    """FP4 KV write for rows of bf16 values (given as float64).

    x: [n, C] with C a multiple of 16.  Returns ``(codes, scales)`` with
    codes uint8 [n, C/2] (two E2M1 nibbles per byte, even channel low) and
    scales uint8 [n, C/16] (E4M3 codes).

    Steps per group of 16 channels ([P1] section 8 ``quantize_and_pack``;
    rounding as stated in the module docstring):
      a = max |x|;  s_code = E4M3_rne_sat(a / 6);  s = decode(s_code);
      m = E2M1 level nearest to |x| / s (0 if s == 0);
      nibble = sign(x) << 3 | m.
    """
    x = np.asarray(x, dtype=np.float64)
    n, C = x.shape
    if C % (2 * GROUP):
        raise ValueError("channel count must be a multiple of 32")
    g = x.reshape(n, C // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    # a/6 in float64: a has <= 8 significant bits, so a/6 is either exact or
    # non-terminating in binary and can never sit on an E4M3 rounding
    # midpoint; the second rounding below is therefore exact rounding.
    s_code = e4m3_encode_rne_sat(amax / 6.0)
    s = e4m3_decode(s_code)
    s_b = np.broadcast_to(s[..., None], g.shape)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(s_b > 0, np.abs(g) / np.where(s_b > 0, s_b, 1.0), 0.0)
    m = e2m1_round_magnitude(r, p1_mode=p1_mode)
    if p1_mode:
        # [P1]: the argmin over the signed level list maps results that
        # round to zero onto +0 and never uses the -0 entry.
        sign = np.signbit(g) & (m != 0)
    else:
        sign = np.signbit(g)
    nib = (sign.astype(np.int64) << 3) | m
    nib = nib.reshape(n, C)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return codes, s_code.astype(np.uint8)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse of :func:`quantize_rows`: float64 [n, 2*codes.shape[1]].

    value = (-1)^sign * E2M1_LEVELS[m] * decode(scale)  ([P1] section 4: the
    FP4 values are dequantized back just before attention).  The products
    have at most 6 significant bits, so they are exact in float64 (and in
    bf16 and fp32).
    """
    codes = np.asarray(codes, dtype=np.int64)
    n, half = codes.shape
    nib = np.empty((n, 2 * half), dtype=np.int64)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = (codes >> 4) & 0xF
    mag = E2M1_LEVELS[nib & 7]
    sgn = np.where(nib & 8, -1.0, 1.0)
    s = e4m3_decode(scales)                         # [n, C/16]
    s = np.repeat(s, GROUP, axis=1)
    return sgn * mag * s

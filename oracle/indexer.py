"""Oracle: CSA2 hierarchical sparse indexer (Full scan, pool, Top-K, Reindex).

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix
------------------
* The first decoder layer in Full mode scores every causally visible
  position; blocks of 8 positions are ranked and the Top-2048 blocks (a
  16,384-position candidate pool) are kept; later Reindex layers score only
  inside the pool and take Top-512, so their cost no longer grows with the
  context ([P3] section 3.2, "Hierarchical Sparse Indexer (decoder)"; [P1]
  section 3, "Hierarchical Sparse Indexer"; [P1] section 8,
  ``HierarchicalSparseIndexer.forward``: Full branch = score all keys and take
  top-k, re-indexing branch = gather the pool's keys and score only those).
* Full mode computes new Top-K indices; Reindex re-scores with its own indexer
  query over the main KV / indexer K of the latest Full layer; Reuse keeps the
  indices ([P3] section 3.2, mode table; [P2] "CSA2: compressão em três
  dimensões").

Readings (the pages are silent; each is listed in the design notes):

* Score of position t: ``s_t = sum_h w_h * ReLU(q_h . k_t)`` -- a weighted
  sum over indexer heads of rectified per-head dot products.  [P1]'s
  simulation uses a single plain dot product; the multi-head weighted form is
  the one this library implements.
* Block score = max of the scores of its (up to 8) positions; the last block
  of a context may be partial.
* Ordering is (score descending, index ascending): equal scores go to the
  lower index.  Selected sets are returned sorted ascending; Top-K outputs
  are padded with -1 when fewer than K positions exist.
* The Full layer's own attention indices are the Top-K of the pool's
  positions by the Full layer's scores (equal to the flat Top-K over the
  whole context, a property the tests check).
* Pool size is min(pool_blocks, number of blocks): short contexts keep every
  block.

Arithmetic: every head dot product is the exact value rounded once to
float64 (the exact products of bf16 x E4M3 or fp32 x fp32 factors are summed
by ``math.fsum``, or -- for speed on large inputs -- by exact int64
fixed-point arithmetic whose range is checked first).  The weighted sum over
heads is then plain float64 arithmetic in ascending head order:
``s = 0; for h: s = s + w_h * relu(d_h)``.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 8          # positions per indexer block ([P3] 3.2)


# --------------------------------------------------------------------------
# head dot products: exact sum, rounded once
# --------------------------------------------------------------------------
def _is_f32_representable(x: np.ndarray) -> bool:
    x = np.asarray(x, dtype=np.float64)
    return bool(np.all(np.asarray(x, dtype=np.float32).astype(np.float64) == x))


def head_dots_fsum(q_h: np.ndarray, K: np.ndarray) -> np.ndarray:
    """d_t = RN64( sum_c q_c * K[t, c] ) with math.fsum over exact products.

    Both factors must be fp32-representable (bf16 and E4M3 are), so every
    float64 product below is exact (<= 48 significant bits, no underflow).
    """
    q_h = np.asarray(q_h, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    if not (_is_f32_representable(q_h) and _is_f32_representable(K)):
        raise ValueError("indexer factors must be fp32-representable")
    prods = K * q_h[None, :]
    return np.array([math.fsum(row) for row in prods], dtype=np.float64)


def _lsb_exponent(x: np.ndarray):
    """Smallest exponent e with x * 2^-e integral for every element (or None).

    Reads the fp32 bit fields of fp32-representable values: a normal value is
    (2^23 + mant) * 2^(E-150), a subnormal one mant * 2^-149; the lowest set
    bit of the significand gives each element's lsb exponent.
    """
    f = np.ascontiguousarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    best = None
    for a in range(0, f.shape[0], 1 << 22):
        c = f[a:a + (1 << 22)]
        E = ((c >> 23) & 0xFF).astype(np.int32)
        sig = np.where(E == 0, c & 0x7FFFFF, (c & 0x7FFFFF) | 0x800000)
        nz = sig != 0
        if not np.any(nz):
            continue
        s = sig[nz].astype(np.int64)
        low = s & (-s)                                # lowest set bit
        tz = np.frexp(low.astype(np.float64))[1] - 1
        e2 = np.where(E[nz] == 0, -149, E[nz] - 150)
        m = int(np.min(e2 + tz))
        best = m if best is None else min(best, m)
    return best


def _int_repr(x: np.ndarray):
    """Write fp32-representable x as X * 2^e with X integral (float64 array).

    Returns (X, e); X holds exact integers (a power-of-two rescale of x), or
    (None, None) if some |X| >= 2^62.
    """
    x = np.asarray(x, dtype=np.float64)
    e = _lsb_exponent(x)
    if e is None:
        return np.zeros(x.shape, dtype=np.float64), 0
    X = np.ldexp(x, -e)                              # exact integers
    if X.size and np.max(np.abs(X)) >= 2.0 ** 62:
        return None, None
    return X, e


def head_dots_exact(q_h: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Correctly rounded float64 head dot products for every row of K."""
    return head_dots_exact_multi(np.asarray(q_h)[None, :], K)[:, 0]


def head_dots_exact_multi(q: np.ndarray, K: np.ndarray,
                          chunk: int = 1 << 16) -> np.ndarray:
    """d[t, h] = RN64(exact q_h . K[t]) for all heads, [n, Hi] float64.

    Uses exact integer fixed-point arithmetic when the ranges provably fit
    (sum_c |Q_c| * max|K| < 2^62 for the head; held in float64 when the bound
    is below 2^53, in int64 otherwise), else math.fsum over the exact float64
    products.  int64 -> float64 conversion rounds to
    nearest-even and the power-of-two rescale is exact, so both paths give
    RN64(exact sum).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    if not (_is_f32_representable(q) and _is_f32_representable(K)):
        raise ValueError("indexer factors must be fp32-representable")
    n, hi = K.shape[0], q.shape[0]
    out = np.empty((n, hi), dtype=np.float64)
    if n == 0:
        return out
    Ki, ek = _int_repr(K)
    kmax = float(np.max(np.abs(Ki))) if Ki is not None else None
    int_heads, Qcols, eqs = [], [], []
    for h in range(hi):
        Q, eq = _int_repr(q[h])
        if Q is not None and Ki is not None and \
                float(np.sum(np.abs(Q))) * kmax < 2.0 ** 62:
            int_heads.append(h)
            Qcols.append(Q)
            eqs.append(eq)
        else:
            out[:, h] = head_dots_fsum(q[h], K)
    if int_heads:
        Qm = np.stack(Qcols, axis=1)                 # [D, h_int], integral
        bound = float(np.max(np.sum(np.abs(Qm), axis=0))) * kmax
        # Below 2^53 every partial sum of the integer terms is an integer that
        # float64 holds exactly, whatever the summation order, so a float64
        # matrix product of the integer-valued operands is exact as well.
        use_f64 = bound < 2.0 ** 53
        Qi = Qm.astype(np.int64)
        for a in range(0, n, chunk):
            if use_f64:
                d_int = Ki[a:a + chunk] @ Qm                         # exact
            else:
                d_int = (Ki[a:a + chunk].astype(np.int64) @ Qi).astype(np.float64)
            for j, h in enumerate(int_heads):
                out[a:a + chunk, h] = np.ldexp(d_int[:, j], eqs[j] + ek)
    return out


def scores(q: np.ndarray, w: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Indexer scores s_t = sum_h w_h * ReLU(d_{t,h}) for every row of K.

    q: [Hi, D] query of the indexer heads, w: [Hi] head weights, K: [n, D]
    indexer keys.  Heads are accumulated in ascending order in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    d = head_dots_exact_multi(q, K)
    s = np.zeros(d.shape[0], dtype=np.float64)
    for h in range(q.shape[0]):
        relu = np.where(d[:, h] > 0, d[:, h], 0.0)
        s = s + w[h] * relu
    return s


def block_scores(s: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """bs_j = max of s over positions [block*j, min(block*j+block, n))."""
    s = np.asarray(s, dtype=np.float64)
    n = s.shape[0]
    nb = -(-n // block)
    pad = np.full(nb * block, -np.inf)
    pad[:n] = s
    return pad.reshape(nb, block).max(axis=1)


def top_order(values: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k best values under (value descending, index ascending)."""
    values = np.asarray(values, dtype=np.float64)
    order = np.lexsort((np.arange(values.shape[0]), -values))
    return order[:k]


def _margin(sorted_vals: np.ndarray, k: int) -> float:
    """Relative gap between the k-th and (k+1)-th best values (inf if none)."""
    if k <= 0 or k >= sorted_vals.shape[0]:
        return math.inf
    a, b = sorted_vals[k - 1], sorted_vals[k]
    den = max(abs(a), abs(b), 1e-300)
    return float((a - b) / den)


def pool_positions(pool: np.ndarray, n_ctx: int, block: int = BLOCK) -> np.ndarray:
    """Positions covered by the pool's blocks, ascending, clipped to n_ctx."""
    pool = np.sort(np.asarray(pool, dtype=np.int64))
    pos = (pool[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return pos[pos < n_ctx]


def select_topk_positions(s_pos: np.ndarray, positions: np.ndarray, topk: int):
    """Top-K of the given positions by score; ascending, padded with -1."""
    kk = min(topk, positions.shape[0])
    sel = positions[top_order(s_pos, kk)]
    out = np.full(topk, -1, dtype=np.int64)
    out[:kk] = np.sort(sel)
    vals = np.sort(np.asarray(s_pos, dtype=np.float64))[::-1]
    return out, _margin(vals, kk)


def full_topk(q, w, K, pool_blocks: int, topk: int, block: int = BLOCK):
    """Full-mode indexer for one sequence: pool and Top-K.

    K holds the indexer keys of every causally visible position [n_ctx, D].
    Returns a dict with ``pool`` (ascending block ids, length
    min(pool_blocks, NB)), ``topk`` (ascending positions, -1 padded),
    ``scores`` / ``block_scores`` (float64) and the relative ``margin_pool`` /
    ``margin_topk`` at each cut (small margins flag near-ties).
    """
    K = np.asarray(K, dtype=np.float64)
    n_ctx = K.shape[0]
    s = scores(q, w, K)
    bs = block_scores(s, block)
    nb = bs.shape[0]
    P = min(pool_blocks, nb)
    pool = np.sort(top_order(bs, P))
    m_pool = _margin(np.sort(bs)[::-1], P)
    pos = pool_positions(pool, n_ctx, block)
    sel, m_top = select_topk_positions(s[pos], pos, topk)
    return {"pool": pool, "topk": sel, "scores": s, "block_scores": bs,
            "margin_pool": m_pool, "margin_topk": m_top}


def reindex_topk(q, w, K, pool, topk: int, block: int = BLOCK):
    """Reindex mode for one sequence: score only the pool's positions.

    K is the full indexer-key array of the latest Full layer [n_ctx, D]; only
    the rows of the pool's positions are read.
    """
    K = np.asarray(K, dtype=np.float64)
    pos = pool_positions(pool, K.shape[0], block)
    s = scores(q, w, K[pos])
    sel, m_top = select_topk_positions(s, pos, topk)
    return {"topk": sel, "scores": s, "positions": pos, "margin_topk": m_top}

"""Oracle: CSA2 sparse MLA-style core attention for one decode query.

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix
------------------
* Core attention reads, under one main query, the main KV entries picked by
  the Top-K indices (a 512-dim latent shared by all heads) and the exact,
  uncompressed SWA KV of the recent window; both branches are merged
  ([P3] section 3.2, figure "异构 KV" and the paragraph after it: nearby
  tokens need exact K/V, far tokens use main KV + Top-K, both are read by the
  same main Q and merged).
* Main KV is dequantized from FP4 just before attention ([P1] section 4).
* The latent is 512-dim and shared across heads ([P2] "CSA2: compressão em
  três dimensões"); a 64-dim high-precision channel sits beside the FP4 part
  ([P4] section 3, "dedicated 64-dimensional high-precision ... channel").
* Reuse layers keep KV and indices and change only the query ([P3] 3.2 mode
  table; [P2] same section).

Readings (each also in the design notes):

* MLA decode form: key = [latent ; rope] (576 channels), value = latent (512
  channels); the query is already absorbed and rotated (576 channels per
  head); the output is the 512-dim latent per head.  The 64-dim channel is
  the bf16 rope part of the key.
* One softmax over the union E = {valid Top-K entries} + {SWA rows}; nothing
  is masked or de-duplicated when a position is in both.  No attention sink.
* logits = scale * q_h . k_e; o_h = sum_e softmax(logits)_e v_e;
  lse_h = m + ln(sum_e exp(logit_e - m)) with m the max logit.  An empty E
  gives o = 0 and lse = -inf.

Multi-query decode (speculative verification: [P2] DSpark paragraph, draft
blocks over the SWA-128 window; [P3] section 3 component table, DSpark row).
Readings:

* The q_len query tokens of a sequence are its newest tokens, oldest first;
  they are the last q_len rows of the valid SWA window and share the layer's
  Top-K set (the indexer context is the committed prefix).
* Query i sees every valid Top-K entry and the window rows
  r < swa_len - (q_len - 1 - i): its own row and the older ones (causal
  within the draft block).  q_len = 1 is the single-query decode above.

Arithmetic is float64 (numpy / BLAS matrix products as library steps).
"""
from __future__ import annotations

import numpy as np

LATENT = 512
ROPE = 64
D_QK = LATENT + ROPE


def sparse_attn_decode(q, latent, rope, topk, swa, swa_len, scale):
    """Joint-softmax attention of one decode query over main KV + SWA.

    q: [H, 576] query (float64 of bf16 values).
    latent: [n_ctx, 512] dequantized main-KV latent (float64).
    rope: [n_ctx, 64] rope part of the main key (float64 of bf16).
    topk: [K] selected positions, -1 = padding.
    swa: [W, 576] SWA key rows (value = first 512 channels); the first
    ``swa_len`` rows are valid.
    Returns (out [H, 512] float64, lse [H] float64).
    """
    q = np.asarray(q, dtype=np.float64)
    topk = np.asarray(topk, dtype=np.int64)
    idx = topk[topk >= 0]
    lat_sel = np.asarray(latent[idx], dtype=np.float64).reshape(idx.shape[0], LATENT)
    rope_sel = np.asarray(rope[idx], dtype=np.float64).reshape(idx.shape[0], ROPE)
    k_main = np.concatenate([lat_sel, rope_sel], axis=1)
    v_main = lat_sel
    swa = np.asarray(swa, dtype=np.float64)[:swa_len]
    keys = np.concatenate([k_main, swa], axis=0)            # [E, 576]
    vals = np.concatenate([v_main, swa[:, :LATENT]], axis=0)  # [E, 512]
    H = q.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, LATENT)), np.full(H, -np.inf)
    logits = scale * (q @ keys.T)                           # [H, E]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    z = p.sum(axis=1, keepdims=True)
    out = (p @ vals) / z
    lse = (m + np.log(z))[:, 0]
    return out, lse


def sparse_attn_decode_mq(q, latent, rope, topk, swa, swa_len, scale):
    """Attention of q_len consecutive decode queries of one sequence.

    q: [q_len, H, 576] (oldest query first); the other arguments as in
    ``sparse_attn_decode`` (one Top-K set, one window of ``swa_len`` valid
    rows).  One key set E = {valid Top-K entries} + {window rows} with a
    visibility mask: query i sees all main entries and window rows
    r < swa_len - (q_len - 1 - i).  Returns (out [q_len, H, 512], lse
    [q_len, H]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    ql, H = q.shape[0], q.shape[1]
    topk = np.asarray(topk, dtype=np.int64)
    idx = topk[topk >= 0]
    lat_sel = np.asarray(latent[idx], dtype=np.float64).reshape(idx.shape[0], LATENT)
    rope_sel = np.asarray(rope[idx], dtype=np.float64).reshape(idx.shape[0], ROPE)
    nm = idx.shape[0]
    swa = np.asarray(swa, dtype=np.float64)[:swa_len]
    keys = np.concatenate([np.concatenate([lat_sel, rope_sel], axis=1), swa], axis=0)   # [E, 576]
    vals = np.concatenate([lat_sel, swa[:, :LATENT]], axis=0)                           # [E, 512]
    E = keys.shape[0]
    # visible[i, e]: main entries always, window row r = e - nm while r < limit_i
    limit = np.maximum(0, swa_len - (ql - 1 - np.arange(ql)))
    r = np.arange(E) - nm
    visible = (r[None, :] < 0) | (r[None, :] < limit[:, None])                         # [q_len, E]
    out = np.zeros((ql, H, LATENT))
    lse = np.full((ql, H), -np.inf)
    if E == 0:
        return out, lse
    logits = scale * np.einsum("qhc,ec->qhe", q, keys)                                  # [q_len, H, E]
    logits = np.where(visible[:, None, :], logits, -np.inf)
    m = logits.max(axis=2, keepdims=True)                                               # [q_len, H, 1]
    has = np.isfinite(m)
    p = np.where(visible[:, None, :], np.exp(logits - np.where(has, m, 0.0)), 0.0)
    z = p.sum(axis=2, keepdims=True)
    out = np.where(has, np.einsum("qhe,ed->qhd", p, vals) / np.where(has, z, 1.0), 0.0)
    lse = np.where(has, m + np.log(np.where(has, z, 1.0)), -np.inf)[:, :, 0]
    return out, lse


def lse_merge(parts):
    """Merge (out, lse) partials of disjoint key sets into the joint result.

    o = sum_i exp(lse_i - L) o_i with L = ln sum_i exp(lse_i): the closed form
    of a softmax split over disjoint key sets.
    """
    outs = [np.asarray(o, dtype=np.float64) for o, _ in parts]
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])  # [P, H]
    mx = np.max(lses, axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    wts = np.exp(lses - safe)
    tot = wts.sum(axis=0)
    L = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    o = sum(w[:, None] * oi for w, oi in zip(wts, outs))
    o = np.where(tot[:, None] > 0, o / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
    return o, L

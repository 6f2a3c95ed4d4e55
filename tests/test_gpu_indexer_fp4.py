"""GPU parity of the FP4 indexer (FP4 query and keys) against the oracle.

The keys are written by the library's FP4 indexer-key quantize call (its
codes and scales must equal the oracle's quantization bit for bit); Full
mode (pool + Top-K) and Reindex mode must return exactly the oracle's ids
(``oracle.indexer_fp4``: the scores of the dequantized query and keys),
on ragged, paged, tied and wide-range inputs; and the scan's approximate
scores must lie within the bound delta the certified selection relies on.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2, synth
from oracle import codec as ocodec
from oracle import indexer as oix
from oracle import indexer_fp4 as ofp4
from tests.gpu_problem import fp4_keys_f64, make_fp4_problem, run_full, run_reindex
from tests.helpers import bf16_f64, ws_offsets

pytestmark = pytest.mark.gpu


def check_full(p, pool, plen, topk):
    pool, plen, topk = pool.cpu().numpy(), plen.cpu().numpy(), topk.cpu().numpy()
    for b in range(p.B):
        n = p.ctx_lens[b]
        r = ofp4.full_topk(p.idx_q_f64[b], p.w_raw[b].astype(np.float64), fp4_keys_f64(p, b), p.P, p.K)
        P_sel = len(r["pool"])
        assert plen[b] == P_sel, (b, plen[b], P_sel)
        np.testing.assert_array_equal(pool[b, :P_sel], r["pool"], err_msg=f"pool b={b} n={n}")
        assert np.all(pool[b, P_sel:] == -1)
        np.testing.assert_array_equal(topk[b], r["topk"], err_msg=f"topk b={b} n={n}")


def test_fp4_idx_key_write_matches_oracle():
    """Codes and scales of the two-plane buffer equal the oracle's, bit for bit,
    including rounding ties, zero and saturating groups, an odd row count and
    skipped destinations (negative, past the cache)."""
    rng = np.random.default_rng(21)
    n, rows = 1001, 1200
    x = (rng.standard_normal((n, 128)) * rng.lognormal(0, 1.0, 128)).astype(np.float32)
    x[0] = 0.0                                                   # a zero row: scale 0
    x[1, :16] = 1e6                                              # amax / 6 above 448: saturates
    lv = ocodec.E2M1_LEVELS
    x[2] = lv[rng.integers(0, 8, 128)] * np.where(rng.random(128) < 0.5, -1, 1)
    x[2, ::16] = 6.0                                             # exact grid: scale 1
    x[3] = np.repeat(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]), 16)   # E2M1 midpoints
    x[3, ::16] = 6.0
    bits = synth.to_bf16_bits(x)
    dst = rng.permutation(rows)[:n].astype(np.int64)
    dst[5] = -1
    dst[6] = rows + 7                                            # skipped (not below cache_rows)
    buf = torch.full((rows * 72,), 0xA5, dtype=torch.uint8, device="cuda")
    xd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    csa2.fp4_idx_k_quantize_scatter(xd, buf, rows, torch.from_numpy(dst).cuda())
    torch.cuda.synchronize()
    codes, scales = csa2.fp4_idx_k_planes(buf, rows)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    oc, os_ = ofp4.quantize(bf16_f64(bits))
    keep = (dst >= 0) & (dst < rows)
    np.testing.assert_array_equal(codes[dst[keep]], oc[keep])
    np.testing.assert_array_equal(scales[dst[keep]], os_[keep])
    untouched = np.setdiff1d(np.arange(rows), dst[keep])
    assert np.all(codes[untouched] == 0xA5) and np.all(scales[untouched] == 0xA5)
    # without dst_rows: row i
    buf2 = torch.zeros(n * 72, dtype=torch.uint8, device="cuda")
    csa2.fp4_idx_k_quantize_scatter(xd, buf2, n)
    torch.cuda.synchronize()
    c2, s2 = csa2.fp4_idx_k_planes(buf2, n)
    np.testing.assert_array_equal(c2.cpu().numpy(), oc)
    np.testing.assert_array_equal(s2.cpu().numpy(), os_)


@pytest.mark.parametrize("paged", [False, True])
def test_fp4_full_ragged(paged):
    p = make_fp4_problem([1, 7, 8, 9, 1000, 16383, 70001], paged=paged, seed=1)
    check_full(p, *run_full(p))


def test_fp4_full_small_pool_deep_selection():
    p = make_fp4_problem([50000, 33333], P=64, K=128, seed=2)
    check_full(p, *run_full(p))


def test_fp4_reindex():
    p = make_fp4_problem([20000, 9000, 17], seed=4, Hi=8)
    pool, plen, _ = run_full(p)
    rng = np.random.default_rng(9)
    raw = synth.to_bf16_bits(rng.standard_normal(p.idx_q_f64.shape).astype(np.float32))
    q64 = bf16_f64(raw)
    qd = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    w2 = rng.random(p.w_raw.shape).astype(np.float32)
    topk = run_reindex(p, pool, plen, qd, torch.from_numpy(w2).cuda()).cpu().numpy()
    pool_np = pool.cpu().numpy()
    for b in range(p.B):
        pl = pool_np[b][pool_np[b] >= 0]
        r = ofp4.reindex_topk(q64[b], w2[b].astype(np.float64), fp4_keys_f64(p, b), pl, p.K)
        np.testing.assert_array_equal(topk[b], r["topk"], err_msg=f"reindex b={b}")
    # Reindex with the Full layer's own query reproduces the Full Top-K
    pool, plen, tk_full = run_full(p)
    np.testing.assert_array_equal(run_reindex(p, pool, plen).cpu().numpy(), tk_full.cpu().numpy())


@pytest.mark.parametrize("paged", [False, True])
def test_fp4_reindex_paged_ragged(paged):
    p = make_fp4_problem([70001, 1000, 9], paged=paged, seed=14, P=256, K=512)
    pool, plen, tk_full = run_full(p)
    check_full(p, pool, plen, tk_full)
    np.testing.assert_array_equal(run_reindex(p, pool, plen).cpu().numpy(), tk_full.cpu().numpy())


def test_fp4_cluster_selection():
    """A context above one selection CTA (a cluster of 2), with a short one."""
    p = make_fp4_problem([200000, 5000], seed=32, P=512, K=256)
    check_full(p, *run_full(p))


def test_fp4_exact_ties():
    """Keys drawn from 3 distinct rows: huge groups of exactly equal scores."""
    p = make_fp4_problem([30000, 5000], kind="ties", P=256, K=512, seed=5)
    check_full(p, *run_full(p))


def test_fp4_wide_range_groups():
    """Groups at scales across the E4M3 range (terms of very different size)."""
    p = make_fp4_problem([40000, 777], kind="wide", P=512, K=512, seed=6)
    check_full(p, *run_full(p))


@pytest.mark.parametrize("kind", ["random", "wide"])
def test_fp4_error_bound_holds(kind):
    """|approximate score - exact score| <= delta for every position."""
    p = make_fp4_problem([60000, 12345], seed=7, kind=kind)
    run_full(p)
    off = ws_offsets(p.dims, p.B)
    ws = p.ws.cpu().numpy()
    pos = ws[off["pos_scores"]:off["pos_scores"] + p.B * p.dims.max_ctx * 4].view(np.float32)
    dl = ws[off["blk_delta"]:off["blk_delta"] + p.B * off["nb_max"] * 4].view(np.float32)
    worst = 0.0
    for b in range(p.B):
        n = p.ctx_lens[b]
        qc, qs = ofp4.quantize(p.idx_q_f64[b])
        kc, ks = ofp4.quantize(fp4_keys_f64(p, b))
        s = ofp4.scores(qc, qs, p.w_raw[b].astype(np.float64), kc, ks)
        v = pos[b * p.dims.max_ctx: b * p.dims.max_ctx + n].astype(np.float64)
        d = np.repeat(dl[b * off["nb_max"]: b * off["nb_max"] + (n + 7) // 8], 8)[:n].astype(np.float64)
        err = np.abs(v - s)
        assert np.all(err <= d), np.max(err / d)
        worst = max(worst, float(np.max(err / d)))
    print(f"{kind}: max observed |v - s| / delta = {worst:.3g}")


def test_fp4_short_contexts_and_padding():
    p = make_fp4_problem([3, 1, 40], seed=8)
    pool, plen, topk = run_full(p)
    assert plen.cpu().tolist() == [1, 1, 5]
    tk = topk.cpu().numpy()
    assert tk[0, :3].tolist() == [0, 1, 2] and np.all(tk[0, 3:] == -1)
    assert tk[1, :1].tolist() == [0] and np.all(tk[1, 1:] == -1)
    assert tk[2, :40].tolist() == list(range(40))


def test_fp4_flat_topk_equals_pool_topk():
    """The Full layer's Top-K from the pool equals the flat Top-K of all
    positions by the same FP4 scores (the oracle's property, on the GPU ids)."""
    p = make_fp4_problem([30011], seed=12, P=2048, K=512)
    _, _, topk = run_full(p)
    qc, qs = ofp4.quantize(p.idx_q_f64[0])
    kc, ks = ofp4.quantize(fp4_keys_f64(p, 0))
    s = ofp4.scores(qc, qs, p.w_raw[0].astype(np.float64), kc, ks)
    flat = np.sort(oix.top_order(s, p.K))
    np.testing.assert_array_equal(topk.cpu().numpy()[0], flat)


def test_fp4_early_inputs_flag_same_ids():
    p = make_fp4_problem([70001, 1000], seed=24)
    pool, plen, topk = run_full(p)
    check_full(p, pool, plen, topk)
    pool2, plen2, tk2 = torch.full_like(pool, -7), torch.zeros_like(plen), torch.full_like(topk, -7)
    csa2.indexer_full_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool2, plen2, tk2, p.ws,
                           flags=csa2.IDX_EARLY_INPUTS)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tk2.cpu().numpy(), topk.cpu().numpy())
    np.testing.assert_array_equal(pool2.cpu().numpy(), pool.cpu().numpy())
    tk_ri = run_reindex(p, pool, plen)
    tk_ri2 = torch.full_like(topk, -7)
    csa2.indexer_reindex_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool, plen, tk_ri2, p.ws,
                              flags=csa2.IDX_EARLY_INPUTS)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tk_ri2.cpu().numpy(), tk_ri.cpu().numpy())

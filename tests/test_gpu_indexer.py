"""GPU parity of the hierarchical indexer against the oracle (bit-exact ids).

Full mode (pool + Top-K) and Reindex mode through the C ABI, on ragged
contexts (partial last block, contexts shorter than the pool, single
positions), paged and contiguous caches, E4M3 and fp32 indexer keys, heavy
exact ties, and the error bound the certified selection relies on.
"""
import numpy as np
import pytest
import torch

from oracle import indexer as oix
from tests.gpu_problem import make_problem, oracle_keys, run_full, run_reindex
from tests.helpers import ws_offsets

pytestmark = pytest.mark.gpu


def check_full(p, pool, plen, topk):
    pool, plen, topk = pool.cpu().numpy(), plen.cpu().numpy(), topk.cpu().numpy()
    for b in range(p.B):
        n = p.ctx_lens[b]
        r = oix.full_topk(p.idx_q_f64[b], p.w_raw[b].astype(np.float64), oracle_keys(p, b),
                          p.P, p.K)
        P_sel = len(r["pool"])
        assert plen[b] == P_sel, (b, plen[b], P_sel)
        np.testing.assert_array_equal(pool[b, :P_sel], r["pool"], err_msg=f"pool b={b} n={n}")
        assert np.all(pool[b, P_sel:] == -1)
        np.testing.assert_array_equal(topk[b], r["topk"], err_msg=f"topk b={b} n={n}")
        print(f"b={b} n={n} margin_pool={r['margin_pool']:.3g} margin_topk={r['margin_topk']:.3g}")


def check_reindex(p, pool, topk, q64, w):
    pool, topk = pool.cpu().numpy(), topk.cpu().numpy()
    for b in range(p.B):
        pl = pool[b][pool[b] >= 0]
        r = oix.reindex_topk(q64[b], w[b].astype(np.float64), oracle_keys(p, b), pl, p.K)
        np.testing.assert_array_equal(topk[b], r["topk"], err_msg=f"reindex b={b}")


@pytest.mark.parametrize("paged", [False, True])
def test_full_fp8_ragged(paged):
    p = make_problem([1, 7, 8, 9, 1000, 16383, 70001], paged=paged, seed=1, with_kv=False)
    check_full(p, *run_full(p))


def test_full_small_pool_deep_selection():
    p = make_problem([50000, 33333], P=64, K=128, seed=2, with_kv=False)
    check_full(p, *run_full(p))


def test_full_fp32_keys():
    p = make_problem([4096, 3001, 64], Hi=4, Di=64, dtype="fp32", P=64, K=128, H=16, seed=3,
                     with_kv=False)
    check_full(p, *run_full(p))


@pytest.mark.parametrize("kind", ["ties", "wide"])
def test_fp32_keys_exact_ties(kind):
    """fp32 keys drawn from 3 rows, so that the bands hold whole tie groups and
    most positions are re-scored exactly: random rows (head dots whose products
    span 63-126 bits, the 128-bit accumulator) and rows whose products span more
    than 126 bits (the multi-limb accumulator); Full, then Reindex on the pool."""
    p = make_problem([3000, 517, 9], Hi=4, Di=64, dtype="fp32", P=64, K=128, H=16, seed=21,
                     kind=kind, with_kv=False)
    pool, plen, tk_full = run_full(p)
    check_full(p, pool, plen, tk_full)
    rng = np.random.default_rng(22)
    q2 = rng.standard_normal(p.idx_q_f64.shape).astype(np.float32)
    w2 = rng.random(p.w_raw.shape).astype(np.float32)
    topk = run_reindex(p, pool, plen, torch.from_numpy(q2).cuda(), torch.from_numpy(w2).cuda())
    check_reindex(p, pool, topk, q2.astype(np.float64), w2)


@pytest.mark.parametrize("dtype", ["fp8", "fp32"])
def test_reindex(dtype):
    kw = dict(Hi=4, Di=64, P=64, K=128) if dtype == "fp32" else {}
    p = make_problem([20000, 9000, 17], dtype=dtype, seed=4, with_kv=False, **kw)
    pool, plen, _ = run_full(p)
    rng = np.random.default_rng(9)
    q2 = rng.standard_normal(p.idx_q_f64.shape).astype(np.float32)
    from compressed_sparse_attention_fp4_gb300 import synth
    from tests.helpers import bf16_f64
    if dtype == "fp8":
        raw = synth.to_bf16_bits(q2)
        q64 = bf16_f64(raw)
        qd = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        q64 = q2.astype(np.float64)
        qd = torch.from_numpy(q2).cuda()
    w2 = rng.random(p.w_raw.shape).astype(np.float32)
    topk = run_reindex(p, pool, plen, qd, torch.from_numpy(w2).cuda())
    check_reindex(p, pool, topk, q64, w2)
    # Reindex with the Full layer's own query reproduces the Full Top-K
    pool, plen, tk_full = run_full(p)
    tk = run_reindex(p, pool, plen)
    np.testing.assert_array_equal(tk.cpu().numpy(), tk_full.cpu().numpy())


def test_full_exact_ties():
    """Keys drawn from 3 distinct rows: huge groups of exactly equal scores."""
    p = make_problem([30000, 5000], kind="ties", P=256, K=512, seed=5, with_kv=False)
    check_full(p, *run_full(p))


def test_full_ties_large_band():
    """Ties spanning more than the in-shared-memory sort capacity."""
    p = make_problem([130000], kind="ties", P=2048, K=512, seed=6, with_kv=False)
    check_full(p, *run_full(p))


def test_full_cluster_ties_topk_side_falls_back():
    """A context above one selection CTA (a cluster of 2) with massive ties:
    the Top-K side's superset of the K best blocks is wider than the pool
    buffer, so that side selects the pool itself first; a short context in the
    same call takes every block."""
    p = make_problem([200000, 3000], kind="ties", P=1024, K=256, seed=30, with_kv=False)
    check_full(p, *run_full(p))


@pytest.mark.parametrize("paged", [False, True])
def test_full_cluster_two_sides(paged):
    """A cluster of 2 per sequence and both selection sides (K <= P), on a
    contiguous and a paged cache."""
    p = make_problem([200000, 3000, 140001], paged=paged, P=1024, K=256, seed=34, with_kv=False)
    check_full(p, *run_full(p))


def test_full_cluster_pool_smaller_than_topk():
    """K > P on a cluster of 2: the Top-K must come from the pool's positions
    (no superset of the K best blocks), selected after the pool."""
    p = make_problem([140000, 900], P=64, K=128, seed=31, with_kv=False)
    check_full(p, *run_full(p))


def test_full_large_batch_selects_in_turn():
    """80 sequences: two selection sides per sequence would not fit one wave of
    one CTA per SM, so each sequence's CTA selects the pool and then its Top-K."""
    lens = [int(x) for x in np.random.default_rng(33).integers(1, 6000, size=80)]
    p = make_problem(lens, P=256, K=128, seed=33, with_kv=False)
    check_full(p, *run_full(p))


@pytest.mark.parametrize("Hi,P,K", [(1, 64, 8), (3, 4, 5), (5, 16, 16), (16, 2048, 2048)])
def test_full_and_reindex_odd_shapes(Hi, P, K):
    """Head counts that are not a multiple of the per-warp layouts, a pool
    smaller than K (the Top-K after the pool), K = P (the superset rarely
    fits: the pool itself) and K = P = 2048, on ragged contexts."""
    p = make_problem([1, 9, 300, 5000, 20001], Hi=Hi, P=P, K=K, seed=40 + Hi, with_kv=False)
    pool, plen, topk = run_full(p)
    check_full(p, pool, plen, topk)
    np.testing.assert_array_equal(run_reindex(p, pool, plen).cpu().numpy(), topk.cpu().numpy())


def test_error_bound_holds():
    """|approximate score - exact score| <= delta for every position."""
    p = make_problem([60000, 12345], seed=7, with_kv=False)
    run_full(p)
    off = ws_offsets(p.dims, p.B)
    ws = p.ws.cpu().numpy()
    pos = ws[off["pos_scores"]:off["pos_scores"] + p.B * p.dims.max_ctx * 4].view(np.float32)
    dl = ws[off["blk_delta"]:off["blk_delta"] + p.B * off["nb_max"] * 4].view(np.float32)
    worst = 0.0
    for b in range(p.B):
        n = p.ctx_lens[b]
        s = oix.scores(p.idx_q_f64[b], p.w_raw[b].astype(np.float64), oracle_keys(p, b))
        v = pos[b * p.dims.max_ctx: b * p.dims.max_ctx + n].astype(np.float64)
        d = np.repeat(dl[b * off["nb_max"]: b * off["nb_max"] + (n + 7) // 8], 8)[:n].astype(np.float64)
        err = np.abs(v - s)
        assert np.all(err <= d), np.max(err / d)
        worst = max(worst, float(np.max(err / d)))
    print(f"max observed |v - s| / delta = {worst:.3g}")


@pytest.mark.parametrize("kind", ["trunc", "cancel"])
def test_error_bound_adversarial(kind):
    """|v - s| <= delta when one product dominates every MMA step and the others
    are small same-sign values just below a power of two (the case that loses
    the most to truncation), and when the large products cancel exactly."""
    p = make_problem([4096, 1000], seed=11, kind=kind, with_kv=False)
    run_full(p)
    off = ws_offsets(p.dims, p.B)
    ws = p.ws.cpu().numpy()
    pos = ws[off["pos_scores"]:off["pos_scores"] + p.B * p.dims.max_ctx * 4].view(np.float32)
    dl = ws[off["blk_delta"]:off["blk_delta"] + p.B * off["nb_max"] * 4].view(np.float32)
    worst = 0.0
    for b in range(p.B):
        n = p.ctx_lens[b]
        s = oix.scores(p.idx_q_f64[b], p.w_raw[b].astype(np.float64), oracle_keys(p, b))
        v = pos[b * p.dims.max_ctx: b * p.dims.max_ctx + n].astype(np.float64)
        d = np.repeat(dl[b * off["nb_max"]: b * off["nb_max"] + (n + 7) // 8], 8)[:n].astype(np.float64)
        err = np.abs(v - s)
        assert np.all(err <= d), np.max(err / d)
        worst = max(worst, float(np.max(err / d)))
    print(f"{kind}: max observed |v - s| / delta = {worst:.3g}")


def test_pool_len_and_padding_short_context():
    p = make_problem([3, 0 + 1, 40], P=2048, K=512, seed=8, with_kv=False)
    pool, plen, topk = run_full(p)
    assert plen.cpu().tolist() == [1, 1, 5]
    tk = topk.cpu().numpy()
    assert tk[0, :3].tolist() == [0, 1, 2] and np.all(tk[0, 3:] == -1)
    assert tk[1, :1].tolist() == [0] and np.all(tk[1, 1:] == -1)
    assert tk[2, :40].tolist() == list(range(40))


def test_full_and_reindex_top1024():
    """Top-K above the pages' 512 (the attention then spans 9 chunks)."""
    p = make_problem([40000, 3000], K=1024, seed=18, with_kv=False)
    pool, plen, topk = run_full(p)
    check_full(p, pool, plen, topk)
    tk = run_reindex(p, pool, plen)
    np.testing.assert_array_equal(tk.cpu().numpy(), topk.cpu().numpy())


def test_eight_heads_odd_band():
    """8 indexer heads: a warp of the exact re-scoring holds (position, head)
    halves of an odd number of positions; Full and Reindex still match."""
    p = make_problem([20000, 9000, 17, 4099], Hi=8, P=512, K=512, seed=19, with_kv=False)
    pool, plen, topk = run_full(p)
    check_full(p, pool, plen, topk)
    rng = np.random.default_rng(29)
    from compressed_sparse_attention_fp4_gb300 import synth
    from tests.helpers import bf16_f64
    raw = synth.to_bf16_bits(rng.standard_normal(p.idx_q_f64.shape).astype(np.float32))
    qd = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    w2 = rng.random(p.w_raw.shape).astype(np.float32)
    tk = run_reindex(p, pool, plen, qd, torch.from_numpy(w2).cuda())
    check_reindex(p, pool, tk, bf16_f64(raw), w2)


@pytest.mark.parametrize("paged", [False, True])
def test_early_inputs_flag_same_ids(paged):
    """With IDX_EARLY_INPUTS the scans stream their first key tiles before the
    wait on the previous kernel; the ids are those of the plain calls (and of
    the oracle), right after a kernel that writes other memory."""
    from compressed_sparse_attention_fp4_gb300 import csa2
    p = make_problem([70001, 9000, 17], paged=paged, seed=23, with_kv=False)
    pool, plen, topk = run_full(p)
    check_full(p, pool, plen, topk)
    scratch = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    pool2 = torch.full_like(pool, -7)
    plen2 = torch.zeros_like(plen)
    tk2 = torch.full_like(topk, -7)
    scratch.fill_(1)                                    # the kernel just before: writes other memory
    csa2.indexer_full_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool2, plen2, tk2, p.ws,
                           flags=csa2.IDX_EARLY_INPUTS)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(pool2.cpu().numpy(), pool.cpu().numpy())
    np.testing.assert_array_equal(plen2.cpu().numpy(), plen.cpu().numpy())
    np.testing.assert_array_equal(tk2.cpu().numpy(), topk.cpu().numpy())
    tk_ri = run_reindex(p, pool, plen)
    tk_ri2 = torch.full_like(topk, -7)
    scratch.fill_(2)
    csa2.indexer_reindex_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool, plen, tk_ri2, p.ws,
                              flags=csa2.IDX_EARLY_INPUTS)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tk_ri2.cpu().numpy(), tk_ri.cpu().numpy())

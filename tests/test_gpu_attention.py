"""GPU parity of the sparse decode attention against the oracle.

Tolerance: normwise relative error max_i|o_i - r_i| / max_i|r_i| <= 2e-3 per
(sequence, head) and |lse - lse_ref| <= 2e-3, on fp32 outputs.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2
from oracle import attention as oatt
from tests.gpu_problem import make_problem
from tests.helpers import bf16_f64, normwise_rel, oracle_latent

pytestmark = pytest.mark.gpu
TOL = 2e-3


def random_topk(p, rng, frac_valid=0.9, sorted_=True):
    tk = np.full((p.B, p.K), -1, dtype=np.int32)
    for b, n in enumerate(p.ctx_lens):
        m = min(n, int(p.K * frac_valid))
        sel = np.sort(rng.choice(n, m, replace=False)) if m else np.zeros(0, np.int64)
        tk[b, :m] = sel
    return tk


def run_attn(p, topk_np, swa_len=None, mode=csa2.MODE_REUSE):
    out = torch.full((p.B, p.H, 512), np.nan, dtype=torch.float32, device="cuda")
    lse = torch.full((p.B, p.H), np.nan, dtype=torch.float32, device="cuda")
    tk = torch.from_numpy(topk_np).cuda()
    sl = p.swa_len if swa_len is None else torch.from_numpy(np.asarray(swa_len, np.int32)).cuda()
    csa2.csa2_sparse_attn_decode(p.dims, p.B, mode, p.q, p.codes, p.scales, p.rope, p.page_table,
                                 p.ctx, tk, p.swa, sl, 1.0 / np.sqrt(576.0), out, lse, p.ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def check(p, topk_np, out, lse, swa_len=None):
    sl = p.swa_len_np if swa_len is None else np.asarray(swa_len)
    worst = 0.0
    for b, n in enumerate(p.ctx_lens):
        lat = oracle_latent(p.latent_raw[b])
        rope = bf16_f64(p.rope_raw[b])
        ro, rl = oatt.sparse_attn_decode(bf16_f64(p.q_raw[b]), lat, rope, topk_np[b],
                                         bf16_f64(p.swa_raw[b]), int(sl[b]), 1.0 / np.sqrt(576.0))
        err = normwise_rel(out[b], ro)
        assert np.all(err <= TOL), (b, err.max())
        fin = np.isfinite(rl)
        assert np.array_equal(fin, np.isfinite(lse[b]))
        assert np.all(np.abs(lse[b][fin] - rl[fin]) <= TOL), (b, np.abs(lse[b][fin] - rl[fin]).max())
        assert np.all(out[b][~fin] == 0)
        worst = max(worst, float(err.max()) if err.size else 0.0)
    print(f"worst normwise rel err {worst:.3g}")


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("mode", [csa2.MODE_REUSE, csa2.MODE_FULL])
def test_attention_random(paged, mode):
    """Reuse mode gathers the entries before waiting for the previous kernel;
    Full (and Reindex) mode after it: both must give the oracle's result."""
    p = make_problem([100, 5000, 3000], paged=paged, seed=11)
    rng = np.random.default_rng(0)
    tk = random_topk(p, rng)
    sl = [0, 7, 128]
    out, lse = run_attn(p, tk, sl, mode=mode)
    check(p, tk, out, lse, sl)


def test_attention_sharp_queries():
    p = make_problem([4000, 2500], seed=12, q_sigma=1.0)
    tk = random_topk(p, np.random.default_rng(1), frac_valid=1.0)
    out, lse = run_attn(p, tk)
    check(p, tk, out, lse)


def test_attention_empty_and_single():
    p = make_problem([50, 60], seed=13)
    tk = np.full((2, p.K), -1, dtype=np.int32)
    tk[1, 0] = 17
    out, lse = run_attn(p, tk, [0, 0])
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    lat = oracle_latent(p.latent_raw[1])
    np.testing.assert_allclose(out[1], np.broadcast_to(lat[17], out[1].shape), rtol=0, atol=1e-6)


def test_attention_16_heads_small_topk():
    p = make_problem([4096], H=16, K=128, P=64, seed=14)
    tk = random_topk(p, np.random.default_rng(2), frac_valid=1.0)
    out, lse = run_attn(p, tk)
    check(p, tk, out, lse)


def test_attention_no_swa_window():
    p = make_problem([3000, 10], W=0, seed=15)
    tk = random_topk(p, np.random.default_rng(3))
    out, lse = run_attn(p, tk, [0, 0])
    check(p, tk, out, lse, [0, 0])


def test_attention_more_than_eight_chunks():
    """Top-1024 + SWA-128 = 9 chunks of 128: the one-CTA-per-chunk kernel and the
    combine kernel (above the cluster limit)."""
    p = make_problem([6000, 1500], K=1024, seed=16)
    tk = random_topk(p, np.random.default_rng(4))
    out, lse = run_attn(p, tk)
    check(p, tk, out, lse)


@pytest.mark.parametrize("mode", [csa2.MODE_REUSE, csa2.MODE_REINDEX])
def test_attention_window_not_on_chunk_boundary(mode):
    """Top-500: the SWA window starts inside a 128-entry chunk, so its rows are
    copied with the FP4 entries of that chunk, not loaded by TMA."""
    p = make_problem([5000, 300], K=500, seed=17)
    tk = random_topk(p, np.random.default_rng(5))
    sl = [128, 77]
    out, lse = run_attn(p, tk, sl, mode=mode)
    check(p, tk, out, lse, sl)


def test_attention_window_tma_short_window():
    """Top-384 (a multiple of 128) with a 100-row window: the window's chunk
    comes by TMA, only partly inside the window."""
    p = make_problem([5000, 60], K=384, W=100, seed=19)
    tk = random_topk(p, np.random.default_rng(6))
    sl = [100, 60]
    out, lse = run_attn(p, tk, sl)
    check(p, tk, out, lse, sl)


def test_attention_48_heads_eight_chunks():
    """48 heads (the second head group half full) and Top-896 + SWA-128 =
    8 chunks of 128: the largest cluster."""
    p = make_problem([9000, 1200], H=48, K=896, seed=20)
    tk = random_topk(p, np.random.default_rng(7))
    out, lse = run_attn(p, tk)
    check(p, tk, out, lse)

"""GPU parity of the multi-query decode attention against the oracle.

q_len = 2..4 queries per sequence (the newest tokens, oldest first) share
the Top-K set and the SWA window; query i sees the window rows below
swa_len - (q_len - 1 - i).  Checked against ``oracle.attention.
sparse_attn_decode_mq`` with the single-query tolerance: normwise relative
error <= 2e-3 per (sequence, query, head) and |lse - lse_ref| <= 2e-3.
q_len = 1 through the multi-query entry must equal the single-query entry
(lse bit for bit; the output up to the order in which the chunks' parts are
added, which is not fixed).
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2, synth
from oracle import attention as oatt
from tests.gpu_problem import make_problem
from tests.helpers import bf16_f64, normwise_rel, oracle_latent
from tests.test_gpu_attention import random_topk, run_attn

pytestmark = pytest.mark.gpu
TOL = 2e-3
SCALE = 1.0 / np.sqrt(576.0)


def mq_queries(p, ql, seed):
    rng = np.random.default_rng(seed)
    raw = synth.to_bf16_bits(rng.standard_normal((p.B, ql, p.H, 576)).astype(np.float32) / np.sqrt(576.0))
    return raw, torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)


def run_mq(p, ql, q_dev, topk_np, swa_len, mode=csa2.MODE_REUSE):
    out = torch.full((p.B, ql, p.H, 512), np.nan, dtype=torch.float32, device="cuda")
    lse = torch.full((p.B, ql, p.H), np.nan, dtype=torch.float32, device="cuda")
    tk = torch.from_numpy(topk_np).cuda()
    sl = torch.from_numpy(np.asarray(swa_len, np.int32)).cuda()
    csa2.csa2_sparse_attn_decode_mq(p.dims, p.B, ql, mode, q_dev, p.codes, p.scales, p.rope, p.page_table,
                                    p.ctx, tk, p.swa, sl, SCALE, out, lse, p.ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def check_mq(p, ql, q_raw, topk_np, out, lse, swa_len):
    worst = 0.0
    for b in range(p.B):
        lat = oracle_latent(p.latent_raw[b])
        rope = bf16_f64(p.rope_raw[b])
        ro, rl = oatt.sparse_attn_decode_mq(bf16_f64(q_raw[b]), lat, rope, topk_np[b], bf16_f64(p.swa_raw[b]),
                                            int(swa_len[b]), SCALE)
        for i in range(ql):
            err = normwise_rel(out[b, i], ro[i])
            assert np.all(err <= TOL), (b, i, err.max())
            fin = np.isfinite(rl[i])
            assert np.array_equal(fin, np.isfinite(lse[b, i])), (b, i)
            assert np.all(np.abs(lse[b, i][fin] - rl[i][fin]) <= TOL)
            assert np.all(out[b, i][~fin] == 0)
            worst = max(worst, float(err.max()))
    print(f"q_len={ql}: worst normwise rel err {worst:.3g}")


@pytest.mark.parametrize("ql", [2, 3, 4])
@pytest.mark.parametrize("mode", [csa2.MODE_REUSE, csa2.MODE_FULL])
def test_multi_query_random(ql, mode):
    p = make_problem([100, 5000, 3000], seed=21 + ql)
    tk = random_topk(p, np.random.default_rng(ql))
    sl = [3, 7, 128]                     # a window shorter than the draft block, a short and a full one
    q_raw, q_dev = mq_queries(p, ql, 100 + ql)
    out, lse = run_mq(p, ql, q_dev, tk, sl, mode)
    check_mq(p, ql, q_raw, tk, out, lse, sl)


@pytest.mark.parametrize("paged", [False, True])
def test_multi_query_paged_16_heads_ragged(paged):
    """16 heads (one partly filled head group), paged cache, a sequence whose
    first queries see no window row, Top-K and window on the pages' sizes."""
    p = make_problem([40, 9000, 700], H=16, paged=paged, seed=31)
    tk = random_topk(p, np.random.default_rng(5), frac_valid=0.7)
    sl = [2, 128, 64]
    q_raw, q_dev = mq_queries(p, 4, 131)
    out, lse = run_mq(p, 4, q_dev, tk, sl)
    check_mq(p, 4, q_raw, tk, out, lse, sl)


def test_multi_query_q1_equals_single_query():
    p = make_problem([100, 5000], seed=41)
    tk = random_topk(p, np.random.default_rng(6))
    sl = [9, 128]
    o1, l1 = run_attn(p, tk, sl)
    om, lm = run_mq(p, 1, p.q.view(p.B, 1, p.H, 576), tk, sl)
    np.testing.assert_allclose(om[:, 0], o1, rtol=1e-5, atol=1e-7)
    np.testing.assert_array_equal(lm[:, 0], l1)


def test_multi_query_limits():
    """q_len outside 1..4, and q_len > 1 with more than 8 chunks of entries,
    are refused on the host."""
    p = make_problem([100], seed=42, K=512)
    tk = torch.zeros((1, 512), dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 5, 64, 512), device="cuda")
    lse = torch.zeros((1, 5, 64), device="cuda")
    q = torch.zeros((1, 5, 64, 576), dtype=torch.bfloat16, device="cuda")
    for ql in (0, 5):
        with pytest.raises(csa2.Csa2Error) as e:
            csa2.csa2_sparse_attn_decode_mq(p.dims, 1, ql, csa2.MODE_FULL, q, p.codes, p.scales, p.rope, None,
                                            p.ctx, tk, p.swa, p.swa_len, SCALE, out, lse, p.ws)
        assert e.value.code == 2
    big = make_problem([100], seed=43, K=1024, with_kv=True)
    tkb = torch.zeros((1, 1024), dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_decode_mq(big.dims, 1, 2, csa2.MODE_FULL, q, big.codes, big.scales, big.rope, None,
                                        big.ctx, tkb, big.swa, big.swa_len, SCALE, out, lse, big.ws)
    assert e.value.code == 2


@pytest.mark.parametrize("mode", [csa2.MODE_REUSE, csa2.MODE_FULL])
def test_multi_query_large_batch_walks_chunks(mode):
    """32 sequences x 4 queries x 2 head groups (256 head groups): the library
    takes the chunk-walking kernel, each query with its own window limit."""
    rng = np.random.default_rng(41)
    lens = rng.integers(300, 3000, 32).tolist()
    lens[0] = 40                         # fewer positions than Top-K
    p = make_problem(lens, seed=41)
    tk = random_topk(p, rng)
    sl = rng.integers(0, 129, p.B).astype(np.int32)
    sl[:3] = [0, 2, 128]                 # no window; shorter than the draft block; full
    q_raw, q_dev = mq_queries(p, 4, 141)
    csa2.profile_enable(True)
    try:
        out, lse = run_mq(p, 4, q_dev, tk, sl, mode)
        rec = csa2.profile_read()
    finally:
        csa2.profile_enable(False)
    assert rec.get("attn_seq_tc", (0, 0.0))[0] == 1, rec
    check_mq(p, 4, q_raw, tk, out, lse, sl)

"""Context-parallel merge on CPU: two and three gloo ranks, one sequence.

Each rank takes a contiguous, block-aligned shard of the context and computes
its local results with the oracle (local Top-P blocks with their exact block
scores; after the pool merge, the local Top-K of the pool positions in its
shard by the Full scores and by the Reindex scores; the
attention partial over its selected entries, the SWA window on the last
rank); the library's merge (`cp.gather_selection`, `cp.gather_attention`:
one all-gather each) must reproduce the single-process oracle: pool and
index sets exactly, attention to float64 rounding.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

N_CTX, P, K, HI, DI, H, W = 20003, 64, 128, 4, 64, 8, 16


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem(seed=3):
    rng = np.random.default_rng(seed)
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    keys = f32(rng.standard_normal((N_CTX, DI)) * rng.lognormal(0, 0.5, DI))
    q, w = f32(rng.standard_normal((HI, DI))), f32(rng.random(HI))
    q2, w2 = f32(rng.standard_normal((HI, DI))), f32(rng.random(HI))
    latent = rng.standard_normal((N_CTX, 512))
    rope = rng.standard_normal((N_CTX, 64))
    aq = rng.standard_normal((H, 576)) * 0.2
    swa = rng.standard_normal((W, 576))
    return keys, q, w, q2, w2, latent, rope, aq, swa


def _local_topk(ids, scores, k):
    """This shard's k best (score desc, id asc) as padded id / score arrays."""
    from oracle import indexer as oix
    sel = oix.top_order(scores, min(k, len(ids)))
    out_i = np.full(k, -1, np.int64)
    out_s = np.zeros(k)
    out_i[:len(sel)] = np.asarray(ids)[sel]
    out_s[:len(sel)] = np.asarray(scores)[sel]
    return torch.from_numpy(out_i), torch.from_numpy(out_s)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from compressed_sparse_attention_fp4_gb300 import cp
    from oracle import attention as oatt
    from oracle import indexer as oix
    keys, q, w, q2, w2, latent, rope, aq, swa = _problem()
    lo, hi = cp.shard_bounds(N_CTX, world, rank)
    # ---- Full layer on the shard: local pool blocks and local flat Top-K -----
    s = oix.scores(q, w, keys[lo:hi])
    bs = oix.block_scores(s)
    b_ids = np.arange(lo // 8, lo // 8 + len(bs))
    pool = cp.gather_selection(*_local_topk(b_ids, bs, P), P)
    # the Full layer's Top-K: the pool positions of this shard, by their Full scores
    pos = oix.pool_positions(pool[pool >= 0].numpy(), N_CTX)
    mine = pos[(pos >= lo) & (pos < hi)]
    topk = cp.gather_selection(*_local_topk(mine, s[mine - lo], K), K)
    # ---- Reindex layer: the same pool positions, the Reindex query ----------
    s2 = oix.scores(q2, w2, keys[mine]) if len(mine) else np.zeros(0)
    topk_ri = cp.gather_selection(*_local_topk(mine, s2, K), K)
    # ---- attention over this shard's selected entries (+ SWA on the last) ---
    t = topk.numpy()
    t_loc = np.where((t >= lo) & (t < hi), t, -1)
    swl = W if rank == world - 1 else 0
    o, l = oatt.sparse_attn_decode(aq, latent, rope, t_loc, swa, swl, 1 / 24.0)
    o_m, l_m = cp.gather_attention(torch.from_numpy(o), torch.from_numpy(l))
    out[rank] = (pool.numpy(), topk.numpy(), topk_ri.numpy(), o_m.numpy(), l_m.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_merge_equals_single_process(world):
    from oracle import attention as oatt
    from oracle import indexer as oix
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    keys, q, w, q2, w2, latent, rope, aq, swa = _problem()
    f = oix.full_topk(q, w, keys, P, K)
    r = oix.reindex_topk(q2, w2, keys, f["pool"], K)
    ro, rl = oatt.sparse_attn_decode(aq, latent, rope, f["topk"], swa, W, 1 / 24.0)
    for rank in range(world):
        pool, topk, topk_ri, o, l = out[rank]
        np.testing.assert_array_equal(pool[:len(f["pool"])], f["pool"])
        assert np.all(pool[len(f["pool"]):] == -1)
        np.testing.assert_array_equal(topk, f["topk"])
        np.testing.assert_array_equal(topk_ri, r["topk"])
        np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l, rl, rtol=1e-12, atol=1e-12)


def test_merge_rules_edge_cases():
    """Ties across ranks go to the lower id; empty partials merge to nothing;
    an all-empty union gives o = 0 and lse = -inf."""
    from compressed_sparse_attention_fp4_gb300 import cp
    ids = torch.tensor([[7, 3, -1], [2, 9, 5]])
    sc = torch.tensor([[1.0, 2.0, 0.0], [2.0, 1.0, 1.0]], dtype=torch.float64)
    # order: (2.0, 2), (2.0, 3), (1.0, 5), (1.0, 7), (1.0, 9)
    assert cp.merge_selection(ids, sc, 4).tolist() == [2, 3, 5, 7]
    assert cp.merge_selection(ids, sc, 7).tolist() == [2, 3, 5, 7, 9, -1, -1]
    o = torch.tensor([[[1.0, 2.0]], [[0.0, 0.0]]], dtype=torch.float64)
    lse = torch.tensor([[0.5], [float("-inf")]], dtype=torch.float64)
    om, lm = cp.merge_attention(o, lse)
    assert om.tolist() == [[1.0, 2.0]] and lm.tolist() == [0.5]
    om, lm = cp.merge_attention(torch.zeros(2, 1, 2, dtype=torch.float64),
                                torch.full((2, 1), float("-inf"), dtype=torch.float64))
    assert om.tolist() == [[0.0, 0.0]] and lm.tolist() == [float("-inf")]
    assert cp.shard_bounds(20003, 2, 0) == (0, 10000) and cp.shard_bounds(20003, 2, 1) == (10000, 20003)

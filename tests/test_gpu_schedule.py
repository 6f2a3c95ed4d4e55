"""End-to-end parity of whole decode steps on the library's workloads.

Each workload runs its layer schedule (Full / Reindex / Reuse) through the C
ABI exactly as the benchmark does (optionally as a CUDA graph); indices must
equal the oracle's bit for bit and attention outputs must be within 2e-3.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import synth, workload
from compressed_sparse_attention_fp4_gb300.step import GraphedStep, run_step
from tests import oracle_jobs
from tests.helpers import normwise_rel, ws_offsets

pytestmark = pytest.mark.gpu
TOL = 2e-3


def check_bound(wl, sb, b, scores):
    """|v_t - s_t| <= delta for every position of sequence b: the Full scan's
    approximate scores and block bounds, read back from the workspace, against
    the oracle's exact scores (the certified selection rests on this)."""
    off = ws_offsets(sb.dims, sb.batch)
    mc, nbm = sb.dims.max_ctx, off["nb_max"]
    n = wl.ctx_lens[b]
    pos = sb.ws[off["pos_scores"] + 4 * b * mc: off["pos_scores"] + 4 * (b * mc + n)]
    dl = sb.ws[off["blk_delta"] + 4 * b * nbm: off["blk_delta"] + 4 * (b * nbm + (n + 7) // 8)]
    v = pos.cpu().numpy().view(np.float32).astype(np.float64)
    d = np.repeat(dl.cpu().numpy().view(np.float32), 8)[:n].astype(np.float64)
    err = np.abs(v - scores)
    ratio = float(np.max(err / d))
    assert np.all(err <= d), (b, ratio)
    return ratio


def check_step(wl, sb, seqs, bound=False):
    """Every layer of every listed sequence against the oracle: pool and index
    sets bit-exact, attention within 2e-3; with `bound`, also the Full scan's
    error bound at every position."""
    out, lse = sb.out.cpu().numpy(), sb.lse.cpu().numpy()
    topk = sb.topk.cpu().numpy()
    pool, plen = sb.pool.cpu().numpy(), sb.pool_len.cpu().numpy()
    seqs = list(seqs)
    refs = oracle_jobs.oracle_sequences(wl.name, seqs, want_scores=bound)
    worst, worst_ratio = 0.0, 0.0
    for b in seqs:
        ref = refs[b]
        for l, r in enumerate(ref):
            if r["mode"] in ("F", "Ri"):
                np.testing.assert_array_equal(topk[l, b], r["topk"], err_msg=f"layer {l} b {b}")
            if r["mode"] == "F":
                P = len(r["pool"])
                assert plen[b] == P
                np.testing.assert_array_equal(pool[b, :P], r["pool"])
                print(f"b={b} margins pool={r['margin_pool']:.3g} topk={r['margin_topk']:.3g}")
                if bound:
                    worst_ratio = max(worst_ratio, check_bound(wl, sb, b, r["scores"]))
            err = normwise_rel(out[l, b], r["out"])
            assert np.all(err <= TOL), (l, b, err.max())
            assert np.all(np.abs(lse[l, b] - r["lse"]) <= TOL)
            worst = max(worst, float(err.max()))
        if wl.planted:
            pl = synth.planted_positions(wl, b)
            in_pool = np.isin(pl // 8, pool[b, :plen[b]]).sum()
            f_layer = [l for l, m in enumerate(wl.schedule) if m == "F"][0]
            in_top = np.isin(pl, topk[f_layer, b]).sum()
            print(f"planted recall b={b}: pool {in_pool}/{len(pl)}, Full Top-K {in_top}/{len(pl)}")
    print(f"{wl.name}: {len(seqs)} sequences; worst normwise attention error {worst:.3g}"
          + (f"; worst |v - s| / delta {worst_ratio:.3g}" if bound else ""))


def test_tiny_workload_eager():
    wl = synth.workload("tiny")
    sb = workload.build(wl)
    run_step(sb)
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch))


def test_tiny_workload_graph_replay():
    wl = synth.workload("tiny")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    sb.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch))


def test_128k_workload():
    """All 8 sequences, every layer; the scan's bound checked at every position."""
    wl = synth.workload("128k")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch), bound=True)


def test_128k_fp4_keys_workload():
    """FP4 indexer keys (the library writes every key, the newest token's in
    the step, before the Full layer's scan): all 8 sequences, every layer; the
    FP4 scan's bound at every position."""
    wl = synth.workload("128k-fp4")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch), bound=True)


def test_128k_four_query_tokens_workload():
    """Four query tokens per sequence and layer (one Top-K set, each query's
    own window limit): all 8 sequences, every layer and query."""
    wl = synth.workload("128k-q4")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch))


def test_1m_workload():
    """The 1,048,576-position sequence, every layer; the bound at every position."""
    wl = synth.workload("1m")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch), bound=True)


def test_1m_fp4_keys_workload():
    """The 1,048,576-position sequence with FP4 indexer keys (the library's FP4
    key write, scan and selection), every layer; the FP4 scan's bound at every
    position."""
    wl = synth.workload("1m-fp4")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch), bound=True)


def test_mix_workload_every_sequence():
    """All 64 serving-mix sequences (paged, N in [8K, 256K]), every layer."""
    wl = synth.workload("mix")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch), bound=True)

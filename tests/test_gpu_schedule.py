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
from oracle import attention as oatt
from oracle import indexer as oix
from tests.helpers import bf16_f64, idxk_f64, normwise_rel, oracle_latent

pytestmark = pytest.mark.gpu
TOL = 2e-3


def oracle_sequence(wl, b, kv):
    """The oracle's index sets and attention outputs for every layer of seq b."""
    n = wl.ctx_lens[b]
    keys = idxk_f64(kv["idx_k"], wl.idx_k_dtype)
    layers = [synth.layer_inputs(wl, b, l) for l in range(len(wl.schedule))]
    conv_q = (lambda x: bf16_f64(x)) if wl.idx_k_dtype == "fp8" else (lambda x: x.astype(np.float64))
    res, pool, cur = [], None, None
    for l, mode in enumerate(wl.schedule):
        li = layers[l]
        rec = {"mode": mode}
        if mode == "F":
            r = oix.full_topk(conv_q(li["idx_q"]), li["idx_w"].astype(np.float64), keys,
                              wl.pool_blocks, wl.topk)
            pool, cur = r["pool"], r["topk"]
            rec.update(pool=pool, margin_pool=r["margin_pool"], margin_topk=r["margin_topk"])
        elif mode == "Ri":
            r = oix.reindex_topk(conv_q(li["idx_q"]), li["idx_w"].astype(np.float64), keys, pool,
                                 wl.topk)
            cur = r["topk"]
            rec.update(margin_topk=r["margin_topk"])
        rec["topk"] = cur
        res.append(rec)
    # dequantize (oracle codec) only the rows attention reads
    need = np.unique(np.concatenate([r["topk"][r["topk"] >= 0] for r in res]))
    lat = np.zeros((n, 512))
    lat[need] = oracle_latent(kv["latent"][need])
    rope = bf16_f64(kv["rope"])
    for l, r in enumerate(res):
        li = layers[l]
        r["out"], r["lse"] = oatt.sparse_attn_decode(bf16_f64(li["q"]), lat, rope, r["topk"],
                                                     bf16_f64(li["swa"]), li["swa_len"], wl.scale)
    return res


def check_step(wl, sb, seqs):
    out, lse = sb.out.cpu().numpy(), sb.lse.cpu().numpy()
    topk = sb.topk.cpu().numpy()
    pool, plen = sb.pool.cpu().numpy(), sb.pool_len.cpu().numpy()
    worst = 0.0
    for b in seqs:
        kv = synth.sequence_kv_parallel(wl, b)
        ref = oracle_sequence(wl, b, kv)
        cur_l = None
        for l, r in enumerate(ref):
            if r["mode"] in ("F", "Ri"):
                cur_l = l
                np.testing.assert_array_equal(topk[l, b], r["topk"], err_msg=f"layer {l} b {b}")
            if r["mode"] == "F":
                P = len(r["pool"])
                assert plen[b] == P
                np.testing.assert_array_equal(pool[b, :P], r["pool"])
                print(f"b={b} margins pool={r['margin_pool']:.3g} topk={r['margin_topk']:.3g}")
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
    print(f"{wl.name}: worst normwise attention error {worst:.3g}")


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
    wl = synth.workload("128k")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch))


def test_1m_workload():
    wl = synth.workload("1m")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    check_step(wl, sb, range(wl.batch))


def test_mix_workload_sampled():
    wl = synth.workload("mix")
    sb = workload.build(wl)
    g = GraphedStep(sb)
    g.replay()
    torch.cuda.synchronize()
    lens = np.array(wl.ctx_lens)
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 17]
    check_step(wl, sb, seqs)

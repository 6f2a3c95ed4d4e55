"""CPU oracle runs of whole workloads, spread over a process pool.

Test plumbing: each job regenerates its own seeded inputs (``synth``) and runs
the oracle on them; the parent compares the results with the GPU's.  The pool
uses the ``spawn`` start method (never ``fork`` after the GPU is in use), and
its workers run single-threaded BLAS so that the pool's processes do not
oversubscribe the host cores.
"""
from __future__ import annotations

import contextlib
import hashlib
import multiprocessing as mp
import os

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


@contextlib.contextmanager
def spawn_pool(jobs: int):
    """A spawn-context pool of min(jobs, host cores) single-threaded workers."""
    n = max(1, min(jobs, len(os.sched_getaffinity(0))))
    saved = {k: os.environ.get(k) for k in _THREAD_VARS}
    for k in _THREAD_VARS:
        os.environ[k] = "1"            # read by the workers' BLAS at start-up
    try:
        pool = mp.get_context("spawn").Pool(n)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield pool
    finally:
        pool.close()
        pool.join()


def oracle_sequence(wl_name: str, b: int, want_scores: bool = False):
    """Index sets and attention outputs of every layer of sequence b of a
    named workload, computed by the oracle from the seeded inputs."""
    from compressed_sparse_attention_fp4_gb300 import synth
    from oracle import attention as oatt
    from oracle import indexer as oix
    from tests.helpers import bf16_f64, idxk_f64, oracle_latent

    wl = synth.workload(wl_name)
    kv = synth.sequence_kv(wl, b)
    n = wl.ctx_lens[b]
    if wl.idx_k_dtype == "fp4":
        # FP4 indexer: the oracle quantizes the bf16 query and keys itself
        from oracle import indexer_fp4 as ix
        keys = bf16_f64(kv["idx_k"])
    else:
        ix = oix
        keys = idxk_f64(kv["idx_k"], wl.idx_k_dtype)
    layers = [synth.layer_inputs(wl, b, l) for l in range(len(wl.schedule))]
    conv_q = (lambda x: bf16_f64(x)) if wl.idx_k_dtype in ("fp8", "fp4") else (lambda x: x.astype(np.float64))
    res, pool, cur = [], None, None
    for l, mode in enumerate(wl.schedule):
        li = layers[l]
        rec = {"mode": mode}
        if mode == "F":
            r = ix.full_topk(conv_q(li["idx_q"]), li["idx_w"].astype(np.float64), keys,
                             wl.pool_blocks, wl.topk)
            pool, cur = r["pool"], r["topk"]
            rec.update(pool=pool, margin_pool=r["margin_pool"], margin_topk=r["margin_topk"])
            if want_scores:
                rec["scores"] = r["scores"]
        elif mode == "Ri":
            r = ix.reindex_topk(conv_q(li["idx_q"]), li["idx_w"].astype(np.float64), keys, pool,
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
    attend = oatt.sparse_attn_decode if wl.q_len == 1 else oatt.sparse_attn_decode_mq
    for l, r in enumerate(res):
        li = layers[l]
        r["out"], r["lse"] = attend(bf16_f64(li["q"]), lat, rope, r["topk"], bf16_f64(li["swa"]),
                                    li["swa_len"], wl.scale)
    return res


def _oracle_sequence_star(args):
    return oracle_sequence(*args)


def oracle_sequences(wl_name: str, seqs, want_scores: bool = False) -> dict:
    """{b: oracle_sequence(wl_name, b)} for every b in seqs, in parallel."""
    seqs = list(seqs)
    with spawn_pool(len(seqs)) as pool:
        out = pool.map(_oracle_sequence_star, [(wl_name, b, want_scores) for b in seqs], chunksize=1)
    return dict(zip(seqs, out))


def codec_chunk(n: int, lo: int, hi: int):
    """Oracle FP4 write of rows [lo, hi) of the codec slab: (codes, scales,
    sha256 of the oracle's dequantized rows as bf16 bit patterns)."""
    from compressed_sparse_attention_fp4_gb300 import synth
    from oracle import codec as ocodec
    from tests.helpers import bf16_f64

    x = synth.codec_slab(n=n, lo=lo, hi=hi)
    codes, scales = ocodec.quantize_rows(bf16_f64(x))
    y = ocodec.dequantize_rows(codes, scales)
    # every dequantized value is exact in bf16: its fp32 bits' upper half
    bits = (np.ascontiguousarray(y, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64), y)
    return codes, scales, hashlib.sha256(bits.tobytes()).hexdigest()


def _codec_chunk_star(args):
    return codec_chunk(*args)


def oracle_codec_slab(n: int, chunk: int = 1 << 16):
    """Oracle codes, scales and dequantized-row hashes of the whole slab, by chunks."""
    spans = [(n, a, min(n, a + chunk)) for a in range(0, n, chunk)]
    with spawn_pool(len(spans)) as pool:
        return spans, pool.map(_codec_chunk_star, spans, chunksize=1)

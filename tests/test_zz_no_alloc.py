"""The allocation-free decode attention call, through the C ABI.

Some callers may not allocate GPU memory on their hot path at all (a plugin
running inside another engine's execution step, a serving loop whose memory
budget is fixed before it starts), so they cannot hand the library a
workspace.  For them the call keeps its scratch in a fixed array inside the
library.  Its results must agree with the workspace call's and with the CPU
oracle on the same inputs (same 2e-3 normwise tolerance as the other
attention tests), on two calls in a row that reuse the array, and the calls
must not change the device's memory use.

The Top-2048 + SWA-128 cases span 17 chunks of 128 entries, above the
cluster limit: there the per-chunk partial outputs and (max, sum) pairs live
in the fixed array and the combine kernel reads them back -- the path the
array exists for.  The Top-512 cases (5 chunks) merge inside one cluster and
touch only the array's error word.

This file is collected last so that a run stopping at the first failure has
run every other test first; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2, synth
from oracle import attention as oatt
from tests.gpu_problem import make_problem
from tests.helpers import bf16_f64, normwise_rel, oracle_latent

pytestmark = pytest.mark.gpu
TOL = 2e-3
SCALE = 1.0 / np.sqrt(576.0)


def _topk(p, rng):
    tk = np.full((p.B, p.K), -1, dtype=np.int32)
    for b, n in enumerate(p.ctx_lens):
        m = min(n, p.K - 3)
        tk[b, :m] = np.sort(rng.choice(n, m, replace=False))
    return tk


def _with_workspace(p, tk, q):
    out = torch.full((p.B, p.H, 512), float("nan"), device="cuda")
    lse = torch.full((p.B, p.H), float("nan"), device="cuda")
    csa2.csa2_sparse_attn_decode(p.dims, p.B, csa2.MODE_REUSE, q, p.codes, p.scales, p.rope,
                                 p.page_table, p.ctx, torch.from_numpy(tk).cuda(), p.swa, p.swa_len,
                                 SCALE, out, lse, p.ws)
    return out, lse


def _no_alloc(p, tk_dev, q, err, out, lse):
    csa2.csa2_sparse_attn_decode_noalloc(p.dims, p.B, csa2.MODE_REUSE, q, p.codes, p.scales,
                                         p.rope, p.page_table, p.ctx, tk_dev, p.swa, p.swa_len,
                                         SCALE, out, lse, err)


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    assert np.all(normwise_rel(oa, ob) <= TOL)
    assert np.all(np.abs(la - lb) <= TOL)


def _oracle(p, tk, q_bits):
    outs, lses = [], []
    for b in range(p.B):
        ro, rl = oatt.sparse_attn_decode(bf16_f64(q_bits[b]), oracle_latent(p.latent_raw[b]),
                                         bf16_f64(p.rope_raw[b]), tk[b], bf16_f64(p.swa_raw[b]),
                                         int(p.swa_len_np[b]), SCALE)
        outs.append(ro)
        lses.append(rl)
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("K,paged", [(2048, False), (2048, True), (512, False), (512, True)])
def test_no_alloc_matches_workspace_call_and_oracle_twice(K, paged):
    p = make_problem([5000, 2300] if K == 2048 else [5000, 700, 64], K=K, paged=paged,
                     seed=31 + K + int(paged))
    rng = np.random.default_rng(5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tk1, tk2 = _topk(p, rng), _topk(p, rng)
    q2_bits = synth.to_bf16_bits((bf16_f64(p.q_raw) * 1.5).astype(np.float32))   # another query
    q2 = torch.from_numpy(q2_bits.view(np.int16)).cuda().view(torch.bfloat16)
    bufs = [(torch.full((p.B, p.H, 512), float("nan"), device="cuda"),
             torch.full((p.B, p.H), float("nan"), device="cuda"),
             torch.from_numpy(t).cuda()) for t in (tk1, tk2)]
    # one call sets up the array's device address; afterwards, no call may
    # change what the device has allocated
    _no_alloc(p, bufs[0][2], p.q, err, bufs[0][0], bufs[0][1])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for (out, lse, tk_dev), q in zip(bufs, (p.q, q2)):
        _no_alloc(p, tk_dev, q, err, out, lse)             # two calls in a row, one array
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_reserved() == reserved0
    got = [(o.cpu().numpy(), l.cpu().numpy()) for o, l, _ in bufs]
    want = [tuple(t.cpu().numpy() for t in _with_workspace(p, tk, q))
            for tk, q in ((tk1, p.q), (tk2, q2))]
    torch.cuda.synchronize()
    for g, w, tk, qb in zip(got, want, (tk1, tk2), (p.q_raw, q2_bits)):
        _close(g, w)
        _close(g, _oracle(p, tk, qb))
    assert int(err.item()) == 0


def test_no_alloc_large_batch_walks_chunks():
    """64 sequences x 2 head groups: the allocation-free call takes the
    chunk-walking kernel (no scratch but the error word) and allocates
    nothing; results as the workspace call's and the oracle's."""
    rng = np.random.default_rng(37)
    p = make_problem(rng.integers(200, 2500, 64).tolist(), seed=37)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tk = _topk(p, rng)
    tk_dev = torch.from_numpy(tk).cuda()
    out = torch.full((p.B, p.H, 512), float("nan"), device="cuda")
    lse = torch.full((p.B, p.H), float("nan"), device="cuda")
    csa2.profile_enable(True)
    try:
        _no_alloc(p, tk_dev, p.q, err, out, lse)
        rec = csa2.profile_read()
    finally:
        csa2.profile_enable(False)
    assert rec.get("attn_seq_tc", (0, 0.0))[0] == 1, rec
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    out.fill_(float("nan"))
    _no_alloc(p, tk_dev, p.q, err, out, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_reserved() == reserved0
    got = (out.cpu().numpy(), lse.cpu().numpy())
    _close(got, tuple(t.cpu().numpy() for t in _with_workspace(p, tk, p.q)))
    _close(got, _oracle(p, tk, p.q_raw))
    assert int(err.item()) == 0


def test_no_alloc_reports_device_errors_and_limit():
    p = make_problem([100], seed=32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tk = torch.full((1, p.K), -1, dtype=torch.int32, device="cuda")
    tk[0, 0] = 100                      # == ctx_len: skipped and reported
    out = torch.empty((1, p.H, 512), device="cuda")
    lse = torch.empty((1, p.H), device="cuda")
    _no_alloc(p, tk, p.q, err, out, lse)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x04
    # the partial path (Top-2048 + SWA-128 = 17 chunks) at batch 64 needs
    # more than the fixed array: rejected on the host, nothing launched
    big = csa2.Dims(**{**p.dims.__dict__, "topk": 2048})
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_decode_noalloc(big, 64, csa2.MODE_REUSE, p.q, p.codes, p.scales,
                                             p.rope, None, p.ctx, tk, p.swa, p.swa_len, SCALE,
                                             p.q, p.q, None)
    assert e.value.code == 3
    # a paged cache whose page table spans more than the largest context is
    # rejected exactly as the workspace call rejects it
    paged = csa2.Dims(**{**p.dims.__dict__, "max_pages": (1 << 20) // 64 + 1, "num_pages": 4})
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_decode_noalloc(paged, 1, csa2.MODE_REUSE, p.q, p.codes, p.scales,
                                             p.rope, p.ctx, p.ctx, tk, p.swa, p.swa_len, SCALE,
                                             out, lse, None)
    assert e.value.code == 2

"""The kernels write only inside their output buffers.

Every output is a slice of a larger buffer whose guard regions on both sides
hold a sentinel bit pattern; after the calls the guards are unchanged, bit
for bit (the canary check of the design's auxiliary subsystems).
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2
from tests.gpu_problem import make_problem

pytestmark = pytest.mark.gpu

GUARD = 4096                       # elements on each side (16 KB of int32 / fp32)
SENTINEL = 0x5A5AA5A5


def guarded(shape, dtype):
    """(view, whole buffer): the view lies between two sentinel-filled guards."""
    n = int(np.prod(shape))
    whole = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.int32, device="cuda")
    view = whole[GUARD:GUARD + n].view(dtype).view(shape)
    return view, whole


def guards_intact(whole):
    g = torch.cat([whole[:GUARD], whole[-GUARD:]])
    return bool(torch.all(g == SENTINEL).item())


@pytest.mark.parametrize("paged", [False, True])
def test_outputs_stay_inside_their_buffers(paged):
    p = make_problem([3000, 1500, 70001], seed=31, paged=paged)
    pool, pool_w = guarded((p.B, p.P), torch.int32)
    plen, plen_w = guarded((p.B,), torch.int32)
    tk, tk_w = guarded((p.B, p.K), torch.int32)
    csa2.indexer_full_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool, plen, tk, p.ws)
    tk2, tk2_w = guarded((p.B, p.K), torch.int32)
    csa2.indexer_reindex_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool, plen, tk2,
                              p.ws)
    out, out_w = guarded((p.B, p.H, 512), torch.float32)
    lse, lse_w = guarded((p.B, p.H), torch.float32)
    csa2.csa2_sparse_attn_decode(p.dims, p.B, csa2.MODE_FULL, p.q, p.codes, p.scales, p.rope,
                                 p.page_table, p.ctx, tk, p.swa, p.swa_len, 1.0 / np.sqrt(576.0), out,
                                 lse, p.ws)
    torch.cuda.synchronize()
    assert csa2.get_device_status(p.ws) == 0
    for name, whole in (("pool", pool_w), ("pool_len", plen_w), ("topk", tk_w), ("reindex topk", tk2_w),
                        ("out", out_w), ("lse", lse_w)):
        assert guards_intact(whole), name
    # the outputs themselves were written (no sentinel left inside)
    assert bool(torch.all(tk.view(torch.int32) != SENTINEL).item())
    assert bool(torch.all(out.view(torch.int32) != SENTINEL).item())
    assert bool(torch.all(lse.view(torch.int32) != SENTINEL).item())

"""Device-side error reporting: bad indices, page ids, lengths and windows
set bits in the workspace error word and are skipped -- no fault, no trap.

Every case feeds an input the kernels' own bounds checks turn into an error
bit; none of them makes an out-of-range access.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2
from tests.gpu_problem import make_problem, run_full

pytestmark = pytest.mark.gpu

CTX, PAGE, TOPK, SWA, TIMEOUT = 0x01, 0x02, 0x04, 0x08, 0x20


def attn(p, tk, sl):
    out = torch.zeros((p.B, p.H, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((p.B, p.H), dtype=torch.float32, device="cuda")
    csa2.csa2_sparse_attn_decode(p.dims, p.B, csa2.MODE_REUSE, p.q, p.codes, p.scales, p.rope,
                                 p.page_table, p.ctx, torch.from_numpy(tk).cuda(), p.swa,
                                 torch.from_numpy(np.asarray(sl, np.int32)).cuda(),
                                 1 / 24.0, out, lse, p.ws)
    return out, lse


def test_topk_index_out_of_range():
    p = make_problem([100, 200], seed=21)
    csa2.clear_device_status(p.ws)
    tk = np.full((2, p.K), -1, dtype=np.int32)
    tk[0, 0] = 5
    tk[0, 1] = 100          # == ctx_len: out of range
    tk[1, 0] = 10 ** 6
    out, lse = attn(p, tk, [0, 0])
    assert csa2.get_device_status(p.ws) & TOPK
    assert torch.isfinite(out).all()
    csa2.clear_device_status(p.ws)
    assert csa2.get_device_status(p.ws) == 0


def test_swa_len_out_of_range():
    p = make_problem([100], seed=22)
    csa2.clear_device_status(p.ws)
    tk = np.full((1, p.K), -1, dtype=np.int32)
    out, lse = attn(p, tk, [p.W + 5])
    assert csa2.get_device_status(p.ws) & SWA
    assert torch.isfinite(out).all()


def test_bad_page_id():
    p = make_problem([300, 130], paged=True, seed=23)
    csa2.clear_device_status(p.ws)
    p.page_table[1, 0] = int(p.dims.num_pages) + 10
    tk = np.full((2, p.K), -1, dtype=np.int32)
    tk[1, :5] = np.arange(5)
    attn(p, tk, [0, 0])
    assert csa2.get_device_status(p.ws) & PAGE
    csa2.clear_device_status(p.ws)
    run_full(p)
    assert csa2.get_device_status(p.ws) & PAGE


def test_ctx_len_above_capacity():
    p = make_problem([100, 200], seed=24, with_kv=False)
    csa2.clear_device_status(p.ws)
    p.ctx[1] = p.dims.max_ctx + 1
    pool, plen, topk = run_full(p)
    assert csa2.get_device_status(p.ws) & CTX
    assert plen.cpu().tolist()[1] == 0
    assert np.all(topk.cpu().numpy()[1] == -1)


def test_bounded_wait_gives_up_and_context_survives():
    """A bounded wait on an mbarrier that nothing arrives at gives up after its
    limit, reports CSA2_DEV_TIMEOUT through the error word, and the context
    still runs the library's kernels afterwards."""
    p = make_problem([3000, 1500], seed=21, with_kv=False)
    csa2.clear_device_status(p.ws)
    csa2.selftest_wait_timeout(p.ws, limit_us=2000)
    assert csa2.get_device_status(p.ws) & TIMEOUT
    csa2.clear_device_status(p.ws)
    assert csa2.get_device_status(p.ws) == 0
    pool, pool_len, tk = run_full(p)                  # a normal call on the same context
    torch.cuda.synchronize()
    assert csa2.get_device_status(p.ws) == 0
    assert int(pool_len.min()) > 0 and int((tk >= 0).sum()) > 0

"""The allocation-free decode attention call, through the C ABI.

For callers that may not allocate GPU memory on their hot path: the scratch
is a fixed array inside the library.  Its results must agree with the
workspace call's on the same inputs (same 2e-3 normwise tolerance as the
other attention tests), on two calls in a row that reuse the array.  This
file is collected last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_fp4_gb300 import csa2
from tests.gpu_problem import make_problem
from tests.helpers import normwise_rel

pytestmark = pytest.mark.gpu
TOL = 2e-3
SCALE = 1.0 / np.sqrt(576.0)


def _topk(p, rng):
    tk = np.full((p.B, p.K), -1, dtype=np.int32)
    for b, n in enumerate(p.ctx_lens):
        m = min(n, p.K - 3)
        tk[b, :m] = np.sort(rng.choice(n, m, replace=False))
    return torch.from_numpy(tk).cuda()


def _with_workspace(p, tk, q):
    out = torch.full((p.B, p.H, 512), float("nan"), device="cuda")
    lse = torch.full((p.B, p.H), float("nan"), device="cuda")
    csa2.csa2_sparse_attn_decode(p.dims, p.B, csa2.MODE_REUSE, q, p.codes, p.scales, p.rope,
                                 p.page_table, p.ctx, tk, p.swa, p.swa_len, SCALE, out, lse, p.ws)
    return out, lse


def _no_alloc(p, tk, q, err):
    out = torch.full((p.B, p.H, 512), float("nan"), device="cuda")
    lse = torch.full((p.B, p.H), float("nan"), device="cuda")
    csa2.csa2_sparse_attn_decode_noalloc(p.dims, p.B, csa2.MODE_REUSE, q, p.codes, p.scales,
                                         p.rope, p.page_table, p.ctx, tk, p.swa, p.swa_len,
                                         SCALE, out, lse, err)
    return out, lse


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    oa, ob, la, lb = oa.cpu().numpy(), ob.cpu().numpy(), la.cpu().numpy(), lb.cpu().numpy()
    assert np.all(normwise_rel(oa, ob) <= TOL)
    assert np.all(np.abs(la - lb) <= TOL)


@pytest.mark.parametrize("paged", [False, True])
def test_no_alloc_matches_workspace_call_twice(paged):
    p = make_problem([5000, 700, 64], paged=paged, seed=31)
    rng = np.random.default_rng(5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tk1 = _topk(p, rng)
    got1 = _no_alloc(p, tk1, p.q, err)
    want1 = _with_workspace(p, tk1, p.q)
    # second call in a row: new indices and a new query, same shared array
    tk2 = _topk(p, rng)
    q2 = (p.q.float() * 1.5).to(torch.bfloat16)
    got2 = _no_alloc(p, tk2, q2, err)
    want2 = _with_workspace(p, tk2, q2)
    torch.cuda.synchronize()
    _close(got1, want1)
    _close(got2, want2)
    assert int(err.item()) == 0


def test_no_alloc_reports_device_errors_and_limit():
    p = make_problem([100], seed=32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tk = torch.full((1, p.K), -1, dtype=torch.int32, device="cuda")
    tk[0, 0] = 100                      # == ctx_len: skipped and reported
    _no_alloc(p, tk, p.q, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x04
    # a batch whose scratch exceeds the fixed array is rejected on the host
    big = csa2.Dims(**{**p.dims.__dict__})
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_decode_noalloc(big, 64, csa2.MODE_REUSE, p.q, p.codes, p.scales,
                                             p.rope, None, p.ctx, tk, p.swa, p.swa_len, SCALE,
                                             p.q, p.q, None)
    assert e.value.code == 3

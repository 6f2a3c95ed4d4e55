"""GPU parity of the chunk-walking attention kernel against the oracle.

For large batches the library runs one CTA per (sequence, query, 32-head
group) that walks the 128-entry chunks in turn (online softmax against a
per-head reference maximum, O accumulated in tensor memory) instead of one
cluster per head group.  These cases have enough sequences for the library
to choose it; each checks that it ran and compares every sequence with the
oracle (tolerances as for the cluster kernel).
"""
import numpy as np
import pytest

from compressed_sparse_attention_fp4_gb300 import csa2
from tests.gpu_problem import make_problem
from tests.test_gpu_attention import check, random_topk, run_attn

pytestmark = pytest.mark.gpu


def run_walk(p, tk, sl, mode=csa2.MODE_REUSE):
    csa2.profile_enable(True)
    try:
        out, lse = run_attn(p, tk, sl, mode=mode)
        rec = csa2.profile_read()
    finally:
        csa2.profile_enable(False)
    assert rec.get("attn_seq_tc", (0, 0.0))[0] == 1, rec
    assert "attn_cluster_tc" not in rec, rec
    return out, lse


def ctx_mix(rng, B):
    n = rng.integers(200, 3000, B).tolist()
    n[0], n[1], n[2] = 1, 60, 700           # one position, fewer than Top-K, a few hundred
    return n


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("mode", [csa2.MODE_REUSE, csa2.MODE_FULL])
def test_walk_random(paged, mode):
    """64 sequences x 2 head groups: Reuse mode gathers the first chunk before
    the wait on the previous kernel, Full mode after it."""
    rng = np.random.default_rng(21)
    p = make_problem(ctx_mix(rng, 64), paged=paged, seed=21)
    tk = random_topk(p, rng)
    sl = rng.integers(0, 129, p.B).astype(np.int32)
    sl[:3] = [0, 128, 5]
    out, lse = run_walk(p, tk, sl, mode=mode)
    check(p, tk, out, lse, sl)


@pytest.mark.parametrize("sigma", [1.0, 4.0])
def test_walk_sharp_queries_move_the_reference(sigma):
    """Large logits: later chunks often exceed the reference maximum by more
    than 2^8, so the accumulated O and sums are rescaled in tensor memory."""
    rng = np.random.default_rng(22)
    p = make_problem(rng.integers(2000, 4000, 64).tolist(), seed=22, q_sigma=sigma)
    tk = random_topk(p, rng, frac_valid=1.0)
    # the entries in decreasing position order, so that the chunks meet
    # their maxima in no particular order
    tk = np.ascontiguousarray(tk[:, ::-1])
    out, lse = run_walk(p, tk, None)
    check(p, tk, out, lse)


def test_walk_empty_single_and_no_window_rows():
    """Sequences without any entry (output 0, lse -inf), with a single main
    entry, with window rows only, and with both."""
    rng = np.random.default_rng(23)
    p = make_problem(rng.integers(100, 1500, 64).tolist(), seed=23)
    tk = random_topk(p, rng)
    sl = np.full(p.B, 128, dtype=np.int32)
    tk[0:8] = -1
    sl[0:4] = 0                             # nothing at all
    tk[8:12] = -1
    tk[8:12, 0] = 0                         # one main entry, no window
    sl[8:12] = 0
    tk[12:16] = -1
    tk[12:16, 7] = 3                        # one main entry in a later slot, plus the window
    out, lse = run_walk(p, tk, sl)
    check(p, tk, out, lse, sl)


def test_walk_without_window():
    """No sliding window (4 chunks of Top-K slots only)."""
    rng = np.random.default_rng(24)
    p = make_problem(rng.integers(600, 2500, 64).tolist(), W=0, seed=24)
    tk = random_topk(p, rng)
    sl = np.zeros(p.B, dtype=np.int32)
    out, lse = run_walk(p, tk, sl)
    check(p, tk, out, lse, sl)

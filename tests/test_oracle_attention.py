"""Pins for the oracle's sparse attention and layer schedules (CPU only).

Checks against PyTorch's own float64 scaled-dot-product attention (selecting
every position reduces the sparse path to dense attention), closed forms
(one entry gives its value; a duplicated entry doubles its weight; a
constant logit shift leaves the output alone) and the mode identities of the
schedule (Reuse with recomputed indices equals Reindex).
"""
import numpy as np
import pytest
import torch

from oracle import attention, indexer, schedule


def rand_inputs(rng, n=300, H=8, W=20):
    latent = rng.standard_normal((n, 512))
    rope = rng.standard_normal((n, 64))
    q = rng.standard_normal((H, 576)) * 0.1
    swa = rng.standard_normal((W, 576))
    return q, latent, rope, swa


def sdpa(q, keys, vals, scale):
    """Dense attention two ways: PyTorch's float64 scaled_dot_product_attention
    (its backend picks the kernel) and the textbook softmax written out in
    NumPy; both must agree before either is used as the reference."""
    qt = torch.tensor(q)[None, :, None, :]                       # [1,H,1,576]
    kt = torch.tensor(keys)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.tensor(vals)[None, None].expand(1, q.shape[0], -1, -1)
    o_t = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()
    logits = scale * (np.asarray(q) @ np.asarray(keys).T)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    z = e.sum(axis=1, keepdims=True)
    o_np = (e @ np.asarray(vals)) / z
    lse = (m + np.log(z))[:, 0]
    assert np.allclose(o_t, o_np, rtol=1e-9, atol=1e-9)
    return o_np, lse


def test_all_positions_equals_dense_sdpa():
    rng = np.random.default_rng(0)
    q, latent, rope, swa = rand_inputs(rng)
    scale = 1 / np.sqrt(576)
    topk = np.arange(300)
    out, lse = attention.sparse_attn_decode(q, latent, rope, topk, swa, 0, scale)
    keys = np.concatenate([latent, rope], 1)
    o_ref, l_ref = sdpa(q, keys, latent, scale)
    assert np.allclose(out, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, l_ref, rtol=1e-12, atol=1e-12)


def test_sparse_plus_swa_equals_dense_on_union():
    rng = np.random.default_rng(1)
    q, latent, rope, swa = rand_inputs(rng)
    scale = 0.07
    topk = np.full(64, -1)
    sel = np.sort(rng.choice(300, 40, replace=False))
    topk[:40] = sel
    out, lse = attention.sparse_attn_decode(q, latent, rope, topk, swa, 13, scale)
    keys = np.concatenate([np.concatenate([latent[sel], rope[sel]], 1), swa[:13]])
    vals = np.concatenate([latent[sel], swa[:13, :512]])
    o_ref, l_ref = sdpa(q, keys, vals, scale)
    assert np.allclose(out, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, l_ref, rtol=1e-12, atol=1e-12)


def test_single_entry_returns_its_value():
    rng = np.random.default_rng(2)
    q, latent, rope, swa = rand_inputs(rng)
    topk = np.array([17, -1, -1])
    out, lse = attention.sparse_attn_decode(q, latent, rope, topk, swa, 0, 0.1)
    assert np.array_equal(out, np.broadcast_to(latent[17], out.shape))
    k = np.concatenate([latent[17], rope[17]])
    assert np.allclose(lse, 0.1 * q @ k, rtol=1e-14, atol=0)


def test_empty_set():
    rng = np.random.default_rng(3)
    q, latent, rope, swa = rand_inputs(rng)
    out, lse = attention.sparse_attn_decode(q, latent, rope, np.full(8, -1), swa, 0, 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_duplicate_entry_counts_twice():
    """A position present in both branches carries twice the weight."""
    rng = np.random.default_rng(4)
    q, latent, rope, swa = rand_inputs(rng, W=4)
    swa[2] = np.concatenate([latent[5], rope[5]])       # SWA row = main entry 5
    scale = 0.05
    out, lse = attention.sparse_attn_decode(q, latent, rope, np.array([5, 9]), swa[2:3], 1, scale)
    l5 = scale * q @ np.concatenate([latent[5], rope[5]])
    l9 = scale * q @ np.concatenate([latent[9], rope[9]])
    w5, w9 = 2 * np.exp(l5), np.exp(l9)
    want = (w5[:, None] * latent[5] + w9[:, None] * latent[9]) / (w5 + w9)[:, None]
    assert np.allclose(out, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, np.log(w5 + w9), rtol=1e-12, atol=1e-12)


def test_constant_logit_shift():
    """Adding c to every logit leaves o unchanged and moves lse by c.

    The shift is made through the data: an extra key channel equal to 1 for
    every key and the query channel c/scale (set on the rope part).
    """
    rng = np.random.default_rng(5)
    q, latent, rope, swa = rand_inputs(rng)
    rope[:, 63] = 0.0
    swa[:, 575] = 0.0
    q[:, 575] = 0.0
    topk = np.arange(0, 300, 3)
    scale = 0.04
    o1, l1 = attention.sparse_attn_decode(q, latent, rope, topk, swa, 20, scale)
    rope2, swa2, q2 = rope.copy(), swa.copy(), q.copy()
    rope2[:, 63] = 1.0
    swa2[:, 575] = 1.0
    c = 3.5
    q2[:, 575] = c / scale
    o2, l2 = attention.sparse_attn_decode(q2, latent, rope2, topk, swa2, 20, scale)
    assert np.allclose(o1, o2, rtol=1e-11, atol=1e-12)
    assert np.allclose(l2 - l1, c, rtol=0, atol=1e-11)


def test_split_merge_closed_form():
    rng = np.random.default_rng(6)
    q, latent, rope, swa = rand_inputs(rng)
    topk = np.sort(rng.choice(300, 50, replace=False))
    full = attention.sparse_attn_decode(q, latent, rope, topk, swa, 20, 0.05)
    a = attention.sparse_attn_decode(q, latent, rope, topk, swa, 0, 0.05)
    b = attention.sparse_attn_decode(q, latent, rope, np.array([-1]), swa, 20, 0.05)
    o, l = attention.lse_merge([a, b])
    assert np.allclose(o, full[0], rtol=1e-12, atol=1e-12)
    assert np.allclose(l, full[1], rtol=1e-12, atol=1e-12)


def _seq(rng, n=1200, Di=16, Hi=3, H=4):
    from tests.test_oracle_indexer import bf16_round, rand_e4m3
    idx_k = rand_e4m3(rng, (n, Di))
    latent = rng.standard_normal((n, 512))
    rope = rng.standard_normal((n, 64))

    def layer():
        return {"q": rng.standard_normal((H, 576)) * 0.1,
                "swa": rng.standard_normal((16, 576)), "swa_len": 16,
                "idx_q": bf16_round(rng.standard_normal((Hi, Di))),
                "idx_w": rng.random(Hi).astype(np.float32).astype(np.float64)}
    return idx_k, latent, rope, layer


def test_reuse_with_recomputed_indices_equals_reindex():
    rng = np.random.default_rng(7)
    idx_k, latent, rope, layer = _seq(rng)
    L = [layer(), layer(), layer()]
    res = schedule.run_sequence(["F", "Ri", "Ru"], idx_k, latent, rope, L,
                                pool_blocks=20, topk=30, scale=0.05)
    # recompute the Reindex indices by hand and feed them to a Reuse layer
    f = indexer.full_topk(L[0]["idx_q"], L[0]["idx_w"], idx_k, 20, 30)
    ri = indexer.reindex_topk(L[1]["idx_q"], L[1]["idx_w"], idx_k, f["pool"], 30)
    o, l = attention.sparse_attn_decode(L[1]["q"], latent, rope, ri["topk"],
                                        L[1]["swa"], 16, 0.05)
    assert np.array_equal(res[1]["topk"], ri["topk"])
    assert np.array_equal(res[1]["out"], o) and np.array_equal(res[1]["lse"], l)
    # the Reuse layer inherits the Reindex layer's indices
    assert np.array_equal(res[2]["topk"], res[1]["topk"])


def test_reuse_with_previous_query_equals_previous_output():
    rng = np.random.default_rng(8)
    idx_k, latent, rope, layer = _seq(rng)
    L = [layer(), layer()]
    L[1]["q"], L[1]["swa"] = L[0]["q"], L[0]["swa"]
    res = schedule.run_sequence(["F", "Ru"], idx_k, latent, rope, L,
                                pool_blocks=20, topk=30, scale=0.05)
    assert np.array_equal(res[0]["out"], res[1]["out"])
    assert np.array_equal(res[0]["lse"], res[1]["lse"])


def test_schedule_order_errors():
    rng = np.random.default_rng(9)
    idx_k, latent, rope, layer = _seq(rng, n=100)
    with pytest.raises(ValueError):
        schedule.run_sequence(["Ru"], idx_k, latent, rope, [layer()], 4, 8, 0.1)
    with pytest.raises(ValueError):
        schedule.run_sequence(["Ri"], idx_k, latent, rope, [layer()], 4, 8, 0.1)


def test_schedule_shapes():
    s = schedule.SCHEDULES
    assert s["128k"].count("F") == 1 and s["128k"].count("Ri") == 1 and s["128k"].count("Ru") == 10
    assert s["mix"].count("F") == 1 and s["mix"].count("Ri") == 1 and s["mix"].count("Ru") == 4

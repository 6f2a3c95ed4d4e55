"""GPU parity of the FP4 KV codec against the oracle (byte-exact).

Calls the library through its C ABI (ctypes binding).
"""
import numpy as np
import pytest
import torch

from oracle import codec as ocodec
from tests.helpers import bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_fp4_gb300 import csa2
    return csa2


def _to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def all_bf16_bits():
    b = np.arange(1 << 16, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return b[np.isfinite(f)].astype(np.uint16)


def test_every_bf16_against_every_scale(lib):
    """Each group: one element = 6*s (fixes the scale at s), 15 test values."""
    bits = all_bf16_bits()
    vals = bf16_f64(bits)
    groups = []
    for s_code in range(0, 0x7F):
        s = ocodec.e4m3_decode(np.array([s_code]))[0]
        top = 6.0 * s if s_code else 0.0
        sel = bits[np.abs(vals) <= top] if s_code else bits[vals == 0]
        if s_code == 0x7E:               # saturated groups: everything larger too
            sel = bits
        n = -(-sel.size // 15)
        pad = np.resize(sel, n * 15).reshape(n, 15)
        anchor = np.full((n, 1), np.float32(top).view(np.uint32) >> 16, dtype=np.uint16)
        if s_code == 0x7E:
            anchor[:] = np.float32(6.0 * 448.0).view(np.uint32) >> 16
        groups.append(np.concatenate([anchor, pad], axis=1))
    g = np.concatenate(groups)
    g = np.resize(g, (-(-g.shape[0] // 32) * 32, 16)).reshape(-1, 512)
    x = _to_dev(g)
    codes, scales = lib.fp4_kv_quantize(x)
    torch.cuda.synchronize()
    oc, os_ = ocodec.quantize_rows(bf16_f64(g))
    np.testing.assert_array_equal(scales.cpu().numpy(), os_)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)


def test_scale_of_every_amax(lib):
    bits = all_bf16_bits()
    pos = bits[bf16_f64(bits) >= 0]
    g = np.zeros((pos.size, 16), dtype=np.uint16)
    g[:, 0] = pos
    g = np.resize(g, (-(-g.shape[0] // 32) * 32, 16)).reshape(-1, 512)
    codes, scales = lib.fp4_kv_quantize(_to_dev(g))
    oc, os_ = ocodec.quantize_rows(bf16_f64(g))
    np.testing.assert_array_equal(scales.cpu().numpy(), os_)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)


def test_dequantize_exact(lib):
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 256, (4096, 256), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (4096, 32), dtype=np.uint8)   # finite codes
    y = lib.fp4_kv_dequantize(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    got = bf16_f64(y.view(torch.int16).cpu().numpy().view(np.uint16))
    want = ocodec.dequantize_rows(codes, scales)
    np.testing.assert_array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_ragged_row_counts_and_scatter(lib):
    from compressed_sparse_attention_fp4_gb300 import synth
    for n in [1, 7, 33, 1000]:
        x = synth.codec_slab(n=n, seed=5)
        c, s = lib.fp4_kv_quantize(_to_dev(x))
        oc, os_ = ocodec.quantize_rows(bf16_f64(x))
        np.testing.assert_array_equal(c.cpu().numpy(), oc)
        np.testing.assert_array_equal(s.cpu().numpy(), os_)
    n = 777
    x = synth.codec_slab(n=n, seed=6)
    perm = np.random.default_rng(1).permutation(2 * n)[:n]
    codes = torch.zeros((2 * n, 256), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((2 * n, 32), dtype=torch.uint8, device="cuda")
    dst = torch.from_numpy(perm.astype(np.int64)).cuda()
    lib.fp4_kv_quantize_scatter(_to_dev(x), dst, codes, scales)
    oc, os_ = ocodec.quantize_rows(bf16_f64(x))
    np.testing.assert_array_equal(codes.cpu().numpy()[perm], oc)
    np.testing.assert_array_equal(scales.cpu().numpy()[perm], os_)
    rest = np.setdiff1d(np.arange(2 * n), perm)
    assert not codes.cpu().numpy()[rest].any()
    # negative destination rows are skipped
    dst2 = dst.clone()
    dst2[::2] = -1
    codes.zero_()
    lib.fp4_kv_quantize_scatter(_to_dev(x), dst2, codes, scales)
    assert not codes.cpu().numpy()[perm[::2]].any()
    # early inputs (written while the kernel before runs, completed after it): the same bytes
    codes.zero_()
    scales.zero_()
    busy = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    busy.fill_(3)                                   # some kernel just before
    lib.fp4_kv_quantize_scatter(_to_dev(x), dst, codes, scales, flags=lib.KV_EARLY_INPUTS)
    np.testing.assert_array_equal(codes.cpu().numpy()[perm], oc)
    np.testing.assert_array_equal(scales.cpu().numpy()[perm], os_)
    assert not codes.cpu().numpy()[rest].any()


def test_codec_workload_full_size(lib):
    """1,048,576 x 512 slab with outlier channels: every row's codes and scales
    byte-exact against the oracle (run in chunks of 65,536 rows over a spawn
    process pool), every dequantized row bit-identical to the oracle's
    dequantization, round-trip error distribution reported."""
    import hashlib

    from compressed_sparse_attention_fp4_gb300 import synth
    from tests import oracle_jobs
    n = 1 << 20
    spans, ref = oracle_jobs.oracle_codec_slab(n)      # CPU pool first, then the GPU
    x = synth.codec_slab(n=n)
    xd = _to_dev(x)
    codes, scales = lib.fp4_kv_quantize(xd)
    y = lib.fp4_kv_dequantize(codes, scales)
    torch.cuda.synchronize()
    for (_, lo, hi), (oc, os_, yhash) in zip(spans, ref):
        np.testing.assert_array_equal(codes[lo:hi].cpu().numpy(), oc, err_msg=f"codes rows {lo}..{hi}")
        np.testing.assert_array_equal(scales[lo:hi].cpu().numpy(), os_, err_msg=f"scales rows {lo}..{hi}")
        got = y[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        assert hashlib.sha256(got.tobytes()).hexdigest() == yhash, f"dequantized rows {lo}..{hi}"
    # round-trip error distribution over the whole slab (relative to group amax)
    xf = xd.float().view(n, 32, 16)
    err = (y.float().view(n, 32, 16) - xf).abs().amax(-1) / xf.abs().amax(-1).clamp_min(1e-30)
    q = torch.quantile(err.flatten()[:1 << 24], torch.tensor([0.5, 0.99, 1.0], device="cuda"))
    print("round-trip max|err|/amax per group: median %.4g p99 %.4g max %.4g" % tuple(q.tolist()))
    # |x - dq| <= s and s <= amax/6 * (1 + 2^-4): at most ~0.177 of the group amax
    assert float(q[2]) <= 0.18


def test_fp4_slab_save_reload_byte_stable(lib, tmp_path):
    """The packed FP4 slab is a byte-stable storage format: written by the GPU,
    saved to a file and loaded back, it is byte-identical, dequantizes to the
    same bf16 values, and quantizing those values again gives the same bytes."""
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((4096, 512)).astype(np.float32)).cuda().to(torch.bfloat16)
    codes, scales = lib.fp4_kv_quantize(x)
    path = tmp_path / "slab.bin"
    np.concatenate([codes.cpu().numpy().ravel(), scales.cpu().numpy().ravel()]).tofile(path)
    raw = np.fromfile(path, dtype=np.uint8)
    c2 = torch.from_numpy(raw[:codes.numel()].reshape(tuple(codes.shape)).copy()).cuda()
    s2 = torch.from_numpy(raw[codes.numel():].reshape(tuple(scales.shape)).copy()).cuda()
    assert torch.equal(c2, codes) and torch.equal(s2, scales)
    y1 = lib.fp4_kv_dequantize(codes, scales)
    y2 = lib.fp4_kv_dequantize(c2, s2)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    c3, s3 = lib.fp4_kv_quantize(y2)
    assert torch.equal(c3, codes) and torch.equal(s3, scales)

"""Test plumbing: format widening for the oracle side and device uploads.

Nothing here computes the method: bf16 / E4M3 inputs are widened to float64
for the oracle, and tensors are moved between host and device.
"""
import numpy as np

from oracle import codec as ocodec


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def idxk_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Indexer keys in storage format -> float64 (E4M3 decoded by the oracle)."""
    if dtype == "fp8":
        return ocodec.e4m3_decode(np.asarray(raw, dtype=np.uint8))
    return np.asarray(raw, dtype=np.float32).astype(np.float64)


def oracle_latent(latent_bits: np.ndarray) -> np.ndarray:
    """The oracle's own FP4 write then read of a bf16 latent block."""
    codes, scales = ocodec.quantize_rows(bf16_f64(latent_bits))
    return ocodec.dequantize_rows(codes, scales)


def normwise_rel(o: np.ndarray, r: np.ndarray) -> np.ndarray:
    """max_i |o_i - r_i| / max_i |r_i| per row (last axis)."""
    num = np.max(np.abs(o - r), axis=-1)
    den = np.max(np.abs(r), axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def ws_offsets(dims, batch):
    """Byte offsets of the workspace regions (mirror of the library layout)."""
    def a256(x):
        return (x + 255) & ~255
    off = 256
    nb_max = (dims.max_ctx + 7) // 8
    r = {"nb_max": nb_max}
    r["pos_scores"] = off; off = a256(off + batch * dims.max_ctx * 4)
    r["blk_scores"] = off; off = a256(off + batch * nb_max * 4)
    r["blk_delta"] = off; off = a256(off + batch * nb_max * 4)
    r["ri_scores"] = off; off = a256(off + batch * dims.pool_blocks * 8 * 4)
    r["ri_delta"] = off; off = a256(off + batch * dims.pool_blocks * 4)
    return r

"""The oracle pins catch plausible mistakes.

Each test plants one mistake in a copy of an oracle function (on the CPU) and
checks that an independent pin from the other oracle tests rejects it: a
wrong tie rule, a dropped sign, a wrong E4M3 bias, an off-by-one block, a
transposed head/channel contraction, ties to the higher index, a missing
SWA branch, a dropped attention scale; for the FP4 indexer, an unquantized
query and dropped scales.
"""
import numpy as np
import pytest

from oracle import attention, codec, indexer, indexer_fp4
from tests import test_oracle_codec as tc
from tests import test_oracle_indexer as ti
from tests import test_oracle_indexer_fp4 as tf


def test_tie_rule_mutation_is_caught(monkeypatch):
    orig = codec.e2m1_round_magnitude
    monkeypatch.setattr(codec, "e2m1_round_magnitude", lambda r, p1_mode=False: orig(r, p1_mode=True))
    with pytest.raises(AssertionError):
        tc.test_element_rounding_exhaustive_threshold_form()
    with pytest.raises(AssertionError):
        tc.test_hand_worked_example()


def test_dropped_sign_mutation_is_caught(monkeypatch):
    orig = codec.quantize_rows

    def no_sign(x, p1_mode=False):
        return orig(np.abs(x), p1_mode)
    monkeypatch.setattr(codec, "quantize_rows", no_sign)
    with pytest.raises(AssertionError):
        tc.test_hand_worked_example()
    with pytest.raises(AssertionError):
        tc.test_sixteen_codes_round_trip()


def test_e4m3_bias_mutation_is_caught(monkeypatch):
    orig = codec.e4m3_decode
    monkeypatch.setattr(codec, "e4m3_decode", lambda c: orig(c) * 2.0)
    with pytest.raises(AssertionError):
        tc.test_e4m3_decode_matches_ocp_definition()


def test_block_size_mutation_is_caught(monkeypatch):
    orig = indexer.block_scores
    monkeypatch.setattr(indexer, "block_scores", lambda s, block=8: orig(s, 7))
    with pytest.raises(AssertionError):
        ti.test_block_scores_brute_force()


def test_transposed_contraction_is_caught(monkeypatch):
    orig = indexer.head_dots_exact_multi

    def transposed(q, K, chunk=1 << 16):
        q = np.asarray(q, dtype=np.float64)
        return orig(q[:, ::-1].copy(), K, chunk)      # channels reversed
    monkeypatch.setattr(indexer, "head_dots_exact_multi", transposed)
    with pytest.raises(AssertionError):
        ti.test_head_dots_match_fraction_fp8()


def test_tie_to_higher_index_is_caught(monkeypatch):
    def top_high(values, k):
        values = np.asarray(values, dtype=np.float64)
        order = np.lexsort((-np.arange(values.shape[0]), -values))
        return order[:k]
    monkeypatch.setattr(indexer, "top_order", top_high)
    with pytest.raises(AssertionError):
        ti.test_top_order_brute_force_with_ties()


def test_missing_swa_branch_is_caught(monkeypatch):
    from tests import test_oracle_attention as ta
    orig = attention.sparse_attn_decode

    def no_swa(q, latent, rope, topk, swa, swa_len, scale):
        return orig(q, latent, rope, topk, swa, 0, scale)
    monkeypatch.setattr(attention, "sparse_attn_decode", no_swa)
    with pytest.raises(AssertionError):
        ta.test_sparse_plus_swa_equals_dense_on_union()


def test_dropped_scale_is_caught(monkeypatch):
    from tests import test_oracle_attention as ta
    orig = attention.sparse_attn_decode

    def no_scale(q, latent, rope, topk, swa, swa_len, scale):
        return orig(q, latent, rope, topk, swa, swa_len, 1.0)
    monkeypatch.setattr(attention, "sparse_attn_decode", no_scale)
    with pytest.raises(AssertionError):
        ta.test_all_positions_equals_dense_sdpa()


def test_fp4_indexer_unquantized_query_is_caught(monkeypatch):
    def raw_query_full(q, w, k, pool_blocks, topk):
        kc, ks = indexer_fp4.quantize(k)
        return indexer.full_topk(q, w, indexer_fp4.dequantize(kc, ks), pool_blocks, topk)
    monkeypatch.setattr(indexer_fp4, "full_topk", raw_query_full)
    with pytest.raises(AssertionError):
        tf.test_depends_only_on_quantized_inputs()


def test_fp4_indexer_dropped_scales_are_caught(monkeypatch):
    monkeypatch.setattr(indexer_fp4, "dequantize",
                        lambda codes, scales: codec.dequantize_rows(codes, np.full_like(scales, 0x38)))  # 1.0
    with pytest.raises(AssertionError):
        tf.test_grid_values_round_trip_and_score_unchanged()
    with pytest.raises(AssertionError):
        tf.test_quantization_error_bound()

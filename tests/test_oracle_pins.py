"""The CPU oracle against what the pages and the mathematics fix (no GPU needed)."""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import accounting
from tests import oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def test_decode_brute_force():
    pins.check_decode_brute(oracle.decode_gqa)


def test_decode_value_width():
    pins.check_decode_value_width(oracle.decode_gqa)


def test_prefill_brute_force():
    pins.check_prefill_brute(oracle.prefill_gqa_causal)


def test_decode_matches_torch_sdpa():
    pins.check_decode_sdpa(oracle.decode_gqa)


def test_prefill_matches_torch_sdpa_causal():
    pins.check_prefill_sdpa(oracle.prefill_gqa_causal)


def test_decode_closed_forms():
    pins.check_decode_closed_forms(oracle.decode_gqa)


def test_prefill_closed_forms():
    pins.check_prefill_closed_forms(oracle.prefill_gqa_causal)


def test_decode_invariants():
    pins.check_decode_invariants(oracle.decode_gqa)


def test_mha_mqa_endpoints():
    pins.check_mha_mqa_endpoints(oracle.decode_gqa, oracle.repeat_kv)


def test_repeat_kv_is_repeat_interleave():
    pins.check_repeat_kv(oracle.repeat_kv)


def test_head_mapping():
    # contiguous groups: with 32 Q heads and 8 groups, heads 0-3 use group 0, 28-31 use 7
    assert [oracle.kv_head_for_query_head(h, 32, 8) for h in (0, 3, 4, 31)] == [0, 0, 1, 7]
    assert all(oracle.kv_head_for_query_head(h, 32, 1) == 0 for h in range(32))
    assert [oracle.kv_head_for_query_head(h, 32, 32) for h in range(32)] == list(range(32))


def test_split_merge_identity():
    pins.check_split_merge(oracle.attend, oracle.attend_partial, oracle.lse_merge)


def test_mla_naive_brute_force():
    pins.check_mla_naive_brute(oracle.mla_decode_naive)


def test_mla_absorbed_equals_naive():
    pins.check_mla_absorbed_equals_naive(oracle.absorb_query, oracle.mla_decode_absorbed,
                                         oracle.apply_uv, oracle.mla_decode_naive)


def test_mla_is_mqa_with_shared_latent():
    pins.check_mla_is_mqa(oracle.mla_decode_absorbed, oracle.decode_gqa)


# ----------------------------------------------------------------------------- grouping rule

@pytest.mark.parametrize("n_kv", [3, 6, 5, 7, 0])
def test_non_divisor_kv_groups_rejected(n_kv):
    with pytest.raises(ValueError):
        oracle.check_grouping(32, n_kv)


def test_valid_group_counts_and_modes():
    g = _golden("coregenaihub_llama3_8b_modes.json")
    assert accounting.valid_kv_group_counts(g["n_q_heads"]) == g["valid_kv_groups_for_32_q_heads"]
    for n_kv in g["rejected_kv_groups_for_32_q_heads"]:
        with pytest.raises(ValueError):
            accounting.savings_vs_mha(g["n_q_heads"], n_kv)
    for row in g["modes"]:
        assert accounting.attention_mode(g["n_q_heads"], row["kv_groups"]) == row["mode"]
        assert g["n_q_heads"] // row["kv_groups"] == row["q_heads_per_group"]


# ----------------------------------------------------------------------------- accounting

def test_llama3_8b_table():
    g = _golden("coregenaihub_llama3_8b_modes.json")
    for row in g["modes"]:
        args = (row["kv_groups"], g["head_dim"], g["dtype"], g["n_layers"])
        assert accounting.kv_bytes_per_token(*args) == row["kv_bytes_per_token"]
        assert accounting.kv_cache_bytes(*args, g["context_tokens"]) == row["cache_bytes"]
        assert accounting.savings_vs_mha(g["n_q_heads"], row["kv_groups"]) == row["savings"]
        assert accounting.kv_projection_params(g["model_dim"], row["kv_groups"], g["head_dim"],
                                               g["n_layers"]) == row["kv_proj_params"]
        assert accounting.attention_projection_params(g["model_dim"], g["n_q_heads"], row["kv_groups"],
                                                      g["head_dim"], g["n_layers"]) == row["all_proj_params"]
    gqa = accounting.kv_bytes_per_token(8, 128, "bf16", 32)
    assert gqa == g["headline_bytes_per_token_kib"] * 1024
    assert accounting.kv_cache_bytes(8, 128, "bf16", 32, 8192) == g["headline_cache_for_8192_gib"] * 2 ** 30
    # Q and O projections do not depend on the grouping
    q_and_o = accounting.attention_projection_params(4096, 32, 32, 128, 32) - \
        accounting.kv_projection_params(4096, 32, 128, 32)
    assert q_and_o == g["q_and_o_params"]


def test_savings_independent_of_context_and_dtype():
    # the ratio is Hq/Hkv: context length and bytes per number cancel
    for dtype in ("fp32", "bf16", "fp8", "int4"):
        for n_tok in (512, 8192, 131072):
            mha = accounting.kv_cache_bytes(32, 128, dtype, 32, n_tok)
            for n_kv in (1, 2, 4, 8, 16, 32):
                assert mha / accounting.kv_cache_bytes(n_kv, 128, dtype, 32, n_tok) == 32 // n_kv
    # fp8 halves bf16; int4 gives a fractional byte count when the product is odd
    assert accounting.kv_bytes_per_token(8, 128, "fp8", 32) * 2 == accounting.kv_bytes_per_token(8, 128, "bf16", 32)
    assert accounting.kv_bytes_per_token(1, 1, "int4", 1) == Fraction(1)
    assert accounting.kv_bytes_per_token(1, 1, "int4", 1) / 2 == Fraction(1, 2)


def test_minimind_gqa_vs_mla_floats():
    g = _golden("minimind_kv_floats.json")
    gqa = accounting.gqa_floats_per_token_per_layer(g["gqa"]["n_kv_heads"], g["gqa"]["head_dim"])
    mla = accounting.mla_floats_per_token_per_layer(g["mla"]["kv_lora_rank"], g["mla"]["rope_dim"])
    assert gqa == g["gqa"]["floats_per_token_per_layer"]
    assert mla == g["mla"]["floats_per_token_per_layer"]
    printed = float(g["compression_printed"].rstrip("x"))
    assert round(gqa / mla, g["compression_rounding_digits"]) == printed
    assert math.isclose(gqa / mla, 768 / 176)


# ----------------------------------------------------------------------------- RoPE + append

def test_rope_is_complex_multiplication_of_pairs():
    pins.check_rope_complex(oracle.rope_rotate)


def test_rope_closed_forms():
    pins.check_rope_closed_forms(oracle.rope_rotate)


def test_rope_relative_position():
    pins.check_rope_relative_position(oracle.rope_rotate)


def test_kv_append_brute_force():
    pins.check_append_brute(oracle.kv_append_rope)


def test_mla_append_brute_force():
    pins.check_mla_append_brute(oracle.mla_append_rope)


# ----------------------------------------------------------------------------- fp8 cache

def test_e4m3_codes_match_torch():
    pins.check_e4m3_table(oracle.e4m3_to_float)


def test_e4m3_closed_forms():
    pins.check_e4m3_closed_forms(oracle.e4m3_to_float)


def test_fp8_decode_identities():
    pins.check_fp8_decode_identities(oracle.decode_gqa_fp8, oracle.e4m3_to_float, oracle.decode_gqa)


# ----------------------------------------------------------------------------- chunked prefill

def test_chunked_prefill_matches_sdpa_with_offset_mask():
    pins.check_chunked_sdpa(oracle.prefill_gqa_chunked)


def test_chunked_prefill_ends_are_prefill_and_decode():
    pins.check_chunked_ends(oracle.prefill_gqa_chunked, oracle.prefill_gqa_causal, oracle.decode_gqa)


def test_mla_chunked_prefill():
    pins.check_mla_chunked(oracle.mla_prefill_absorbed, oracle.mla_prefill_naive, oracle.absorb_query,
                           oracle.apply_uv, oracle.mla_decode_absorbed)

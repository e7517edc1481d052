"""KV-cache byte and projection-parameter accounting (test infrastructure).

"MHA, MQA và GQA" (coregenaihub interactive ebook): bytes of KV cache per token are
``2 × KV groups × head dim × bytes per number × layers`` (K and V, one vector each per
group per layer); the cache for n tokens of one sequence is n times that (no paging
overhead); the saving against MHA is Hq / Hkv, independent of context length and number
type; the K and V projections shrink by the same factor while Q and O do not.
"Attention Architecture Experiments" (minimind docs), section "Benchmark": floats per
token per layer are 2·Hkv·D for GQA and kv_lora_rank + rope_dim for MLA.
"""

from fractions import Fraction

from .attention import check_grouping

BYTES_PER_NUMBER = {"fp32": Fraction(4), "bf16": Fraction(2), "fp8": Fraction(1), "int4": Fraction(1, 2)}


def kv_bytes_per_token(n_kv_heads, head_dim, dtype, n_layers):
    """2 × Hkv × D × bytes × layers. Sub-byte types give a fractional count, which the
    ebook calls correct accounting; the value is returned as a Fraction."""
    return 2 * int(n_kv_heads) * int(head_dim) * BYTES_PER_NUMBER[dtype] * int(n_layers)


def kv_cache_bytes(n_kv_heads, head_dim, dtype, n_layers, n_tokens):
    """Cache for ``n_tokens`` of one sequence, without paging overhead."""
    return kv_bytes_per_token(n_kv_heads, head_dim, dtype, n_layers) * int(n_tokens)


def savings_vs_mha(n_q_heads, n_kv_heads):
    """Hq / Hkv; rejects a KV-group count that does not divide Hq."""
    return check_grouping(n_q_heads, n_kv_heads)


def valid_kv_group_counts(n_q_heads):
    """The divisors of Hq: the only KV-group counts the ebook's sim accepts."""
    return [d for d in range(1, int(n_q_heads) + 1) if n_q_heads % d == 0]


def attention_mode(n_q_heads, n_kv_heads):
    """'MHA' at Hkv = Hq, 'MQA' at Hkv = 1, else 'GQA' (the two ends of one scale)."""
    check_grouping(n_q_heads, n_kv_heads)
    if n_kv_heads == n_q_heads:
        return "MHA"
    if n_kv_heads == 1:
        return "MQA"
    return "GQA"


def kv_projection_params(model_dim, n_kv_heads, head_dim, n_layers):
    """Weights of W_K and W_V (no bias): 2 × dim × (Hkv × D) per layer."""
    return 2 * int(model_dim) * int(n_kv_heads) * int(head_dim) * int(n_layers)


def attention_projection_params(model_dim, n_q_heads, n_kv_heads, head_dim, n_layers):
    """Weights of all four projections: W_Q and W_O (dim × Hq·D each, independent of the
    grouping) plus W_K and W_V."""
    check_grouping(n_q_heads, n_kv_heads)
    q_and_o = 2 * int(model_dim) * int(n_q_heads) * int(head_dim) * int(n_layers)
    return q_and_o + kv_projection_params(model_dim, n_kv_heads, head_dim, n_layers)


def gqa_floats_per_token_per_layer(n_kv_heads, head_dim):
    """2 · Hkv · D numbers cached per token per layer (K and V)."""
    return 2 * int(n_kv_heads) * int(head_dim)


def mla_floats_per_token_per_layer(kv_lora_rank, rope_dim):
    """r + dr numbers cached per token per layer (latent c and the shared RoPE key)."""
    return int(kv_lora_rank) + int(rope_dim)

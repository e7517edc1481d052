"""Plain fp64 MLA decode (test infrastructure; see the package docstring).

Source: the qqstock article on DeepSeek MLA. Section 1: K and V are rebuilt from one
low-rank latent c per token (``compressed_kv``, width kv_lora_rank = r) by two up
projections. Section 2: the up projections can be absorbed ("合并与吸收") so attention runs
on c directly. Section 3: a decoupled RoPE key (``k_rope_linear``, width rope_head_dim =
dr) is shared by all heads and carried beside c. Section 6: MLA computes like MQA, with V
sharing the activation (c) of the un-RoPE'd K. The article's ``MultiHeadLatentAttention``
code gives the shapes: ``decompress_k_nope`` maps r → Hq·d_nope, ``decompress_v_linear``
maps r → Hq·d_v, the key is ``[k_nope ‖ k_rope]`` with k_rope broadcast to every head,
the query ``[q_nope ‖ q_rope]``, and attention is SDPA (default scale
1/sqrt(d_nope + dr)).

Weight layout used here, as ``nn.Linear`` stores it split per head:
  W_UK [Hq, d_nope, r]   k_nope[t, h] = W_UK[h] @ c_t
  W_UV [Hq, d_v,    r]   v[t, h]      = W_UV[h] @ c_t

Not applied (the cached values are taken as given): RoPE itself, RMSNorm, the article's
ad-hoc ``key_rope / num_heads`` line, dropout, and the output projection.
"""

import numpy as np

from .attention import attend


def absorb_query(q_nope, w_uk):
    """q_lat[b, h] = W_UK[h]ᵀ · q_nope[b, h] (qqstock article, section 2).

    q_nope [B, Hq, d_nope], w_uk [Hq, d_nope, r] → q_lat [B, Hq, r] float64. Then
    q_nope · k_nope = q_nopeᵀ W_UK[h] c = q_lat · c, so scores need only c.
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    return np.einsum("hnr,bhn->bhr", w_uk, q_nope)


def apply_uv(o_lat, w_uv):
    """o[b, h] = W_UV[h] · o_lat[b, h]: the value up projection applied once after the
    softmax average instead of once per cached token (qqstock article, section 2).
    o_lat [B, Hq, r], w_uv [Hq, d_v, r] → o [B, Hq, d_v] float64."""
    o_lat = np.asarray(o_lat, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    return np.einsum("hvr,bhr->bhv", w_uv, o_lat)


def mla_decode_absorbed(q_lat, q_rope, c_cache, kr_cache, seq_lens, scale):
    """Absorbed MLA decode: o_lat[b, h] = Σ_t softmax_t(scale·(q_lat·c_t + q_rope·kr_t)) c_t.

    q_lat [B, Hq, r], q_rope [B, Hq, dr], c_cache [B, S_max, r], kr_cache [B, S_max, dr],
    seq_lens [B]. Every head reads the same latent row [c_t ‖ kr_t], and the value is c_t
    itself: MQA with key width r + dr and value width r (qqstock article, section 6).
    Returns o_lat [B, Hq, r] float64 (before W_UV).
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    c_cache = np.asarray(c_cache, dtype=np.float64)
    kr_cache = np.asarray(kr_cache, dtype=np.float64)
    bsz, n_q, r = q_lat.shape
    out = np.zeros((bsz, n_q, r), dtype=np.float64)
    for b in range(bsz):
        s = int(seq_lens[b])
        q_row = np.concatenate([q_lat[b], q_rope[b]], axis=1)          # [Hq, r+dr]
        k_row = np.concatenate([c_cache[b, :s], kr_cache[b, :s]], axis=1)  # [S, r+dr]
        out[b] = attend(q_row, k_row, c_cache[b, :s], scale)
    return out


def mla_decode_naive(q_nope, q_rope, c_cache, kr_cache, w_uk, w_uv, seq_lens, scale):
    """Decompress-then-attend MLA decode, the way the article's code runs it.

    Per head h and cached token t: k = [W_UK[h] c_t ‖ kr_t], v = W_UV[h] c_t; the query is
    [q_nope ‖ q_rope]; o[b, h] = softmax(scale · q·kᵀ) · v. Returns o [B, Hq, d_v]
    float64. Equal to ``apply_uv(mla_decode_absorbed(absorb_query(q_nope, W_UK), ...),
    W_UV)`` in exact arithmetic.
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    c_cache = np.asarray(c_cache, dtype=np.float64)
    kr_cache = np.asarray(kr_cache, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    bsz, n_q, _ = q_nope.shape
    d_v = w_uv.shape[1]
    out = np.zeros((bsz, n_q, d_v), dtype=np.float64)
    for b in range(bsz):
        s = int(seq_lens[b])
        c = c_cache[b, :s]                                   # [S, r]
        for h in range(n_q):
            k_nope = c @ w_uk[h].T                           # [S, d_nope]
            keys = np.concatenate([k_nope, kr_cache[b, :s]], axis=1)
            vals = c @ w_uv[h].T                             # [S, d_v]
            q_row = np.concatenate([q_nope[b, h], q_rope[b, h]])[None, :]
            out[b, h] = attend(q_row, keys, vals, scale)[0]
    return out

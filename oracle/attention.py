"""Plain fp64 attention over a KV cache (test infrastructure; see the package docstring).

Everything follows "模型架构｜MQA & GQA 调研" (lichtung612 blog), section "代码":
``repeat_kv`` expands the KV heads to the query heads, ``Attention.forward`` writes the new
token into ``cache_k``/``cache_v`` and then attends over ``cache[:bsz, :start_pos+seqlen]``
with ``scores = xq·keysᵀ / sqrt(head_dim)``, ``scores + mask``, a softmax taken in fp32
(here fp64) and ``scores·values``.

No splitting, no online softmax, no fusion: each output row is the softmax-weighted
average of the value rows it may see, computed in one pass with a max-subtracted
exponential (an exact rewrite of the softmax, done for range only).
"""

import math

import numpy as np


def check_grouping(n_q_heads, n_kv_heads):
    """Reject a KV-head count that does not divide the query-head count.

    "MHA, MQA và GQA" (coregenaihub), step "Ba" of the sim walk-through and quiz item 2:
    with 32 Q heads the sim refuses 3 (or 6) KV groups instead of rounding, because every
    group must hold the same whole number of query heads; the valid counts are the
    divisors of the Q-head count. Returns the group size G = Hq / Hkv (``n_rep`` in the
    lichtung612 code).
    """
    n_q_heads = int(n_q_heads)
    n_kv_heads = int(n_kv_heads)
    if n_q_heads < 1 or n_kv_heads < 1:
        raise ValueError(f"head counts must be positive, got Hq={n_q_heads}, Hkv={n_kv_heads}")
    if n_q_heads % n_kv_heads != 0:
        raise ValueError(
            f"Hkv={n_kv_heads} does not divide Hq={n_q_heads} "
            f"(remainder {n_q_heads % n_kv_heads})"
        )
    return n_q_heads // n_kv_heads


def kv_head_for_query_head(h, n_q_heads, n_kv_heads):
    """KV head read by query head ``h``.

    lichtung612 blog, section "代码", ``repeat_kv``: ``x[:, :, :, None, :]`` is expanded to
    ``(bs, slen, n_kv_heads, n_rep, head_dim)`` and reshaped to ``n_kv_heads * n_rep``
    heads, so the ``n_rep`` copies of KV head j sit at query positions
    ``j*n_rep .. j*n_rep + n_rep - 1``: query head h reads KV head ``h // n_rep``.
    """
    g = check_grouping(n_q_heads, n_kv_heads)
    if not 0 <= h < n_q_heads:
        raise IndexError(f"query head {h} out of range [0, {n_q_heads})")
    return h // g


def repeat_kv(x, n_rep):
    """NumPy restatement of the page's ``repeat_kv``: ``(bs, slen, n_kv, hd)`` →
    ``(bs, slen, n_kv * n_rep, hd)`` by inserting a new axis after the head axis,
    broadcasting it to ``n_rep`` and merging it into the head axis (lichtung612 blog,
    section "代码"). Materialises the copies; used only to pin the GQA↔MHA identity."""
    x = np.asarray(x)
    if n_rep == 1:
        return x
    bs, slen, n_kv, hd = x.shape
    return np.broadcast_to(x[:, :, :, None, :], (bs, slen, n_kv, n_rep, hd)).reshape(
        bs, slen, n_kv * n_rep, hd
    )


def attend(q_rows, keys, values, scale, allowed=None):
    """softmax(scale · q_rows · keysᵀ [masked]) · values, in fp64.

    q_rows [M, Dk], keys [N, Dk], values [N, Dv]; ``allowed`` is an optional boolean
    [M, N] mask (True = the key is visible). A masked score is excluded from the softmax
    exactly, which is what adding -inf before the softmax does (lichtung612 blog,
    ``scores = scores + mask``). A row that sees no key at all is defined as zero.
    Returns [M, Dv] float64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    m = q_rows.shape[0]
    out = np.zeros((m, values.shape[1]), dtype=np.float64)
    if keys.shape[0] == 0 or m == 0:
        return out
    scores = float(scale) * (q_rows @ keys.T)
    if allowed is not None:
        scores = np.where(allowed, scores, -np.inf)
    row_max = scores.max(axis=1, keepdims=True)
    live = np.isfinite(row_max[:, 0])
    if not live.any():
        return out
    s = scores[live]
    e = np.exp(s - row_max[live])
    p = e / e.sum(axis=1, keepdims=True)
    out[live] = p @ values
    return out


def attend_partial(q_rows, keys, values, scale):
    """Attention over one contiguous piece of the keys, returned as (o, lse).

    o [M, Dv] is the piece's normalised output (the same as :func:`attend` on the piece)
    and lse [M] = ln Σ_t exp(scale · q·k_t) over the piece (natural log). An empty piece
    gives o = 0 and lse = -inf. These are the split partials that :func:`lse_merge`
    combines.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    m = q_rows.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((m, np.asarray(values).shape[1])), np.full(m, -np.inf)
    scores = float(scale) * (q_rows @ keys.T)
    row_max = scores.max(axis=1)
    lse = row_max + np.log(np.exp(scores - row_max[:, None]).sum(axis=1))
    return attend(q_rows, keys, values, scale), lse


def lse_merge(o_parts, lse_parts):
    """Combine split partials: out = Σ_i e^{lse_i − M} o_i / Σ_i e^{lse_i − M}, M = max_i lse_i.

    o_parts [n, M, Dv], lse_parts [n, M]. Pieces with lse = -inf carry no weight; a row
    whose every piece is empty is zero. In exact arithmetic this equals :func:`attend`
    over the union of the pieces, because e^{lse_i} is the piece's softmax denominator
    and o_i its normalised numerator.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    big = lse_parts.max(axis=0)
    out = np.zeros(o_parts.shape[1:], dtype=np.float64)
    live = np.isfinite(big)
    if not live.any():
        return out
    w = np.exp(lse_parts[:, live] - big[None, live])
    out[live] = (w[:, :, None] * o_parts[:, live, :]).sum(axis=0) / w.sum(axis=0)[:, None]
    return out


def decode_gqa_unit(q, k_cache, v_cache, seq_lens, scale, b, j):
    """Output rows of the G query heads that share KV head ``j`` of sequence ``b``.

    Decode attends every cached position ``0 .. seq_lens[b]-1``, which includes the token
    just appended (lichtung612 blog, ``Attention.forward`` writes
    ``cache_k[:bsz, start_pos:start_pos+seqlen]`` before it reads
    ``cache_k[:bsz, :start_pos+seqlen]``). Returns [G, D] float64.
    """
    n_q = q.shape[1]
    n_kv = k_cache.shape[2]
    g = check_grouping(n_q, n_kv)
    s = int(seq_lens[b])
    heads = slice(j * g, (j + 1) * g)
    return attend(q[b, heads, :], k_cache[b, :s, j, :], v_cache[b, :s, j, :], scale)


def decode_gqa(q, k_cache, v_cache, seq_lens, scale):
    """One decode step of GQA attention (MHA when Hkv = Hq, MQA when Hkv = 1).

    q [B, Hq, D]; k_cache, v_cache [B, S_max, Hkv, D] (the page's
    ``(max_batch_size, max_seq_len, n_kv_heads, head_dim)`` cache); seq_lens [B] with
    0 ≤ S_b ≤ S_max. Query head h reads KV head h // (Hq/Hkv) (see
    :func:`kv_head_for_query_head`). Returns out [B, Hq, D] float64; a sequence with
    S_b = 0 gives zeros.
    """
    q = np.asarray(q)
    k_cache = np.asarray(k_cache)
    v_cache = np.asarray(v_cache)
    bsz, n_q, _ = q.shape
    n_kv = k_cache.shape[2]
    g = check_grouping(n_q, n_kv)
    seq_lens = np.asarray(seq_lens).astype(np.int64)
    if seq_lens.shape != (bsz,) or (seq_lens < 0).any() or (seq_lens > k_cache.shape[1]).any():
        raise ValueError("seq_lens must be [B] with 0 <= S_b <= S_max")
    out = np.zeros((bsz, n_q, v_cache.shape[3]), dtype=np.float64)
    for b in range(bsz):
        for j in range(n_kv):
            out[b, j * g:(j + 1) * g] = decode_gqa_unit(q, k_cache, v_cache, seq_lens, scale, b, j)
    return out


def causal_allowed(q_len, k_len):
    """Visibility mask for causal attention of ``q_len`` new tokens over ``k_len`` keys.

    Query i sits at absolute position (k_len − q_len) + i — the page's
    ``start_pos + i`` — and sees keys 0 .. that position (lichtung612 blog: the mask is
    added to scores of width ``cache_len + seqlen``). With k_len = q_len this is the
    plain lower triangle (``is_causal=True`` in the qqstock MLA code).
    """
    if k_len < q_len:
        raise ValueError("causal attention needs at least as many keys as queries")
    offset = k_len - q_len
    return np.arange(k_len)[None, :] <= (np.arange(q_len)[:, None] + offset)


def prefill_gqa_causal(q, k, v, cu_seqlens, scale, heads=None):
    """Causal GQA attention of packed variable-length sequences over themselves.

    q [T, Hq, D], k/v [T, Hkv, D]; sequence b occupies rows cu_seqlens[b] ..
    cu_seqlens[b+1]-1 of all three. Row i of a sequence attends keys 0 .. i of the same
    sequence through KV head h // G. ``heads`` optionally restricts the query heads
    computed (others stay zero). Returns out [T, Hq, D] float64.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    total, n_q, _ = q.shape
    n_kv = k.shape[1]
    g = check_grouping(n_q, n_kv)
    cu = np.asarray(cu_seqlens).astype(np.int64)
    if cu[0] != 0 or (np.diff(cu) < 0).any() or cu[-1] != total:
        raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at T")
    out = np.zeros((total, n_q, v.shape[2]), dtype=np.float64)
    head_list = range(n_q) if heads is None else heads
    for b in range(len(cu) - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        n = hi - lo
        if n == 0:
            continue
        allowed = causal_allowed(n, n)
        for h in head_list:
            j = h // g
            out[lo:hi, h] = attend(q[lo:hi, h], k[lo:hi, j], v[lo:hi, j], scale, allowed)
    return out


def default_scale(head_dim):
    """1/sqrt(head_dim): the page's ``/ math.sqrt(self.head_dim)``."""
    return 1.0 / math.sqrt(head_dim)

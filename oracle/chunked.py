"""Chunked prefill over an existing KV cache, for GQA and for MLA (fp64, CPU).

Test infrastructure: only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may use it.

Sources (by page title and section):
  * "模型架构｜MQA & GQA 调研" (lichtung612 blog), section "代码": ``Attention.forward``
    takes ``seqlen`` new tokens at ``start_pos``, writes their keys and values into the cache
    first, reads the cache up to ``start_pos + seqlen`` and adds a mask to scores of width
    ``cache_len + seqlen``: new token i (absolute position start_pos + i) sees cached
    positions 0 .. start_pos + i.
  * qqstock article on DeepSeek MLA, sections 2, 3 and 6 and its code: prefill with
    ``is_causal=True`` over the recombined [nope ‖ rope] query and key; with W_UK absorbed the
    same attention runs on the latent rows [c ‖ kr] with c as the value, and W_UV is applied
    to the result.

A chunk of n_b new tokens of sequence b is packed at rows cu_q[b] .. cu_q[b+1]-1 of the
query; ``start_pos[b]`` is the number of tokens cached before it, and the cache already holds
the chunk (rows start_pos[b] .. start_pos[b] + n_b - 1). With start_pos = 0 and a cache that
holds only the chunk this is ``prefill_gqa_causal``; with n_b = 1 it is one decode step.

Pinned by ``tests/test_oracle_pins.py``: PyTorch's float64 SDPA with an explicit mask, the
prefill and decode oracles at the two ends, the article's ``is_causal`` SDPA path for MLA,
and absorbed = decompressed MLA.
"""

import numpy as np

from .attention import attend, causal_allowed, check_grouping


def _chunks(cu_q, start_pos, s_max):
    cu = np.asarray(cu_q).astype(np.int64)
    start = np.asarray(start_pos).astype(np.int64)
    if cu[0] != 0 or (np.diff(cu) < 0).any() or start.shape != (len(cu) - 1,):
        raise ValueError("cu_q must start at 0 and be non-decreasing, with one start_pos per sequence")
    if (start < 0).any() or (start + np.diff(cu) > s_max).any():
        raise ValueError("every chunk must fit in the cache: 0 <= start_pos, start_pos + n <= S_max")
    return [(int(cu[b]), int(cu[b + 1]), int(start[b])) for b in range(len(cu) - 1)]


def prefill_gqa_chunked(q, k_cache, v_cache, cu_q, start_pos, scale):
    """GQA attention of each sequence's new tokens over its cache, bottom-right causal.

    q [T, Hq, D]; k_cache, v_cache [B, S_max, Hkv, D]; cu_q [B+1]; start_pos [B].
    Returns out [T, Hq, D] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    n_q = q.shape[1]
    n_kv = k_cache.shape[2]
    g = check_grouping(n_q, n_kv)
    out = np.zeros((q.shape[0], n_q, v_cache.shape[3]), dtype=np.float64)
    for b, (lo, hi, start) in enumerate(_chunks(cu_q, start_pos, k_cache.shape[1])):
        n = hi - lo
        if n == 0:
            continue
        keys = start + n
        allowed = causal_allowed(n, keys)
        for h in range(n_q):
            j = h // g
            out[lo:hi, h] = attend(q[lo:hi, h], k_cache[b, :keys, j], v_cache[b, :keys, j], scale, allowed)
    return out


def mla_prefill_absorbed(q_lat, q_rope, c_cache, kr_cache, cu_q, start_pos, scale):
    """Absorbed MLA over a chunk: o_lat[row, h] = Σ_t softmax_t(scale·(q_lat·c_t + q_rope·kr_t)) c_t
    over the visible cached rows t (bottom-right causal).

    q_lat [T, Hq, r], q_rope [T, Hq, dr], c_cache [B, S_max, r], kr_cache [B, S_max, dr].
    Returns o_lat [T, Hq, r] float64.
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    c_cache = np.asarray(c_cache, dtype=np.float64)
    kr_cache = np.asarray(kr_cache, dtype=np.float64)
    out = np.zeros(q_lat.shape, dtype=np.float64)
    for b, (lo, hi, start) in enumerate(_chunks(cu_q, start_pos, c_cache.shape[1])):
        n = hi - lo
        if n == 0:
            continue
        keys = start + n
        allowed = causal_allowed(n, keys)
        k_rows = np.concatenate([c_cache[b, :keys], kr_cache[b, :keys]], axis=1)
        for h in range(q_lat.shape[1]):
            q_rows = np.concatenate([q_lat[lo:hi, h], q_rope[lo:hi, h]], axis=1)
            out[lo:hi, h] = attend(q_rows, k_rows, c_cache[b, :keys], scale, allowed)
    return out


def mla_prefill_naive(q_nope, q_rope, c_cache, kr_cache, w_uk, w_uv, cu_q, start_pos, scale):
    """Decompress-then-attend MLA over a chunk, as the article's code runs it: per head,
    keys [W_UK[h] c_t ‖ kr_t], values W_UV[h] c_t, query [q_nope ‖ q_rope], bottom-right causal.
    Returns out [T, Hq, d_v] float64."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    c_cache = np.asarray(c_cache, dtype=np.float64)
    kr_cache = np.asarray(kr_cache, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    n_q = q_nope.shape[1]
    out = np.zeros((q_nope.shape[0], n_q, w_uv.shape[1]), dtype=np.float64)
    for b, (lo, hi, start) in enumerate(_chunks(cu_q, start_pos, c_cache.shape[1])):
        n = hi - lo
        if n == 0:
            continue
        keys = start + n
        allowed = causal_allowed(n, keys)
        c = c_cache[b, :keys]
        for h in range(n_q):
            k_rows = np.concatenate([c @ w_uk[h].T, kr_cache[b, :keys]], axis=1)
            q_rows = np.concatenate([q_nope[lo:hi, h], q_rope[lo:hi, h]], axis=1)
            out[lo:hi, h] = attend(q_rows, k_rows, c @ w_uv[h].T, scale, allowed)
    return out

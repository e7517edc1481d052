"""Rotary position embedding and the KV-cache append of one decode step (fp64, CPU).

Test infrastructure: only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may use it.

Sources (by page title and section):
  * "模型架构｜MQA & GQA 调研" (lichtung612 blog), section "代码": ``Attention.forward``
    rotates the new query and key with ``apply_rotary_emb(xq, xk, freqs_cis)``, writes the
    rotated key and the value into the cache at ``start_pos`` and only then reads the cache
    up to ``start_pos + seqlen`` (so the decode sees the new token).
  * qqstock article on DeepSeek MLA, section 3 and its ``MultiHeadLatentAttention`` code:
    the decoupled RoPE key (one head, width rope_head_dim) and the per-head rope part of the
    query are rotated with the same ``cis`` table; the latent c is cached unrotated.

Reading (the pages print neither ``apply_rotary_emb`` nor how ``freqs_cis`` is built):
``freqs_cis[p, j]`` is a unit complex number cos φ + i·sin φ for position p and pair j,
passed in as an argument (as ``forward`` receives it); a head vector of width W is viewed
as W/2 complex numbers made of consecutive elements (2j, 2j+1), the layout a complex view
of a trailing axis of 2 gives, and each is multiplied by its table entry. The table is
stored as [positions, W/2, 2] real pairs (cos, sin).

Decode appends one token per sequence: ``positions[b]`` is that sequence's start_pos.
A position outside [0, S_max) appends nothing: the cache is left as it was, the rotated
query row is 0 and the new length is 0 (the decode then returns 0 for that sequence).

Pinned by ``tests/test_oracle_pins.py`` (complex multiplication through
``torch.view_as_complex``, closed forms, norm preservation, the relative-position property
for a table of angles p·θ_j, and brute-force appends).
"""

import numpy as np


def rope_rotate(x, cis):
    """Rotate consecutive pairs of x's last axis: (x0 + i·x1)·(c + i·s).

    x [..., W] (W even), cis [..., W/2, 2] broadcastable against x's pairs.
    """
    x = np.asarray(x, dtype=np.float64)
    cis = np.asarray(cis, dtype=np.float64)
    if x.shape[-1] % 2:
        raise ValueError("the rotated width must be even")
    c, s = cis[..., 0], cis[..., 1]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    re = x0 * c - x1 * s
    im = x0 * s + x1 * c
    return np.stack([re, im], axis=-1).reshape(re.shape[:-1] + (2 * re.shape[-1],))


def _append(q, rot_new, plain_new, positions, freqs_cis, rot_cache, plain_cache):
    """Shared steps of both appends: rotate q and the new key part at their position,
    write the rotated key part and the plain part into the caches at that position."""
    q = np.asarray(q, dtype=np.float64)
    rot_new = np.asarray(rot_new, dtype=np.float64)
    plain_new = np.asarray(plain_new, dtype=np.float64)
    freqs_cis = np.asarray(freqs_cis, dtype=np.float64)
    rot_cache = np.array(rot_cache, dtype=np.float64)        # copies: the inputs stay as they were
    plain_cache = np.array(plain_cache, dtype=np.float64)
    positions = np.asarray(positions).astype(np.int64)
    B = q.shape[0]
    s_max = rot_cache.shape[1]
    q_rot = np.zeros_like(q)
    new_lens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        p = int(positions[b])
        if p < 0 or p >= s_max:
            continue
        cis = freqs_cis[p]                                     # [W/2, 2]
        q_rot[b] = rope_rotate(q[b], cis)
        rot_cache[b, p] = rope_rotate(rot_new[b], cis)
        plain_cache[b, p] = plain_new[b]
        new_lens[b] = p + 1
    return q_rot, rot_cache, plain_cache, new_lens


def kv_append_rope(q, k_new, v_new, positions, freqs_cis, k_cache, v_cache):
    """One GQA decode step's cache write [MQA&GQA "代码"]: the new query and key rotated at
    start_pos, the rotated key and the value written into the cache at that row.

    q [B, Hq, D], k_new/v_new [B, Hkv, D], positions [B], freqs_cis [S_max, D/2, 2],
    k_cache/v_cache [B, S_max, Hkv, D]. Returns (q_rot, k_cache', v_cache', new_lens).
    """
    return _append(q, k_new, v_new, positions, freqs_cis, k_cache, v_cache)


def mla_append_rope(q_rope, c_new, kr_new, positions, freqs_cis, c_cache, kr_cache):
    """One MLA decode step's cache write [MLA section 3]: q_rope and the shared rope key
    rotated at start_pos, kr and the unrotated latent c written at that row.

    q_rope [B, Hq, dr], c_new [B, r], kr_new [B, dr], positions [B],
    freqs_cis [S_max, dr/2, 2], c_cache [B, S_max, r], kr_cache [B, S_max, dr].
    Returns (q_rope_rot, c_cache', kr_cache', new_lens).
    """
    q_rot, kr_cache, c_cache, new_lens = _append(q_rope, kr_new, c_new, positions, freqs_cis, kr_cache, c_cache)
    return q_rot, c_cache, kr_cache, new_lens

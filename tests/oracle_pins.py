"""Checks that pin the CPU oracle to things other than itself.

Each ``check_*`` raises AssertionError on a mismatch. ``test_oracle_pins.py`` runs them
on the real oracle; ``test_oracle_mutations.py`` plants plausible mistakes in the oracle
(on the CPU) and shows that at least one check catches each.

Kinds of pin used:
  * brute force: pure-Python scalar loops (``math.exp``, ``math.fsum``) over K/V heads
    expanded with ``torch.repeat_interleave`` — the library call the lichtung612 blog's
    ``repeat_kv`` docstring names as its equivalent — so the head mapping is not retyped;
  * a library routine: ``torch.nn.functional.scaled_dot_product_attention`` in float64
    on the CPU (with ``is_causal=True`` for prefill, as the qqstock MLA code calls it);
  * closed forms and invariants: one key → that value row; equal keys or scale 0 → the
    mean of the values; a dominant score → its value row; permutation of the keys; affine
    maps of V; the split/merge identity over every contiguous partition;
  * the MLA associativity identity (absorbed = decompressed) and MLA = MQA with key width
    r + dr and V = c (qqstock article, sections 2 and 6).
"""

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

TOL_EXACT = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _expand_heads(x, n_rep, axis):
    """Expand KV heads to query heads with torch.repeat_interleave (library routine)."""
    return torch.repeat_interleave(torch.from_numpy(np.ascontiguousarray(x)), n_rep, dim=axis).numpy()


# ----------------------------------------------------------------------------- brute force

def brute_decode(q, k_cache, v_cache, seq_lens, scale):
    """Scalar-loop decode over per-query-head expanded caches."""
    bsz, n_q, dk = q.shape
    n_rep = n_q // k_cache.shape[2]
    ke = _expand_heads(k_cache, n_rep, 2)
    ve = _expand_heads(v_cache, n_rep, 2)
    dv = ve.shape[3]
    out = np.zeros((bsz, n_q, dv))
    for b in range(bsz):
        s_len = int(seq_lens[b])
        for h in range(n_q):
            if s_len == 0:
                continue
            sc = [scale * math.fsum(float(q[b, h, d]) * float(ke[b, t, h, d]) for d in range(dk))
                  for t in range(s_len)]
            top = max(sc)
            e = [math.exp(x - top) for x in sc]
            z = math.fsum(e)
            for d in range(dv):
                out[b, h, d] = math.fsum(e[t] * float(ve[b, t, h, d]) for t in range(s_len)) / z
    return out


def brute_prefill(q, k, v, cu, scale):
    """Scalar-loop causal prefill: row i of a sequence sees its keys 0..i."""
    total, n_q, dk = q.shape
    n_rep = n_q // k.shape[1]
    ke = _expand_heads(k, n_rep, 1)
    ve = _expand_heads(v, n_rep, 1)
    dv = ve.shape[2]
    out = np.zeros((total, n_q, dv))
    for b in range(len(cu) - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        for i in range(hi - lo):
            for h in range(n_q):
                sc = [scale * math.fsum(float(q[lo + i, h, d]) * float(ke[lo + t, h, d]) for d in range(dk))
                      for t in range(i + 1)]
                top = max(sc)
                e = [math.exp(x - top) for x in sc]
                z = math.fsum(e)
                for d in range(dv):
                    out[lo + i, h, d] = math.fsum(e[t] * float(ve[lo + t, h, d]) for t in range(i + 1)) / z
    return out


def brute_mla_naive(q_nope, q_rope, c, kr, w_uk, w_uv, seq_lens, scale):
    """Scalar-loop decompress-then-attend MLA (k = [W_UK c ‖ kr], v = W_UV c)."""
    bsz, n_q, d_nope = q_nope.shape
    r = c.shape[2]
    dr = kr.shape[2]
    dv = w_uv.shape[1]
    out = np.zeros((bsz, n_q, dv))
    for b in range(bsz):
        s_len = int(seq_lens[b])
        for h in range(n_q):
            if s_len == 0:
                continue
            sc = []
            vals = []
            for t in range(s_len):
                k_nope = [math.fsum(float(w_uk[h, n, i]) * float(c[b, t, i]) for i in range(r))
                          for n in range(d_nope)]
                dot = math.fsum([float(q_nope[b, h, n]) * k_nope[n] for n in range(d_nope)]
                                + [float(q_rope[b, h, i]) * float(kr[b, t, i]) for i in range(dr)])
                sc.append(scale * dot)
                vals.append([math.fsum(float(w_uv[h, e, i]) * float(c[b, t, i]) for i in range(r))
                             for e in range(dv)])
            top = max(sc)
            e = [math.exp(x - top) for x in sc]
            z = math.fsum(e)
            for d in range(dv):
                out[b, h, d] = math.fsum(e[t] * vals[t][d] for t in range(s_len)) / z
    return out


def tiny_decode_case(seed, n_kv, n_q=8, bsz=2, d=6, s_max=11, lens=None, dv=None):
    rng = _rng(seed)
    q = rng.standard_normal((bsz, n_q, d))
    k = rng.standard_normal((bsz, s_max, n_kv, d))
    v = rng.standard_normal((bsz, s_max, n_kv, dv or d))
    if lens is None:
        lens = rng.integers(1, s_max + 1, size=bsz)
    return q, k, v, np.asarray(lens)


def check_decode_brute(decode_gqa):
    for n_kv, lens in ((1, (11, 4)), (2, (1, 9)), (4, (7, 11)), (8, (0, 5))):
        q, k, v, lens = tiny_decode_case(10 + n_kv, n_kv, lens=lens)
        scale = 0.37
        got = decode_gqa(q, k, v, lens, scale)
        ref = brute_decode(q, k, v, lens, scale)
        assert np.abs(got - ref).max() <= TOL_EXACT, (n_kv, np.abs(got - ref).max())


def check_decode_value_width(decode_gqa):
    """K and V widths may differ (MLA uses key width r+dr and value width r)."""
    q, k, v, lens = tiny_decode_case(77, 1, n_q=4, d=7, dv=3, lens=(5, 9))
    got = decode_gqa(q, k, v, lens, 0.5)
    ref = brute_decode(q, k, v, lens, 0.5)
    assert np.abs(got - ref).max() <= TOL_EXACT


def check_prefill_brute(prefill):
    rng = _rng(5)
    lens = [1, 7, 0, 12]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    q = rng.standard_normal((total, 4, 5))
    k = rng.standard_normal((total, 2, 5))
    v = rng.standard_normal((total, 2, 5))
    got = prefill(q, k, v, cu, 0.45)
    ref = brute_prefill(q, k, v, cu, 0.45)
    assert np.abs(got - ref).max() <= TOL_EXACT, np.abs(got - ref).max()


# ----------------------------------------------------------------------------- library

def check_decode_sdpa(decode_gqa):
    """torch SDPA (float64, CPU) over K/V expanded with repeat_interleave."""
    for n_kv in (1, 2, 4, 8):
        q, k, v, lens = tiny_decode_case(40 + n_kv, n_kv, d=16, s_max=33)
        scale = 1.0 / math.sqrt(16)
        got = decode_gqa(q, k, v, lens, scale)
        n_rep = 8 // n_kv
        for b in range(q.shape[0]):
            s_len = int(lens[b])
            kb = torch.repeat_interleave(torch.from_numpy(k[b, :s_len]), n_rep, dim=1).transpose(0, 1)
            vb = torch.repeat_interleave(torch.from_numpy(v[b, :s_len]), n_rep, dim=1).transpose(0, 1)
            qb = torch.from_numpy(q[b])[:, None, :]
            ref = F.scaled_dot_product_attention(qb, kb, vb, scale=scale)[:, 0, :].numpy()
            assert np.abs(got[b] - ref).max() <= TOL_EXACT, (n_kv, b)


def check_prefill_sdpa(prefill):
    rng = _rng(9)
    lens = [33, 1, 64, 17]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    n_q, n_kv, d = 8, 2, 16
    q = rng.standard_normal((total, n_q, d))
    k = rng.standard_normal((total, n_kv, d))
    v = rng.standard_normal((total, n_kv, d))
    got = prefill(q, k, v, cu, 1.0 / math.sqrt(d))
    for b in range(len(lens)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        qb = torch.from_numpy(q[lo:hi]).transpose(0, 1)
        kb = torch.repeat_interleave(torch.from_numpy(k[lo:hi]), n_q // n_kv, dim=1).transpose(0, 1)
        vb = torch.repeat_interleave(torch.from_numpy(v[lo:hi]), n_q // n_kv, dim=1).transpose(0, 1)
        ref = F.scaled_dot_product_attention(qb, kb, vb, is_causal=True).transpose(0, 1).numpy()
        assert np.abs(got[lo:hi] - ref).max() <= TOL_EXACT, b


# ----------------------------------------------------------------------------- closed forms

def check_decode_closed_forms(decode_gqa):
    rng = _rng(3)
    q, k, v, _ = tiny_decode_case(3, 2, s_max=9)
    # one cached token: softmax of one score is 1, so out = V[0] exactly
    out = decode_gqa(q, k, v, np.array([1, 1]), 0.8)
    for b in range(2):
        for h in range(8):
            assert np.array_equal(out[b, h], v[b, 0, h // 4]), (b, h)
    # all keys equal: every score equal, uniform weights → mean of V
    k_same = np.repeat(k[:, :1], 9, axis=1)
    out = decode_gqa(q, k_same, v, np.array([9, 5]), 0.8)
    for b, s_len in ((0, 9), (1, 5)):
        for h in range(8):
            assert np.abs(out[b, h] - v[b, :s_len, h // 4].mean(axis=0)).max() <= TOL_EXACT
    # scale 0: uniform weights as well
    out = decode_gqa(q, k, v, np.array([6, 9]), 0.0)
    for b, s_len in ((0, 6), (1, 9)):
        for h in range(8):
            assert np.abs(out[b, h] - v[b, :s_len, h // 4].mean(axis=0)).max() <= TOL_EXACT
    # a dominant score: key 3 parallel to q with a huge norm → weight 1 on V[3]
    q1 = rng.standard_normal((1, 1, 6))
    k1 = rng.standard_normal((1, 7, 1, 6)) * 1e-3
    k1[0, 3, 0] = q1[0, 0] * 1e4
    v1 = rng.standard_normal((1, 7, 1, 6))
    out = decode_gqa(q1, k1, v1, np.array([7]), 1.0)
    assert np.abs(out[0, 0] - v1[0, 3, 0]).max() <= TOL_EXACT
    # an empty cache gives zeros (the library's defined edge case)
    out = decode_gqa(q, k, v, np.array([0, 3]), 0.8)
    assert np.all(out[0] == 0.0) and np.any(out[1] != 0.0)


def check_prefill_closed_forms(prefill):
    rng = _rng(21)
    lens = [5, 3]
    cu = np.array([0, 5, 8])
    q = rng.standard_normal((8, 4, 6))
    k = rng.standard_normal((8, 1, 6))
    v = rng.standard_normal((8, 1, 6))
    out = prefill(q, k, v, cu, 0.6)
    for b in range(2):
        lo = int(cu[b])
        for h in range(4):
            # row 0 of each sequence sees only key 0
            assert np.array_equal(out[lo, h], v[lo, 0])
    # the last row of a sequence equals decode over the whole sequence as a cache
    from oracle import decode_gqa
    for b in range(2):
        lo, hi = int(cu[b]), int(cu[b + 1])
        dec = decode_gqa(q[hi - 1][None], k[lo:hi][None], v[lo:hi][None], np.array([lens[b]]), 0.6)
        assert np.abs(out[hi - 1] - dec[0]).max() <= TOL_EXACT


def check_decode_invariants(decode_gqa):
    q, k, v, lens = tiny_decode_case(8, 2, s_max=10, lens=(10, 10))
    base = decode_gqa(q, k, v, lens, 0.7)
    perm = _rng(8).permutation(10)
    out = decode_gqa(q, k[:, perm], v[:, perm], lens, 0.7)
    assert np.abs(out - base).max() <= TOL_EXACT
    out = decode_gqa(q, k, 2.5 * v - 1.25, lens, 0.7)
    assert np.abs(out - (2.5 * base - 1.25)).max() <= 1e-11


def check_mha_mqa_endpoints(decode_gqa, repeat_kv):
    # MHA: Hkv = Hq, head h uses its own KV head
    q, k, v, lens = tiny_decode_case(31, 8)
    out = decode_gqa(q, k, v, lens, 0.5)
    for h in range(8):
        one = decode_gqa(q[:, h:h + 1], k[:, :, h:h + 1], v[:, :, h:h + 1], lens, 0.5)
        assert np.abs(out[:, h] - one[:, 0]).max() <= TOL_EXACT
    # MQA: Hkv = 1, every head uses KV head 0
    q, k, v, lens = tiny_decode_case(32, 1)
    out = decode_gqa(q, k, v, lens, 0.5)
    for h in range(8):
        one = decode_gqa(q[:, h:h + 1], k, v, lens, 0.5)
        assert np.abs(out[:, h] - one[:, 0]).max() <= TOL_EXACT
    # GQA equals MHA over repeat_kv-expanded caches
    for n_kv in (2, 4):
        q, k, v, lens = tiny_decode_case(33 + n_kv, n_kv)
        out = decode_gqa(q, k, v, lens, 0.5)
        mha = decode_gqa(q, repeat_kv(k, 8 // n_kv), repeat_kv(v, 8 // n_kv), lens, 0.5)
        assert np.abs(out - mha).max() <= TOL_EXACT


def check_repeat_kv(repeat_kv):
    """The page's expand/reshape equals torch.repeat_interleave on the head axis (its
    docstring says so): query head h holds KV head h // n_rep."""
    x = _rng(4).standard_normal((2, 3, 4, 5))
    for n_rep in (1, 2, 3):
        ref = torch.repeat_interleave(torch.from_numpy(x), n_rep, dim=2).numpy()
        assert np.array_equal(repeat_kv(x, n_rep), ref)


def check_split_merge(attend, attend_partial, lse_merge):
    rng = _rng(12)
    q = rng.standard_normal((3, 8))
    k = rng.standard_normal((6, 8))
    v = rng.standard_normal((6, 5))
    whole = attend(q, k, v, 0.9)
    # every partition of 0..5 into contiguous pieces (2^5 compositions), empty pieces too
    for cuts in itertools.product((0, 1), repeat=5):
        edges = [0] + [i + 1 for i, c in enumerate(cuts) if c] + [6]
        parts = [attend_partial(q, k[a:b], v[a:b], 0.9) for a, b in zip(edges[:-1], edges[1:])]
        parts.append(attend_partial(q, k[:0], v[:0], 0.9))
        got = lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.abs(got - whole).max() <= 1e-13, edges
    # a longer range split at random points, with the lse checked against its definition
    k = rng.standard_normal((300, 8)) * 2
    v = rng.standard_normal((300, 5))
    whole = attend(q, k, v, 0.9)
    edges = [0] + sorted(rng.choice(np.arange(1, 300), 9, replace=False).tolist()) + [300]
    parts = [attend_partial(q, k[a:b], v[a:b], 0.9) for a, b in zip(edges[:-1], edges[1:])]
    got = lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(got - whole).max() <= 1e-13
    for (a, b), (_, lse) in zip(zip(edges[:-1], edges[1:]), parts):
        direct = np.log(np.exp(0.9 * (q @ k[a:b].T)).sum(axis=1))
        assert np.abs(lse - direct).max() <= 1e-12


def mla_case(seed, bsz=2, n_q=3, d_nope=4, r=6, dr=3, dv=5, s_max=7, lens=(7, 3)):
    rng = _rng(seed)
    return dict(
        q_nope=rng.standard_normal((bsz, n_q, d_nope)),
        q_rope=rng.standard_normal((bsz, n_q, dr)),
        c=rng.standard_normal((bsz, s_max, r)),
        kr=rng.standard_normal((bsz, s_max, dr)),
        w_uk=rng.standard_normal((n_q, d_nope, r)) / math.sqrt(r),
        w_uv=rng.standard_normal((n_q, dv, r)) / math.sqrt(r),
        lens=np.asarray(lens),
    )


def check_mla_naive_brute(mla_decode_naive):
    m = mla_case(51)
    scale = 1.0 / math.sqrt(4 + 3)
    got = mla_decode_naive(m["q_nope"], m["q_rope"], m["c"], m["kr"], m["w_uk"], m["w_uv"], m["lens"], scale)
    ref = brute_mla_naive(m["q_nope"], m["q_rope"], m["c"], m["kr"], m["w_uk"], m["w_uv"], m["lens"], scale)
    assert np.abs(got - ref).max() <= TOL_EXACT


def check_mla_absorbed_equals_naive(absorb_query, mla_decode_absorbed, apply_uv, mla_decode_naive):
    for seed, shape in ((61, {}), (62, dict(bsz=3, n_q=16, d_nope=96, r=128, dr=48, dv=96, s_max=40, lens=(40, 1, 23)))):
        m = mla_case(seed, **shape)
        d_nope = m["q_nope"].shape[2]
        dr = m["q_rope"].shape[2]
        scale = 1.0 / math.sqrt(d_nope + dr)
        q_lat = absorb_query(m["q_nope"], m["w_uk"])
        o_lat = mla_decode_absorbed(q_lat, m["q_rope"], m["c"], m["kr"], m["lens"], scale)
        got = apply_uv(o_lat, m["w_uv"])
        ref = mla_decode_naive(m["q_nope"], m["q_rope"], m["c"], m["kr"], m["w_uk"], m["w_uv"], m["lens"], scale)
        assert np.abs(got - ref).max() <= 1e-10, seed


def check_mla_is_mqa(mla_decode_absorbed, decode_gqa):
    """Absorbed MLA is MQA with key [c ‖ kr] (width r+dr) and value c (width r)."""
    m = mla_case(71, n_q=4, r=8, dr=4)
    rng = _rng(71)
    q_lat = rng.standard_normal((2, 4, 8))
    o_lat = mla_decode_absorbed(q_lat, m["q_rope"], m["c"], m["kr"], m["lens"], 0.3)
    q = np.concatenate([q_lat, m["q_rope"]], axis=2)
    kc = np.concatenate([m["c"], m["kr"]], axis=2)[:, :, None, :]
    vc = m["c"][:, :, None, :]
    ref = decode_gqa(q, kc, vc, m["lens"], 0.3)
    assert np.abs(o_lat - ref).max() <= TOL_EXACT


# ----------------------------------------------------------------------------- RoPE + append

def _unit_cis(angles):
    return np.stack([np.cos(angles), np.sin(angles)], axis=-1)


def check_rope_complex(rope_rotate):
    """Consecutive pairs as complex numbers: torch.view_as_complex of a trailing axis of 2,
    times torch.polar(1, φ), the complex multiplication the pages' cis table implies."""
    rng = _rng(81)
    x = rng.standard_normal((3, 4, 10))
    ang = rng.uniform(-math.pi, math.pi, 5)
    xc = torch.view_as_complex(torch.from_numpy(x).reshape(3, 4, 5, 2).contiguous())
    cis = torch.polar(torch.ones(5, dtype=torch.float64), torch.from_numpy(ang))
    ref = torch.view_as_real(xc * cis).reshape(3, 4, 10).numpy()
    got = rope_rotate(x, _unit_cis(ang))
    assert np.abs(got - ref).max() <= TOL_EXACT


def check_rope_closed_forms(rope_rotate):
    rng = _rng(82)
    x = rng.standard_normal((2, 8))
    assert np.array_equal(rope_rotate(x, _unit_cis(np.zeros(4))), x)                 # angle 0
    quarter = np.tile(np.array([0.0, 1.0]), (4, 1))                                   # angle π/2
    want = np.empty_like(x)
    want[:, 0::2], want[:, 1::2] = -x[:, 1::2], x[:, 0::2]
    assert np.array_equal(rope_rotate(x, quarter), want)
    got = rope_rotate(x, _unit_cis(rng.uniform(0, 2 * math.pi, 4)))                  # |z| kept per pair
    assert np.allclose(np.hypot(got[:, 0::2], got[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]), rtol=0, atol=1e-12)


def check_rope_relative_position(rope_rotate):
    """With angles p·θ_j the score of a rotated query and key depends on their offset only."""
    rng = _rng(83)
    w = 16
    theta = 10000.0 ** (-np.arange(w // 2) * 2.0 / w)
    table = lambda p: _unit_cis(p * theta)                       # noqa: E731
    q, k = rng.standard_normal(w), rng.standard_normal(w)
    for m, n, t in ((5, 2, 7), (0, 9, 31), (40, 40, 3)):
        a = rope_rotate(q, table(m)) @ rope_rotate(k, table(n))
        b = rope_rotate(q, table(m + t)) @ rope_rotate(k, table(n + t))
        assert abs(a - b) <= 1e-9 * (1 + abs(a)), (m, n, t)


def _cmul_pairs(vec, cis_row):
    """Scalar loop: pair j of vec times cos + i·sin of row j, with Python complex numbers."""
    out = []
    for j in range(len(vec) // 2):
        z = complex(vec[2 * j], vec[2 * j + 1]) * complex(cis_row[j][0], cis_row[j][1])
        out += [z.real, z.imag]
    return out


def append_case(seed, bsz=4, n_q=4, n_kv=2, d=6, s_max=5, positions=(0, 4, 2, 5)):
    rng = _rng(seed)
    return dict(q=rng.standard_normal((bsz, n_q, d)), k_new=rng.standard_normal((bsz, n_kv, d)),
                v_new=rng.standard_normal((bsz, n_kv, d)), pos=np.asarray(positions),
                cis=_unit_cis(rng.uniform(-math.pi, math.pi, (s_max, d // 2))),
                k=rng.standard_normal((bsz, s_max, n_kv, d)), v=rng.standard_normal((bsz, s_max, n_kv, d)))


def check_append_brute(kv_append_rope):
    a = append_case(84, positions=(0, 4, 2, 5))             # 5 = S_max: nothing appended
    q_rot, k2, v2, lens = kv_append_rope(a["q"], a["k_new"], a["v_new"], a["pos"], a["cis"], a["k"], a["v"])
    bsz, s_max = a["k"].shape[:2]
    for b in range(bsz):
        p = int(a["pos"][b])
        ok = 0 <= p < s_max
        assert lens[b] == (p + 1 if ok else 0)
        for t in range(s_max):
            for j in range(a["k"].shape[2]):
                if ok and t == p:
                    assert np.abs(np.array(_cmul_pairs(a["k_new"][b, j], a["cis"][p])) - k2[b, t, j]).max() <= TOL_EXACT
                    assert list(v2[b, t, j]) == list(a["v_new"][b, j])
                else:
                    assert list(k2[b, t, j]) == list(a["k"][b, t, j])
                    assert list(v2[b, t, j]) == list(a["v"][b, t, j])
        for h in range(a["q"].shape[1]):
            want = _cmul_pairs(a["q"][b, h], a["cis"][p]) if ok else [0.0] * a["q"].shape[2]
            assert np.abs(np.array(want) - q_rot[b, h]).max() <= TOL_EXACT


def check_mla_append_brute(mla_append_rope):
    rng = _rng(85)
    bsz, n_q, r, dr, s_max = 3, 4, 6, 4, 5
    q_rope = rng.standard_normal((bsz, n_q, dr))
    c_new, kr_new = rng.standard_normal((bsz, r)), rng.standard_normal((bsz, dr))
    c, kr = rng.standard_normal((bsz, s_max, r)), rng.standard_normal((bsz, s_max, dr))
    cis = _unit_cis(rng.uniform(-math.pi, math.pi, (s_max, dr // 2)))
    pos = np.asarray([3, -1, 0])
    q_rot, c2, kr2, lens = mla_append_rope(q_rope, c_new, kr_new, pos, cis, c, kr)
    assert list(lens) == [4, 0, 1]
    for b in range(bsz):
        p = int(pos[b])
        for t in range(s_max):
            if t == p:
                assert list(c2[b, t]) == list(c_new[b])                      # c is not rotated
                assert np.abs(np.array(_cmul_pairs(kr_new[b], cis[p])) - kr2[b, t]).max() <= TOL_EXACT
            else:
                assert list(c2[b, t]) == list(c[b, t]) and list(kr2[b, t]) == list(kr[b, t])
        for h in range(n_q):
            want = _cmul_pairs(q_rope[b, h], cis[p]) if p >= 0 else [0.0] * dr
            assert np.abs(np.array(want) - q_rot[b, h]).max() <= TOL_EXACT


# ----------------------------------------------------------------------------- fp8 cache

def check_e4m3_table(e4m3_to_float):
    """All 256 codes against PyTorch's float8_e4m3fn widening (NaN where it gives NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_to_float(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def check_e4m3_closed_forms(e4m3_to_float):
    v = e4m3_to_float(np.array([0x38, 0x7E, 0x01, 0x08, 0xB8, 0x00, 0x80, 0x7F], dtype=np.uint8))
    assert list(v[:7]) == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0, 0.0, -0.0] and np.isnan(v[7])


def fp8_case(seed, bsz=3, n_q=4, n_kv=2, d=8, s_max=9, lens=(9, 4, 0)):
    rng = _rng(seed)
    codes = lambda: rng.integers(0, 0x7F, size=(bsz, s_max, n_kv, d)).astype(np.uint8) | \
        (rng.integers(0, 2, size=(bsz, s_max, n_kv, d)).astype(np.uint8) << 7)    # noqa: E731 (no NaN code)
    return dict(q=rng.standard_normal((bsz, n_q, d)), k=codes(), v=codes(),
                ks=rng.uniform(0.001, 0.01, (bsz, s_max, n_kv)), vs=rng.uniform(0.001, 0.01, (bsz, s_max, n_kv)),
                lens=np.asarray(lens))


def check_fp8_decode_identities(decode_gqa_fp8, e4m3_to_float, decode_gqa):
    c = fp8_case(86)
    ones = np.ones_like(c["ks"])
    # unit scales: the decode over the decoded values
    got = decode_gqa_fp8(c["q"], c["k"], c["v"], ones, ones, c["lens"], 0.01)
    ref = decode_gqa(c["q"], e4m3_to_float(c["k"]), e4m3_to_float(c["v"]), c["lens"], 0.01)
    assert np.abs(got - ref).max() <= TOL_EXACT
    # a uniform V scale scales the output; a uniform K scale is a factor on the softmax scale
    base = decode_gqa_fp8(c["q"], c["k"], c["v"], ones * 0.004, ones, c["lens"], 0.5)
    assert np.abs(decode_gqa_fp8(c["q"], c["k"], c["v"], ones * 0.004, ones * 3.0, c["lens"], 0.5)
                  - 3.0 * base).max() <= TOL_EXACT * 10
    assert np.abs(decode_gqa_fp8(c["q"], c["k"], c["v"], ones, ones, c["lens"], 0.5 * 0.004) - base).max() <= TOL_EXACT
    # per-row scales: brute force, one row at a time
    got = decode_gqa_fp8(c["q"], c["k"], c["v"], c["ks"], c["vs"], c["lens"], 0.3)
    kd = e4m3_to_float(c["k"])
    vd = e4m3_to_float(c["v"])
    for b, s in enumerate(c["lens"]):
        for t in range(int(s)):
            for j in range(kd.shape[2]):
                kd[b, t, j] = [x * c["ks"][b, t, j] for x in kd[b, t, j]]
                vd[b, t, j] = [x * c["vs"][b, t, j] for x in vd[b, t, j]]
    assert np.abs(got - brute_decode(c["q"], kd, vd, c["lens"], 0.3)).max() <= TOL_EXACT


# ----------------------------------------------------------------------------- chunked prefill

def chunk_case(seed, n_q=4, n_kv=2, d=6, s_max=12, chunks=((3, 4), (0, 5), (7, 1), (2, 0))):
    """chunks: (start_pos, n_new) per sequence; the cache holds start_pos + n_new rows."""
    rng = _rng(seed)
    bsz = len(chunks)
    cu = np.concatenate([[0], np.cumsum([n for _, n in chunks])])
    return dict(q=rng.standard_normal((int(cu[-1]), n_q, d)), k=rng.standard_normal((bsz, s_max, n_kv, d)),
                v=rng.standard_normal((bsz, s_max, n_kv, d)), cu=cu, start=np.array([s for s, _ in chunks]))


def check_chunked_sdpa(prefill_gqa_chunked):
    """torch SDPA in float64 over repeat_interleave'd heads, with the mask written as the rule
    'new token i of a chunk at start_pos sees cached columns 0 .. start_pos + i'."""
    c = chunk_case(87)
    scale = 0.37
    got = prefill_gqa_chunked(c["q"], c["k"], c["v"], c["cu"], c["start"], scale)
    g = c["q"].shape[1] // c["k"].shape[2]
    for b in range(len(c["start"])):
        lo, hi, s = int(c["cu"][b]), int(c["cu"][b + 1]), int(c["start"][b])
        if hi == lo:
            continue
        n, keys = hi - lo, s + hi - lo
        q = torch.from_numpy(c["q"][lo:hi]).transpose(0, 1)                              # [Hq, n, D]
        k = torch.from_numpy(c["k"][b, :keys]).repeat_interleave(g, dim=1).transpose(0, 1)
        v = torch.from_numpy(c["v"][b, :keys]).repeat_interleave(g, dim=1).transpose(0, 1)
        mask = torch.tensor([[col <= s + row for col in range(keys)] for row in range(n)])
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale).transpose(0, 1).numpy()
        assert np.abs(got[lo:hi] - ref).max() <= TOL_EXACT, b


def check_chunked_ends(prefill_gqa_chunked, prefill_gqa_causal, decode_gqa):
    """start_pos = 0 with the chunk as the whole cache is the causal prefill; each new token
    is the decode step over the cache up to and including itself."""
    c = chunk_case(88, chunks=((0, 5), (0, 3)))
    k_packed = np.concatenate([c["k"][0, :5], c["k"][1, :3]])
    v_packed = np.concatenate([c["v"][0, :5], c["v"][1, :3]])
    got = prefill_gqa_chunked(c["q"], c["k"], c["v"], c["cu"], c["start"], 0.5)
    assert np.abs(got - prefill_gqa_causal(c["q"], k_packed, v_packed, c["cu"], 0.5)).max() <= TOL_EXACT
    c = chunk_case(89)
    got = prefill_gqa_chunked(c["q"], c["k"], c["v"], c["cu"], c["start"], 0.5)
    for b in range(len(c["start"])):
        for i in range(int(c["cu"][b + 1] - c["cu"][b])):
            row = int(c["cu"][b]) + i
            lens = np.zeros(len(c["start"]), dtype=np.int64)
            lens[b] = c["start"][b] + i + 1
            dec = decode_gqa(np.broadcast_to(c["q"][row], (len(lens),) + c["q"].shape[1:]), c["k"], c["v"], lens, 0.5)
            assert np.abs(got[row] - dec[b]).max() <= TOL_EXACT, (b, i)


def check_mla_chunked(mla_prefill_absorbed, mla_prefill_naive, absorb_query, apply_uv, mla_decode_absorbed):
    rng = _rng(90)
    n_q, d_nope, r, dr, dv, s_max = 3, 4, 6, 4, 5, 10
    chunks = ((4, 3), (0, 6), (9, 1))
    cu = np.concatenate([[0], np.cumsum([n for _, n in chunks])])
    start = np.array([s for s, _ in chunks])
    T, bsz = int(cu[-1]), len(chunks)
    q_nope, q_rope = rng.standard_normal((T, n_q, d_nope)), rng.standard_normal((T, n_q, dr))
    c, kr = rng.standard_normal((bsz, s_max, r)), rng.standard_normal((bsz, s_max, dr))
    w_uk, w_uv = rng.standard_normal((n_q, d_nope, r)) / 3, rng.standard_normal((n_q, dv, r)) / 3
    scale = 1.0 / math.sqrt(d_nope + dr)
    naive = mla_prefill_naive(q_nope, q_rope, c, kr, w_uk, w_uv, cu, start, scale)
    # absorbed = decompressed (associativity), through the pinned absorption steps
    q_lat = absorb_query(q_nope, w_uk)                 # the packed rows play the batch axis
    o_lat = mla_prefill_absorbed(q_lat, q_rope, c, kr, cu, start, scale)
    assert np.abs(apply_uv(o_lat, w_uv) - naive).max() <= 1e-10
    # each new token is an absorbed decode step over the cache up to itself
    for b in range(bsz):
        for i in range(int(cu[b + 1] - cu[b])):
            row = int(cu[b]) + i
            lens = np.array([start[b] + i + 1])
            dec = mla_decode_absorbed(q_lat[row][None], q_rope[row][None], c[b][None], kr[b][None], lens, scale)
            assert np.abs(o_lat[row] - dec[0]).max() <= TOL_EXACT, (b, i)
    # the article's own path for a whole prompt: SDPA with is_causal over the recombined heads
    b = 1
    lo, hi = int(cu[b]), int(cu[b + 1])
    cb = torch.from_numpy(c[b, :hi - lo])
    k = torch.stack([torch.cat([cb @ torch.from_numpy(w_uk[h]).T, torch.from_numpy(kr[b, :hi - lo])], 1)
                     for h in range(n_q)])
    v = torch.stack([cb @ torch.from_numpy(w_uv[h]).T for h in range(n_q)])
    q = torch.from_numpy(np.concatenate([q_nope[lo:hi], q_rope[lo:hi]], axis=2)).transpose(0, 1)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(0, 1).numpy()
    assert np.abs(naive[lo:hi] - ref).max() <= TOL_EXACT

"""The decode step's cache write fused with RoPE (attn_kv_append_rope, attn_mla_append_rope)
against the fp64 CPU oracle, then the decode over the appended cache.

Tolerances follow from the arithmetic, per element: a rotated value y = x0·c − x1·s (or
x0·s + x1·c) is formed in fp32 from exact inputs, so it is within γ = 3·2⁻²⁴·(|x0·c| + |x1·s|)
of the exact value; bf16 outputs add one rounding, 2⁻⁸·(|y| + γ). Copied values (v, c) and
every cache row that is not appended must be bit-identical; new lengths exact.
"""

import math

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _rot_bound(x, cis, positions, bf16):
    """Per-element bound for the rotated rows of x [B, H, W] at positions (valid rows only)."""
    b_idx = np.clip(positions, 0, cis.shape[0] - 1)
    c = np.abs(cis[b_idx, :, 0])[:, None, :]                     # [B, 1, W/2]
    s = np.abs(cis[b_idx, :, 1])[:, None, :]
    ax0, ax1 = np.abs(x[..., 0::2]), np.abs(x[..., 1::2])
    mag = np.empty_like(x)
    mag[..., 0::2] = ax0 * c + ax1 * s
    mag[..., 1::2] = ax0 * s + ax1 * c
    gamma = 3 * 2.0 ** -24 * mag
    return gamma, (lambda y: 2.0 ** -8 * (np.abs(y) + gamma) + gamma) if bf16 else (lambda y: gamma)


def _positions(B, s_max, seed, invalid=()):
    p = np.random.default_rng(seed).integers(0, s_max, size=B).astype(np.int32)
    for i, v in enumerate(invalid):
        p[i] = v
    return p


def _check_gqa(B, Hq, Hkv, D, s_max, dtype, seed, invalid=(), in_place=False):
    new = W.append_inputs(B, Hq, Hkv, D, s_max, DEV, seed, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device=DEV).manual_seed(seed + 1)
    k_cache = torch.randn((B, s_max, Hkv, D), generator=g, device=DEV).to(tdt)
    v_cache = torch.randn((B, s_max, Hkv, D), generator=g, device=DEV).to(tdt)
    pos = _positions(B, s_max, seed, invalid)
    k0, v0 = to_f64(k_cache), to_f64(v_cache)
    q0 = to_f64(new["q"])
    q_out = new["q"] if in_place else None
    got_q, lens = mk.kv_append_rope(new["q"], new["k_new"], new["v_new"], torch.from_numpy(pos).to(DEV),
                                    new["freqs_cis"], k_cache, v_cache, q_out=q_out)
    torch.cuda.synchronize()
    cis = to_f64(new["freqs_cis"])
    ref_q, ref_k, ref_v, ref_lens = oracle.kv_append_rope(q0, to_f64(new["k_new"]), to_f64(new["v_new"]), pos, cis,
                                                          k0, v0)
    assert np.array_equal(lens.cpu().numpy(), ref_lens)
    valid = (pos >= 0) & (pos < s_max)
    _, qb = _rot_bound(q0, cis, pos, dtype == "bf16")
    gq = to_f64(got_q)
    assert np.all(np.abs(gq - ref_q)[valid] <= qb(ref_q)[valid])
    assert np.all(gq[~valid] == 0)
    _, kb = _rot_bound(to_f64(new["k_new"]), cis, pos, dtype == "bf16")
    gk, gv = to_f64(k_cache), to_f64(v_cache)
    rows = np.clip(pos, 0, s_max - 1)
    ref_rows = ref_k[np.arange(B), rows]                         # [B, Hkv, D]
    k_bound = kb(ref_rows)
    for b in range(B):
        if valid[b]:
            p = pos[b]
            assert np.all(np.abs(gk[b, p] - ref_rows[b]) <= k_bound[b])
            rest = np.ones(s_max, bool)
            rest[p] = False
            assert np.array_equal(gk[b, rest], k0[b, rest])
        else:
            assert np.array_equal(gk[b], k0[b])
    assert np.array_equal(gv, ref_v)                 # the value row is copied, everything else untouched
    return new, pos


@pytest.mark.parametrize("B,Hq,Hkv,D,dtype", [(32, 8, 4, 96, "bf16"), (4, 32, 8, 128, "bf16"), (5, 8, 2, 64, "fp32"),
                                              (3, 4, 4, 8, "bf16"), (2, 2, 1, 4, "fp32")])
def test_kv_append_rope(B, Hq, Hkv, D, dtype):
    _check_gqa(B, Hq, Hkv, D, 64, dtype, 31 + D, invalid=(-1, 64) if B > 2 else ())


def test_kv_append_rope_in_place_query():
    _check_gqa(6, 8, 4, 96, 33, "bf16", 77, in_place=True)


def test_kv_append_rope_every_position():
    # a cache of 17 rows, one sequence per row, plus one past the end
    B = 18
    new = W.append_inputs(B, 8, 4, 96, 17, DEV, 5)
    k = torch.zeros((B, 17, 4, 96), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros_like(k)
    pos = torch.arange(B, dtype=torch.int32, device=DEV)
    _, lens = mk.kv_append_rope(new["q"], new["k_new"], new["v_new"], pos, new["freqs_cis"], k, v)
    torch.cuda.synchronize()
    assert lens.tolist() == list(range(1, 18)) + [0]
    for b in range(17):
        assert torch.equal(v[b, b], new["v_new"][b])
        assert int(v[b].count_nonzero()) == int(new["v_new"][b].count_nonzero())
    assert int(v[17].count_nonzero()) == 0 and int(k[17].count_nonzero()) == 0


def test_mla_append_rope():
    B, Hq, r, dr, s_max = 9, 16, 128, 48, 40
    new = W.append_inputs(B, Hq, 1, dr, s_max, DEV, 41)
    g = torch.Generator(device=DEV).manual_seed(42)
    c_new = torch.randn((B, r), generator=g, device=DEV).to(torch.bfloat16)
    kr_new = new["k_new"][:, 0].contiguous()
    c_cache = torch.randn((B, s_max, r), generator=g, device=DEV).to(torch.bfloat16)
    kr_cache = torch.randn((B, s_max, dr), generator=g, device=DEV).to(torch.bfloat16)
    pos = _positions(B, s_max, 43, invalid=(s_max, -3))
    c0, kr0, q0 = to_f64(c_cache), to_f64(kr_cache), to_f64(new["q"])
    got_q, lens = mk.mla_append_rope(new["q"], c_new, kr_new, torch.from_numpy(pos).to(DEV), new["freqs_cis"],
                                     c_cache, kr_cache)
    torch.cuda.synchronize()
    cis = to_f64(new["freqs_cis"])
    ref_q, ref_c, ref_kr, ref_lens = oracle.mla_append_rope(q0, to_f64(c_new), to_f64(kr_new), pos, cis, c0, kr0)
    assert np.array_equal(lens.cpu().numpy(), ref_lens)
    valid = (pos >= 0) & (pos < s_max)
    _, qb = _rot_bound(q0, cis, pos, True)
    gq = to_f64(got_q)
    assert np.all(np.abs(gq - ref_q)[valid] <= qb(ref_q)[valid]) and np.all(gq[~valid] == 0)
    assert np.array_equal(to_f64(c_cache), ref_c)
    _, kb = _rot_bound(to_f64(kr_new)[:, None, :], cis, pos, True)
    gkr = to_f64(kr_cache)
    ref_rows = ref_kr[np.arange(B), np.clip(pos, 0, s_max - 1)][:, None, :]   # [B, 1, dr]
    kr_bound = kb(ref_rows)
    for b in range(B):
        if valid[b]:
            p = pos[b]
            assert np.all(np.abs(gkr[b, p] - ref_rows[b, 0]) <= kr_bound[b, 0])
            rest = np.ones(s_max, bool)
            rest[p] = False
            assert np.array_equal(gkr[b, rest], kr0[b, rest])
        else:
            assert np.array_equal(gkr[b], kr0[b])


def test_append_then_decode():
    """A MiniMind-shaped decode step: append the new token at each sequence's length, then
    decode over the cache that now holds it, against the oracle doing the same in fp64."""
    w = W.MINIMIND_GQA
    s_max = 2049
    base = W.decode_inputs(W.DecodeWorkload("append_step", 1, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, s_max,
                                            "bf16", length_range=(512, 2048), sub=3), DEV)
    new = W.append_inputs(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, s_max, DEV, 91)
    k_cache, v_cache = base["k_cache"], base["v_cache"]
    k0, v0 = to_f64(k_cache), to_f64(v_cache)
    pos = base["seq_lens"]                                       # the new token goes after the cached ones
    q_rot, lens = mk.kv_append_rope(new["q"], new["k_new"], new["v_new"], pos, new["freqs_cis"], k_cache, v_cache)
    out = mk.decode_gqa(q_rot, k_cache, v_cache, lens, scale=w.scale)
    torch.cuda.synchronize()
    p = pos.cpu().numpy()
    cis = to_f64(new["freqs_cis"])
    q0 = to_f64(new["q"])
    rq, rk, rv, rl = oracle.kv_append_rope(q0, to_f64(new["k_new"]), to_f64(new["v_new"]), p, cis, k0, v0)
    ref = oracle.decode_gqa(rq, rk, rv, rl, w.scale)
    # the bf16 q_rot and new key row move each score by at most δ (see module docstring)
    _, qb = _rot_bound(q0, cis, p, True)
    _, kb = _rot_bound(to_f64(new["k_new"]), cis, p, True)
    dq, dk = qb(rq), kb(rk[np.arange(w.batch), p])
    g = w.n_q_heads // w.n_kv_heads
    tol = np.zeros_like(ref)
    for b in range(w.batch):
        s = int(rl[b])
        for j in range(w.n_kv_heads):
            kmax = np.abs(rk[b, :s, j]).max()
            vmax = np.abs(rv[b, :s, j]).max()
            for h in range(j * g, (j + 1) * g):
                delta = w.scale * (dq[b, h].sum() * kmax + np.abs(rq[b, h]) @ dk[b, j])
                tol[b, h] = math.expm1(2 * delta) * vmax + 3e-3
    assert np.all(np.abs(to_f64(out) - ref) <= tol)

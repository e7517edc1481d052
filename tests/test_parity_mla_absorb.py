"""The MLA up-projections around the absorbed decode (W_UK folded into the query, W_UV applied
to the latent output) and the whole three-launch decode step, against the fp64 CPU oracle.

Tolerances follow from the arithmetic, per element:
  - q_lat: fp32 sums of d_nope products rounded to bf16, so |got − x| ≤ 2^-8·|x| + γ with
    γ = d_nope·2^-24·Σ_n |q_n·w_n| (fp32 accumulation) plus the rounding of that error.
  - out = W_UV·o_lat in fp32: |got − x| ≤ r·2^-24·Σ_r |w_r·o_r|.
  - the full step against the decompress-then-attend oracle: the bf16 q_lat moves each score
    by at most δ = scale·Σ_r |q_lat_r − x_r|·|c_r|, which moves the latent average by at most
    (e^{2δ} − 1)·max|c|; add the decode's 3e-3 and map through Σ_r |W_UV[h, v, r]|.
"""

import math

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from tests import mla_bounds as mb
from workloads import to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
U_F32 = mb.U_F32


def _rand(shape, seed, std=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * std).to(torch.bfloat16)


_absorb_bound = mb.absorb_bound


@pytest.mark.parametrize("B,H,dn,r", [(1, 16, 96, 128), (17, 16, 96, 128), (33, 3, 1, 32), (5, 128, 96, 128),
                                      (16, 2, 512, 256), (7, 4, 128, 96), (9, 2, 300, 224)])
def test_absorb_query(B, H, dn, r):
    qn = _rand((B, H, dn), 11 + B)
    wuk = _rand((H, dn, r), 12 + H, std=1 / math.sqrt(128))
    got = mk.mla_absorb_query(qn, wuk)
    torch.cuda.synchronize()
    q64, w64 = to_f64(qn), to_f64(wuk)
    ref = oracle.absorb_query(q64, w64)
    err = np.abs(to_f64(got) - ref)
    assert np.all(err <= _absorb_bound(q64, w64, ref))


def test_absorb_query_exact_products():
    # one-hot queries pick a row of W_UK: every sum has one non-zero term, so q_lat is that
    # bf16 row exactly
    B, H, dn, r = 4, 3, 96, 128
    qn = torch.zeros((B, H, dn), dtype=torch.bfloat16, device=DEV)
    for b in range(B):
        for h in range(H):
            qn[b, h, (7 * b + 13 * h) % dn] = 1.0
    wuk = _rand((H, dn, r), 5)
    got = mk.mla_absorb_query(qn, wuk)
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(H):
            assert torch.equal(got[b, h], wuk[h, (7 * b + 13 * h) % dn])


@pytest.mark.parametrize("B,H,r,dv", [(1, 16, 128, 96), (17, 16, 128, 96), (33, 3, 32, 1), (5, 128, 128, 128),
                                      (16, 2, 256, 256), (3, 5, 96, 130), (9, 2, 224, 7)])
def test_apply_uv(B, H, r, dv):
    g = torch.Generator(device=DEV).manual_seed(3 + B + H)
    o = torch.randn((B, H, r), generator=g, device=DEV) * 0.5
    wuv = _rand((H, dv, r), 4 + r, std=1 / math.sqrt(128))
    got = mk.mla_apply_uv(o, wuv)
    torch.cuda.synchronize()
    o64, w64 = to_f64(o), to_f64(wuv)
    ref = oracle.apply_uv(o64, w64)
    bound = r * U_F32 * np.einsum("hvr,bhr->bhv", np.abs(w64), np.abs(o64)) + 1e-30
    err = np.abs(to_f64(got) - ref)
    assert np.all(err <= bound)
    assert err.max() <= 1e-5


def _full_step_tolerance(inp, scale):
    return mb.full_step_tolerance(inp, scale, oracle)


@pytest.mark.parametrize("lens,hq,n_split", [((0, 1, 127, 128, 129, 1000, 2049), 16, 0),
                                             ((300, 5, 2049, 64), 64, 3),
                                             ((1,) * 3 + (700,) * 14, 16, 0)])
def test_full_mla_step_against_decompressed_attention(lens, hq, n_split):
    w = W.MlaWorkload("mla_step", 3, len(lens), hq, 96, 128, 48, 96, max(lens), lengths=lens, sub=21)
    inp = W.mla_inputs(w, DEV)
    out = mk.decode_mla(inp["q_nope"], inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["w_uk"], inp["w_uv"],
                        inp["seq_lens"], w.scale, n_split=n_split)
    torch.cuda.synchronize()
    ref = oracle.mla_decode_naive(to_f64(inp["q_nope"]), to_f64(inp["q_rope"]), to_f64(inp["c_cache"]),
                                  to_f64(inp["kr_cache"]), to_f64(inp["w_uk"]), to_f64(inp["w_uv"]),
                                  inp["seq_lens"].cpu().numpy(), w.scale)
    err = np.abs(to_f64(out) - ref)
    assert np.all(err <= _full_step_tolerance(inp, w.scale))
    empty = torch.tensor([s == 0 for s in lens], device=DEV)
    assert torch.all(out[empty] == 0)


def test_full_step_is_the_three_calls():
    lens = (10, 400, 3000)
    w = W.MlaWorkload("mla_step3", 3, len(lens), 32, 96, 128, 48, 96, 3000, lengths=lens, sub=22)
    inp = W.mla_inputs(w, DEV)
    out = mk.decode_mla(inp["q_nope"], inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["w_uk"], inp["w_uv"],
                        inp["seq_lens"], w.scale)
    q_lat = mk.mla_absorb_query(inp["q_nope"], inp["w_uk"])
    o_lat = mk.decode_mla_absorbed(q_lat, inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["seq_lens"], w.scale)
    out2 = mk.mla_apply_uv(o_lat, inp["w_uv"])
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    mk.check_status()


def test_full_mla_step_at_the_bench_size():
    """The bench's MLA step (B=64, S=4096, 16 heads) in its launch configuration; every
    sequence's outputs against the decompress-then-attend oracle, eight sequences at a time."""
    w = W.MINIMIND_MLA
    inp = W.mla_inputs(w, DEV)
    out = mk.decode_mla(inp["q_nope"], inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["w_uk"], inp["w_uv"],
                        inp["seq_lens"], w.scale)
    torch.cuda.synchronize()
    for b0 in range(0, w.batch, 8):
        pick = list(range(b0, min(b0 + 8, w.batch)))
        sub = {k: (v[pick] if k not in ("w_uk", "w_uv") else v) for k, v in inp.items()}
        ref = oracle.mla_decode_naive(to_f64(sub["q_nope"]), to_f64(sub["q_rope"]), to_f64(sub["c_cache"]),
                                      to_f64(sub["kr_cache"]), to_f64(sub["w_uk"]), to_f64(sub["w_uv"]),
                                      sub["seq_lens"].cpu().numpy(), w.scale)
        err = np.abs(to_f64(out[pick]) - ref)
        assert np.all(err <= _full_step_tolerance(sub, w.scale)), pick


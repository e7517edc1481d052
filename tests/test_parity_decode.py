"""GQA/MHA/MQA decode and the LSE merge on the GPU against the fp64 CPU oracle.

Tolerances (max |Δ| over every output element): 1e-5 for the fp32 cache, 3e-3 for the
bf16 caches (fp32 accumulation and fp32 output in both cases).
"""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 3e-3
DEV = "cuda"


def _oracle_decode(inp, scale, batches=None):
    q = to_f64(inp["q"])
    lens = inp["seq_lens"].cpu().numpy()
    k, v = inp["k_cache"], inp["v_cache"]
    B, Hq, D = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in (range(B) if batches is None else batches):
        s = int(lens[b])
        kb = to_f64(k[b, :s])
        vb = to_f64(v[b, :s])
        for j in range(Hkv):
            out[b, j * g:(j + 1) * g] = oracle.attend(q[b, j * g:(j + 1) * g], kb[:, j], vb[:, j], scale)
    return out


def _max_err(got, ref, batches=None):
    g = got.detach().cpu().double().numpy()
    if batches is not None:
        g, ref = g[list(batches)], ref[list(batches)]
    return float(np.abs(g - ref).max())


@pytest.mark.parametrize("hkv", [2, 8, 1])
@pytest.mark.parametrize("n_split", [0, 1, 2, 3, 7])
def test_tiny_fp32(hkv, n_split):
    w = W.TINY_FP32[hkv]
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale,
                        n_split=n_split)
    torch.cuda.synchronize()
    ref = oracle.decode_gqa(to_f64(inp["q"]), to_f64(inp["k_cache"]), to_f64(inp["v_cache"]),
                            inp["seq_lens"].cpu().numpy(), w.scale)
    assert _max_err(out, ref) <= TOL_F32


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 8), (8, 1), (32, 1), (12, 4), (6, 2), (64, 2)])
def test_shapes_and_ragged_lengths(dtype, D, hq, hkv):
    # lengths cover: empty, one token, one short of a tile, a ragged tail, and S_max
    lens = (0, 1, 127, 129, 300, 517)
    w = W.DecodeWorkload("ragged", 0, len(lens), hq, hkv, D, 517, dtype, lengths=lens, sub=7)
    inp = W.decode_inputs(w, DEV)
    tol = TOL_F32 if dtype == "fp32" else TOL_BF16
    ref = _oracle_decode(inp, w.scale)
    for n_split in (0, 1, 5):
        out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale,
                            n_split=n_split)
        torch.cuda.synchronize()
        assert _max_err(out, ref) <= tol, n_split
        assert torch.all(out[0] == 0)


def test_single_token_is_v0():
    w = W.DecodeWorkload("one", 0, 3, 8, 2, 128, 64, "bf16", lengths=(1, 1, 1))
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"])
    v0 = inp["v_cache"][:, 0].float().repeat_interleave(4, dim=1)
    assert torch.equal(out, v0)


def test_more_splits_than_tiles():
    w = W.DecodeWorkload("few", 0, 2, 8, 2, 64, 200, "fp32", lengths=(3, 200))
    inp = W.decode_inputs(w, DEV)
    ref = _oracle_decode(inp, w.scale)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], n_split=64)
    torch.cuda.synchronize()
    assert _max_err(out, ref) <= TOL_F32


def test_max_s_bound_smaller_than_capacity():
    w = W.DecodeWorkload("bound", 0, 4, 16, 4, 128, 4096, "bf16", lengths=(700, 5, 1000, 999))
    inp = W.decode_inputs(w, DEV)
    ref = _oracle_decode(inp, w.scale)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], max_s=1000)
    torch.cuda.synchronize()
    assert _max_err(out, ref) <= TOL_BF16


def test_deterministic_and_stream_ordered_workspace():
    w = W.MINIMIND_GQA
    inp = W.decode_inputs(w, DEV)
    n = 2
    ws = torch.zeros(mk.decode_gqa_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.s_max,
                                                  mk.ATTN_BF16, n), dtype=torch.uint8, device=DEV)
    inp2 = W.decode_inputs(w, DEV, seed=w.seed + 5)
    a = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], n_split=n, workspace=ws)
    b = mk.decode_gqa(inp2["q"], inp2["k_cache"], inp2["v_cache"], inp2["seq_lens"], n_split=n, workspace=ws)
    a2 = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], n_split=n, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, a2)
    assert _max_err(b, _oracle_decode(inp2, w.scale)) <= TOL_BF16


def test_minimind_gqa_full():
    w = W.MINIMIND_GQA
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale,
                        max_s=int(inp["seq_lens"].max()))
    torch.cuda.synchronize()
    assert _max_err(out, _oracle_decode(inp, w.scale)) <= TOL_BF16


@pytest.mark.parametrize("hkv", [8, 1, 32])
def test_llama3_8b_full(hkv):
    w = W.LLAMA3_8B[hkv]
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale)
    torch.cuda.synchronize()
    # every output; the oracle widens one sequence's cache at a time (MHA holds 8 GiB of it)
    ref = _oracle_decode(inp, w.scale)
    assert _max_err(out, ref) <= TOL_BF16
    del inp
    torch.cuda.empty_cache()


def test_merge_partials_against_oracle():
    g = torch.Generator(device=DEV)
    g.manual_seed(77)
    rows, n, dv = 37, 9, 128
    o = torch.randn((rows, n, dv), generator=g, device=DEV)
    lse = torch.randn((rows, n), generator=g, device=DEV) * 5
    lse[3, :] = float("-inf")            # a row with only empty pieces
    lse[5, ::2] = float("-inf")          # some empty pieces
    out = mk.merge_partials(o, lse)
    torch.cuda.synchronize()
    on, ln = to_f64(o), to_f64(lse)
    for r in range(rows):
        ref = oracle.lse_merge(on[r][:, None, :], ln[r][:, None])[0]
        assert np.abs(out[r].cpu().double().numpy() - ref).max() <= 1e-5
    assert torch.all(out[3] == 0)


def _bf16_weight_bound(inp, hq, hkv, residual=False):
    """Per output element, what bf16 weights allow in the decode: each weight p is rounded to
    nearest (p' = p·(1 + e), |e| <= 2^-8) and O' = Σ p' v / Σ p' normalises by the rounded
    weights, so O' - O = Σ w e (v - O) / (1 + Σ w e) with w the exact weights: at most
    2^-8 · (max v - min v) over the sequence's keys (times 1 + 2^-7). The tensor-core form keeps
    each weight's bf16 residual as well (relative error near 2^-16); a sixteenth of the bound
    is used for it. Plus a margin for the fp32 arithmetic."""
    v = to_f64(inp["v_cache"])                                     # [B, S_max, Hkv, D]
    lens = inp["seq_lens"].cpu().numpy()
    B, _, Hkv, D = v.shape
    spread = np.zeros((B, Hkv, D))
    for b in range(B):
        s = int(lens[b])
        if s > 0:
            spread[b] = v[b, :s].max(axis=0) - v[b, :s].min(axis=0)
    bound = 2.0 ** -8 * (1 + 2.0 ** -7) * np.repeat(spread, hq // hkv, axis=1)
    return (bound / 16 if residual else bound) + 1e-5


@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 1)])
def test_sharp_weights_within_the_bf16_weight_bound(hq, hkv):
    """A large scale (0.5) concentrates the weights on a few keys, so their bf16 rounding no
    longer averages out (above the 3e-3 that holds at the pages' scale). Every element against
    the derived bound: the register-MMA decode (Hkv = 2) with bf16 weights, the tensor-core form
    (MQA here) with their residual."""
    w = W.DecodeWorkload("decode_sharp", 1, 4, hq, hkv, 128, 700, "bf16", lengths=(700, 300, 129, 1), sub=60)
    inp = W.decode_inputs(w, DEV)
    scale = 0.5
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=scale)
    torch.cuda.synchronize()
    err = np.abs(to_f64(out) - _oracle_decode(inp, scale))
    bound = _bf16_weight_bound(inp, hq, hkv, residual=hkv == 1)
    assert bool((err <= bound).all()), float((err - bound).max())


@pytest.mark.parametrize("hq,hkv,d,B", [(32, 4, 128, 600), (32, 8, 128, 1200), (8, 4, 96, 2000), (32, 1, 128, 1500)])
def test_large_batches(hq, hkv, d, B):
    """Batches past what the deepest ring leaves room for: the kernel keeps 8 bytes of tables
    a sequence in shared memory beside its ring, and runs a two-stage ring where the default
    depth would not fit (here past 402, 930 and 1834 sequences; MQA at D = 128 past 706 on the
    stream kernel). Short ragged lengths (0-48 keys, where bf16 weights do not average out):
    every output within the derived bound."""
    w = W.DecodeWorkload("decode_large_b", 1, B, hq, hkv, d, 48, "bf16", length_range=(0, 48), sub=61)
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale)
    torch.cuda.synchronize()
    mk.check_status()
    err = np.abs(to_f64(out) - _oracle_decode(inp, w.scale))
    bound = _bf16_weight_bound(inp, hq, hkv)
    assert bool((err <= bound).all()), float((err - bound).max())


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1)])
def test_long_context(hq, hkv):
    """131072 cached tokens (and a ragged 70001): the split plan's tile counts run to thousands
    per segment; every output compared (register-MMA GQA, and MQA on the tensor cores)."""
    w = W.DecodeWorkload("decode_128k", 1, 2, hq, hkv, 128, 131072, "bf16", lengths=(131072, 70001), sub=62)
    inp = W.decode_inputs(w, DEV)
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=w.scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert _max_err(out, _oracle_decode(inp, w.scale)) <= TOL_BF16

"""Decode on the tcgen05 tensor cores (16 or more query heads per cached row: wide GQA and
MQA at D = 128, and MLA) against the fp64 CPU oracle, max |Δ| ≤ 3e-3 on bf16 inputs.

Covers every mode of the kernel's work split (one block per segment, a balanced split with
shared segments merged in-kernel, more blocks than tiles), ragged and empty sequences, the
rescale of the running reference when scores keep growing along the cache, and repeat calls
on one workspace (its arrival counters must come back to zero).
"""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

TOL = 3e-3
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


def _err(got, ref):
    return float(np.abs(got.detach().cpu().double().numpy() - ref).max())


def _decode(inp, scale, **kw):
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=scale, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hq,hkv", [(32, 1), (16, 1), (32, 2), (64, 1), (48, 3), (128, 4)])
def test_gqa_wide_groups_ragged(hq, hkv):
    # lengths: empty, one token, a tile boundary on each side, several tiles with a tail
    lens = (0, 1, 127, 128, 129, 300, 1000, 2049)
    w = W.DecodeWorkload("tc_ragged", 0, len(lens), hq, hkv, 128, 2049, "bf16", lengths=lens, sub=11)
    inp = W.decode_inputs(w, DEV)
    ref = _oracle_decode(inp, w.scale)
    for n_split in (0, 1, 3, 64):
        out = _decode(inp, w.scale, n_split=n_split)
        assert _err(out, ref) <= TOL, n_split
        assert torch.all(out[0] == 0)


def test_gqa_more_blocks_than_tiles():
    w = W.DecodeWorkload("tc_sparse", 0, 3, 32, 1, 128, 130, "bf16", lengths=(5, 130, 7), sub=12)
    inp = W.decode_inputs(w, DEV)
    ref = _oracle_decode(inp, w.scale)
    for n_split in (0, 64, 256):
        assert _err(_decode(inp, w.scale, n_split=n_split), ref) <= TOL, n_split


def test_gqa_one_block_per_segment():
    # 100 sequences of one KV head: between half and all of the SMs, so each segment gets a block
    w = W.DecodeWorkload("tc_aligned", 0, 100, 32, 1, 128, 700, "bf16", length_range=(1, 700), sub=13)
    inp = W.decode_inputs(w, DEV)
    assert _err(_decode(inp, w.scale), _oracle_decode(inp, w.scale)) <= TOL


def test_gqa_single_token_is_v0():
    w = W.DecodeWorkload("tc_one", 0, 3, 32, 1, 128, 64, "bf16", lengths=(1, 1, 1), sub=14)
    inp = W.decode_inputs(w, DEV)
    out = _decode(inp, w.scale)
    assert torch.equal(out, inp["v_cache"][:, 0].float().repeat_interleave(32, dim=1))


def test_gqa_all_empty():
    w = W.DecodeWorkload("tc_empty", 0, 4, 32, 1, 128, 64, "bf16", lengths=(0, 0, 0, 0), sub=15)
    inp = W.decode_inputs(w, DEV)
    out = torch.full((4, 32, 128), float("nan"), device=DEV)
    mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"], out=out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def _ramp_keys(inp, hkv, growth):
    """Keys along the cache that point ever more along the summed query rows of their group,
    so most heads' scores grow with the token index by many multiples of 2^8 (base 2)."""
    q = inp["q"].float()
    B, Hq, D = q.shape
    g = Hq // hkv
    S = inp["k_cache"].shape[1]
    u = q.view(B, hkv, g, D).sum(2) / g ** 0.5                      # [B, Hkv, D]
    t = torch.arange(S, device=q.device, dtype=torch.float32)[None, :, None, None]
    k = inp["k_cache"].float() * 0.25 + growth * t * u[:, None]
    inp["k_cache"] = k.to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("hq,hkv", [(32, 1), (32, 2)])
def test_gqa_growing_scores_rescale(hq, hkv):
    lens = (1000, 517, 129, 2000)
    w = W.DecodeWorkload("tc_ramp", 0, len(lens), hq, hkv, 128, 2000, "bf16", lengths=lens, sub=16)
    inp = W.decode_inputs(w, DEV)
    _ramp_keys(inp, hkv, 0.02)
    ref = _oracle_decode(inp, w.scale)
    for n_split in (0, 1, 5):
        assert _err(_decode(inp, w.scale, n_split=n_split), ref) <= TOL, n_split


def test_gqa_workspace_reuse_is_deterministic():
    w = W.DecodeWorkload("tc_reuse", 0, 16, 32, 1, 128, 3000, "bf16", length_range=(1, 3000), sub=17)
    inp = W.decode_inputs(w, DEV)
    inp2 = W.decode_inputs(w, DEV, seed=w.seed + 5)
    need = mk.decode_gqa_workspace_size(16, 32, 1, 128, 3000, mk.ATTN_BF16)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    a = _decode(inp, w.scale, workspace=ws)
    b = _decode(inp2, w.scale, workspace=ws)
    a2 = _decode(inp, w.scale, workspace=ws)
    assert torch.equal(a, a2)
    assert _err(b, _oracle_decode(inp2, w.scale)) <= TOL
    # every call leaves the arrival counters (the workspace's fixed 64 KiB head) at zero
    assert int(ws[:64 << 10].count_nonzero()) == 0


# --------------------------------------------------------------------------------- MLA

def absorb_on_device(q_nope, w_uk):
    return torch.einsum("hnr,bhn->bhr", w_uk.float(), q_nope.float()).to(torch.bfloat16).contiguous()


def _mla(inp, scale, **kw):
    q_lat = absorb_on_device(inp["q_nope"], inp["w_uk"])
    out = mk.decode_mla_absorbed(q_lat, inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["seq_lens"], scale, **kw)
    torch.cuda.synchronize()
    ref = oracle.mla_decode_absorbed(to_f64(q_lat), to_f64(inp["q_rope"]), to_f64(inp["c_cache"]),
                                     to_f64(inp["kr_cache"]), inp["seq_lens"].cpu().numpy(), scale)
    return out, ref


@pytest.mark.parametrize("hq", [64, 128, 48])
def test_mla_many_heads_ragged(hq):
    lens = (0, 1, 127, 128, 129, 1000, 2049)
    w = W.MlaWorkload("mla_tc", 3, len(lens), hq, 96, 128, 48, 96, 2049, lengths=lens, sub=5)
    inp = W.mla_inputs(w, DEV)
    for n_split in (0, 2):
        out, ref = _mla(inp, w.scale, n_split=n_split)
        assert _err(out, ref) <= TOL, n_split
        assert torch.all(out[0] == 0)


def test_mla_growing_scores_rescale():
    lens = (1500, 700, 2000)
    w = W.MlaWorkload("mla_ramp", 3, len(lens), 16, 96, 128, 48, 96, 2000, lengths=lens, sub=6)
    inp = W.mla_inputs(w, DEV)
    qr = inp["q_rope"].float()
    u = qr.sum(1) / qr.shape[1] ** 0.5                                 # [B, dr]
    t = torch.arange(2000, device=DEV, dtype=torch.float32)[None, :, None]
    inp["kr_cache"] = (inp["kr_cache"].float() * 0.25 + 0.03 * t * u[:, None]).to(torch.bfloat16).contiguous()
    for n_split in (0, 1):
        out, ref = _mla(inp, w.scale, n_split=n_split)
        assert _err(out, ref) <= TOL, n_split


def test_one_workspace_across_shapes_and_paths():
    # One zero-filled workspace reused by a sequence of calls whose shapes differ: tcgen05 MQA,
    # MLA, the register-MMA GQA decode with forced splits, then MQA again with another batch.
    # Each call's counters sit in the workspace's fixed counter region and no partial is ever
    # written there, so each call must give exactly what it gives on a fresh workspace.
    mqa = W.DecodeWorkload("ws_mqa", 0, 16, 32, 1, 128, 3000, "bf16", length_range=(1, 3000), sub=31)
    mqa2 = W.DecodeWorkload("ws_mqa2", 0, 3, 32, 1, 128, 3000, "bf16", lengths=(2999, 5, 1400), sub=32)
    gqa = W.DecodeWorkload("ws_gqa", 1, 5, 8, 4, 96, 2048, "bf16", length_range=(1, 2048), sub=33)
    mla = W.MlaWorkload("ws_mla", 3, 6, 16, 96, 128, 48, 96, 2049, lengths=(2049, 1, 128, 900, 0, 1500), sub=34)
    calls = []
    for w in (mqa, gqa, mqa2):
        inp = W.decode_inputs(w, DEV)
        calls.append(("gqa", w, inp, 3 if w is gqa else 0))
    mla_inp = W.mla_inputs(mla, DEV)
    calls.insert(1, ("mla", mla, mla_inp, 0))
    need = 0
    for kind, w, inp, n_split in calls:
        if kind == "gqa":
            need = max(need, mk.decode_gqa_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.s_max,
                                                          mk.ATTN_BF16, n_split))
        else:
            need = max(need, mk.decode_mla_workspace_size(w.batch, w.n_q_heads, 128, 48, w.s_max, n_split))
    shared = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for rnd in range(2):
        for kind, w, inp, n_split in calls:
            if kind == "gqa":
                fresh = _decode(inp, w.scale, n_split=n_split)
                got = _decode(inp, w.scale, n_split=n_split, workspace=shared)
                ref = _oracle_decode(inp, w.scale)
            else:
                fresh, ref = _mla(inp, w.scale, n_split=n_split)
                got, _ = _mla(inp, w.scale, n_split=n_split, workspace=shared)
            assert torch.equal(got, fresh), (kind, w.name, rnd)
            assert _err(got, ref) <= TOL, (kind, w.name, rnd)
    assert int(shared[:64 << 10].count_nonzero()) == 0

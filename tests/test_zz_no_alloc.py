"""attn_decode_gqa_noalloc, the decode entry point for callers that may not allocate.

Some callers cannot hand the library a workspace: a plugin inside a host program that owns
every device allocation, or a serving loop that must not call cudaMalloc because it can
synchronise the device and stall other streams. attn_decode_gqa_noalloc keeps the split
partials in a fixed array built into the library instead. These tests call it through the
C ABI (ctypes, raw device pointers) and check it against attn_decode_gqa, which takes a
caller workspace, on calls in a row that share the array — of one shape, and of a
sequence of different shapes and dtypes (a serving loop changes its batch every step), where
each call must still find its arrival counters at zero.

This file is named to be collected last, so a run that stops at the first failure has run
every other test before it. It needs nothing from the tests before it.
"""

import ctypes

import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

TOL_BF16 = 3e-3     # the decode parity tolerance for bf16 caches
TOL_F32 = 1e-5      # and for fp32 caches
DEV = "cuda"


def _noalloc(inp, out, scale, max_s, n_split):
    q, k, v, lens = inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"]
    B, Hq, D = q.shape
    S_max, Hkv = k.shape[1], k.shape[2]
    code = mk.ATTN_BF16 if q.dtype == torch.bfloat16 else mk.ATTN_F32
    return mk.lib().attn_decode_gqa_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(lens.data_ptr()), ctypes.c_void_p(out.data_ptr()), B, Hq, Hkv, D, scale, S_max, max_s,
        code, n_split, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _with_workspace(inp, scale, max_s, n_split):
    """attn_decode_gqa with a fresh zero-filled workspace of its own."""
    q = inp["q"]
    B, Hq, D = q.shape
    Hkv = inp["k_cache"].shape[2]
    code = mk.ATTN_BF16 if q.dtype == torch.bfloat16 else mk.ATTN_F32
    need = mk.decode_gqa_workspace_size(B, Hq, Hkv, D, max_s, code, n_split)
    ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=DEV)
    return mk.decode_gqa(q, inp["k_cache"], inp["v_cache"], inp["seq_lens"], scale=scale, max_s=max_s,
                         n_split=n_split, workspace=ws)


def _oracle_err(out, inp, scale):
    ref = oracle.decode_gqa(to_f64(inp["q"]), to_f64(inp["k_cache"]), to_f64(inp["v_cache"]),
                            inp["seq_lens"].cpu().numpy(), scale)
    return float(abs(out.double().cpu().numpy() - ref).max())


@pytest.mark.parametrize("shape,n_split", [
    # MiniMind-shaped GQA decode with 4 forced splits (partials in the built-in array)
    (dict(batch=32, n_q_heads=8, n_kv_heads=4, head_dim=96, s_max=2048, length_range=(512, 2048)), 4),
    # MQA over long caches; the library's own split choice
    (dict(batch=4, n_q_heads=32, n_kv_heads=1, head_dim=128, s_max=8192, lengths=(8192, 5000, 1, 8000)), 0),
])
def test_noalloc_matches_workspace_entry_point_twice(shape, n_split):
    w1 = W.DecodeWorkload("noalloc_a", 1, dtype="bf16", **shape)
    w2 = W.DecodeWorkload("noalloc_b", 1, dtype="bf16", sub=3, **shape)
    a, b = W.decode_inputs(w1, DEV), W.decode_inputs(w2, DEV)
    max_s = w1.s_max
    n_used = mk.decode_gqa_num_splits(w1.batch, w1.n_q_heads, w1.n_kv_heads, w1.head_dim, max_s, mk.ATTN_BF16,
                                      n_split)
    assert n_used > 1, "the case must exercise the split scratch"
    ref_a = _with_workspace(a, w1.scale, max_s, n_split)
    ref_b = _with_workspace(b, w2.scale, max_s, n_split)
    out_a = torch.full_like(ref_a, float("nan"))
    out_b = torch.full_like(ref_b, float("nan"))
    # two calls in a row: the second overwrites the shared array the first used
    assert _noalloc(a, out_a, w1.scale, max_s, n_split) == 0, mk.last_error()
    assert _noalloc(b, out_b, w2.scale, max_s, n_split) == 0, mk.last_error()
    torch.cuda.synchronize()
    assert (out_a - ref_a).abs().max().item() <= TOL_BF16
    assert (out_b - ref_b).abs().max().item() <= TOL_BF16
    # the same plan and kernels as the workspace entry point: the very same bits
    assert torch.equal(out_a, ref_a) and torch.equal(out_b, ref_b)


# A serving loop's sequence of calls on the one shared array: the batch, the head layout,
# the split count and the dtype change from call to call, so each call's counters and
# partials land at places that earlier calls used for other things.
_SEQUENCE = [
    ("minimind_b32", dict(batch=32, n_q_heads=8, n_kv_heads=4, head_dim=96, s_max=2048,
                          length_range=(512, 2048), dtype="bf16"), 4),
    ("b5_hq8_hkv4", dict(batch=5, n_q_heads=8, n_kv_heads=4, head_dim=96, s_max=2048,
                         length_range=(1, 2048), dtype="bf16"), 3),
    ("mqa_b4", dict(batch=4, n_q_heads=32, n_kv_heads=1, head_dim=128, s_max=8192,
                    lengths=(8192, 3000, 1, 6000), dtype="bf16"), 0),
    ("fp32_tiny", dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, s_max=128, lengths=(37, 128),
                       dtype="fp32"), 3),
    ("minimind_b32_again", dict(batch=32, n_q_heads=8, n_kv_heads=4, head_dim=96, s_max=2048,
                                length_range=(512, 2048), dtype="bf16"), 4),
]


def test_noalloc_sequence_of_shapes_shares_the_array():
    for i, (name, shape, n_split) in enumerate(_SEQUENCE):
        w = W.DecodeWorkload("noalloc_seq_" + name, 1, sub=20 + i, **shape)
        inp = W.decode_inputs(w, DEV)
        ref = _with_workspace(inp, w.scale, w.s_max, n_split)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(inp, out, w.scale, w.s_max, n_split) == 0, mk.last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), name
        tol = TOL_BF16 if shape["dtype"] == "bf16" else TOL_F32
        assert _oracle_err(out, inp, w.scale) <= tol, name


def test_noalloc_rejects_sizes_above_its_array():
    cap = mk.lib().attn_decode_gqa_noalloc_max_scratch()
    assert cap == 16 << 20
    # fp32 cache, 64 sequences x 32 heads x 64 splits x 128 floats = 64 MiB of partials:
    # refused before launch
    B, Hq, Hkv, D, S, n = 64, 32, 1, 128, 8192, 64
    assert mk.decode_gqa_workspace_size(B, Hq, Hkv, D, S, mk.ATTN_F32, n) > cap
    p = ctypes.c_void_p(1 << 20)
    rc = mk.lib().attn_decode_gqa_noalloc(p, p, p, p, p, B, Hq, Hkv, D, 0.088, S, S, mk.ATTN_F32, n,
                                          ctypes.c_void_p(0))
    assert rc == -4
    assert "above the built-in" in mk.last_error()

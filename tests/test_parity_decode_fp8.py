"""GQA decode over an E4M3 cache with per-row K and V scales (attn_decode_gqa_fp8) against
the fp64 CPU oracle.

The codes widen exactly (to fp32, or to fp16 for the tensor-core kernel), the bf16 query is
exact in fp32 (in fp16 too for |q| in [2^-14, 65504], within 2^-25 below), so the scores are
products summed in fp32; the tensor-core kernel multiplies V by each weight times its row's V
scale (and 2^10) split into an fp16 head and residual, which leaves about 2^-22 of the weight.
The bound is the fp32 cache path's, max |Δ| ≤ 1e-5.
"""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

TOL = 1e-5
DEV = "cuda"


def _run(inp, scale, **kw):
    out = mk.decode_gqa_fp8(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_scale"], inp["v_scale"],
                            inp["seq_lens"], scale=scale, **kw)
    torch.cuda.synchronize()
    return out


def _ref(inp, scale):
    return oracle.decode_gqa_fp8(to_f64(inp["q"]), inp["k_cache"].cpu().numpy(), inp["v_cache"].cpu().numpy(),
                                 to_f64(inp["k_scale"]), to_f64(inp["v_scale"]), inp["seq_lens"].cpu().numpy(),
                                 scale)


# up to 16 query heads per KV head: the tensor-core kernel (one 8-column block of heads up
# to 8, two up to 16); (32, 1, 128), (24, 1, 64), (64, 1, 64): the CUDA-core kernel
@pytest.mark.parametrize("hq,hkv,d", [(8, 4, 96), (8, 8, 64), (8, 1, 128), (32, 8, 128), (6, 3, 96), (16, 1, 128),
                                      (12, 1, 96), (32, 1, 128), (24, 1, 64), (64, 1, 64)])
def test_fp8_ragged(hq, hkv, d):
    lens = (0, 1, 127, 128, 129, 300, 1000)
    w = W.DecodeWorkload("fp8_ragged", 5, len(lens), hq, hkv, d, 1000, "bf16", lengths=lens, sub=hq + d)
    inp = W.fp8_decode_inputs(w, DEV)
    ref = _ref(inp, w.scale)
    for n_split in (0, 1, 3):
        out = _run(inp, w.scale, n_split=n_split)
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL, n_split
        assert torch.all(out[0] == 0)


@pytest.mark.parametrize("hq,hkv", [(8, 4), (64, 1)])
def test_fp8_single_token_is_the_scaled_value_row(hq, hkv):
    # One token: weight 1, so out = e4m3(v) · v_scale. The CUDA-core kernel (64 heads per KV
    # head) forms that product once in fp32: exact equality. The tensor-core kernel multiplies
    # the code by the scale (times 2^10) split into an fp16 head and an fp16 residual, which
    # sum to it within 2^-22 of it, and adds the two exact products in the MMA's fp32
    # accumulator (one more rounding, up to 2^-23), then divides by 2^10 exactly: within
    # 2^-21 of |v|, checked against 2^-20 of |v| per element.
    w = W.DecodeWorkload("fp8_one", 5, 3, hq, hkv, 96 if hkv == 4 else 64, 8, "bf16", lengths=(1, 1, 1), sub=1)
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale)
    v = inp["v_cache"][:, 0].view(torch.float8_e4m3fn).float() * inp["v_scale"][:, 0, :, None]
    v = v.repeat_interleave(hq // hkv, dim=1)
    if hq // hkv > 16:
        assert torch.equal(out, v)
    else:
        assert bool(((out - v).abs() <= 2.0 ** -20 * v.abs()).all())


def test_fp8_minimind_full_size():
    """The MiniMind decode batch (B=32, lengths U[512, 2048]) with an fp8 cache, every output."""
    w = W.MINIMIND_GQA
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale, max_s=int(inp["seq_lens"].max()))
    assert float(np.abs(to_f64(out) - _ref(inp, w.scale)).max()) <= TOL


def test_fp8_one_workspace_across_calls():
    """Calls of different shapes on one zero-filled workspace: each finds its arrival counters
    at zero (the counter region is left zero by every call) and gives the same bits as a call
    on a fresh workspace."""
    shapes = [W.MINIMIND_GQA,
              W.DecodeWorkload("fp8_ws_b", 5, 7, 16, 1, 128, 1000, "bf16", lengths=(0, 1, 127, 300, 1000, 64, 65),
                               sub=7),
              W.MINIMIND_GQA]
    sizes = [mk.decode_gqa_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.s_max, mk.ATTN_FP8_E4M3, 0)
             for w in shapes]
    ws = torch.zeros(max(sizes), dtype=torch.uint8, device=DEV)
    for w in shapes:
        inp = W.fp8_decode_inputs(w, DEV)
        fresh = torch.zeros(max(sizes), dtype=torch.uint8, device=DEV)
        ref = _run(inp, w.scale, workspace=fresh)
        out = _run(inp, w.scale, workspace=ws)
        assert torch.equal(out, ref)
        assert int(ws[:64 << 10].count_nonzero()) == 0
        assert float(np.abs(to_f64(out) - _ref(inp, w.scale)).max()) <= TOL


@pytest.mark.parametrize("hq,hkv,s_max", [(8, 2, 1001), (4, 1, 999), (16, 4, 1000)])
def test_fp8_more_than_32_sequences(hq, hkv, s_max):
    """40 sequences (the block start is found over two groups of 32), an odd cache capacity
    (S_max·Hkv not a multiple of 4: the row scales arrive by 4-byte copies, not one bulk copy
    per tile) and every split count: the balanced split, a cap of one block per segment, three."""
    w = W.DecodeWorkload("fp8_b40", 5, 40, hq, hkv, 64, s_max, "bf16", length_range=(0, s_max), sub=hq + s_max)
    inp = W.fp8_decode_inputs(w, DEV)
    ref = _ref(inp, w.scale)
    for n_split in (0, 1, 3):
        out = _run(inp, w.scale, n_split=n_split)
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL, n_split


@pytest.mark.parametrize("hq,hkv,d,B", [(8, 4, 96, 3000), (16, 2, 128, 2500)])
def test_fp8_large_batches(hq, hkv, d, B):
    """Thousands of short ragged sequences: past what the tensor-core kernel's per-sequence
    tables leave room for, the call runs on the CUDA-core E4M3 kernel (and its merge); every
    output at the fp8 bound."""
    w = W.DecodeWorkload("fp8_large_b", 5, B, hq, hkv, d, 48, "bf16", length_range=(0, 48), sub=B)
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale)
    mk.check_status()
    assert float(np.abs(to_f64(out) - _ref(inp, w.scale)).max()) <= TOL


def test_fp8_long_context():
    """131072 and 70001 cached tokens over the E4M3 cache (tensor-core form), every output."""
    w = W.DecodeWorkload("fp8_128k", 5, 2, 8, 4, 96, 131072, "bf16", lengths=(131072, 70001), sub=99)
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale)
    mk.check_status()
    assert float(np.abs(to_f64(out) - _ref(inp, w.scale)).max()) <= TOL

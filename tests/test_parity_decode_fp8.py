"""GQA decode over an E4M3 cache with per-row K and V scales (attn_decode_gqa_fp8) against
the fp64 CPU oracle.

The codes widen to fp32 exactly and the bf16 query is exact in fp32, so the kernel does the
fp32 cache path's arithmetic on exact inputs; the bound is that path's, max |Δ| ≤ 1e-5.
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


@pytest.mark.parametrize("hq,hkv,d", [(8, 4, 96), (8, 8, 64), (8, 1, 128), (32, 8, 128), (6, 3, 96)])
def test_fp8_ragged(hq, hkv, d):
    lens = (0, 1, 127, 128, 129, 300, 1000)
    w = W.DecodeWorkload("fp8_ragged", 5, len(lens), hq, hkv, d, 1000, "bf16", lengths=lens, sub=hq + d)
    inp = W.fp8_decode_inputs(w, DEV)
    ref = _ref(inp, w.scale)
    for n_split in (0, 1, 3):
        out = _run(inp, w.scale, n_split=n_split)
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL, n_split
        assert torch.all(out[0] == 0)


def test_fp8_single_token_is_the_scaled_value_row():
    # one token: weight 1, so out = fp32(e4m3(v) · v_scale) exactly
    w = W.DecodeWorkload("fp8_one", 5, 3, 8, 4, 96, 8, "bf16", lengths=(1, 1, 1), sub=1)
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale)
    v = inp["v_cache"][:, 0].view(torch.float8_e4m3fn).float() * inp["v_scale"][:, 0, :, None]
    assert torch.equal(out, v.repeat_interleave(2, dim=1))


def test_fp8_minimind_full_size():
    """The MiniMind decode batch (B=32, lengths U[512, 2048]) with an fp8 cache, every output."""
    w = W.MINIMIND_GQA
    inp = W.fp8_decode_inputs(w, DEV)
    out = _run(inp, w.scale, max_s=int(inp["seq_lens"].max()))
    assert float(np.abs(to_f64(out) - _ref(inp, w.scale)).max()) <= TOL

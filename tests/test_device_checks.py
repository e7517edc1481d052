"""Device-side checks of the length arrays (attn_set_device_checks): with the checks on, a
length, offset or start position outside its stated bounds makes the call return
ATTN_ERR_INPUT before anything else is launched; valid inputs give the same outputs as with
the checks off.

Every call below that passes an out-of-bounds length first asserts that the checks are on:
with them off those lengths would send the kernels past the end of the cache.
"""

import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture
def checks_on():
    prev = mk.set_device_checks(True)
    assert mk.device_checks()
    yield
    mk.set_device_checks(prev)


def _expect_input_error(fn, rule):
    assert mk.device_checks(), "the device checks must be on before passing bad lengths"
    with pytest.raises(mk.MlakvError) as e:
        fn()
    assert e.value.code == mk.ATTN_ERR_INPUT
    assert rule in str(e.value), str(e.value)
    mk.check_status()                          # nothing was launched that could have failed


def _gqa(dtype="bf16", B=3, S_max=256, hq=8, hkv=2, d=128):
    w = W.DecodeWorkload("checks", 6, B, hq, hkv, d, S_max, dtype, lengths=(5,) * B, sub=90)
    return W.decode_inputs(w, DEV), w


def test_decode_length_above_max_s(checks_on):
    for dtype, hq, hkv in (("bf16", 8, 2), ("fp32", 8, 2), ("bf16", 32, 1)):
        inp, w = _gqa(dtype, hq=hq, hkv=hkv)
        lens = torch.tensor([5, 300, 7], dtype=torch.int32, device=DEV)      # 300 > max_s = 100
        _expect_input_error(lambda: mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], lens, scale=w.scale,
                                                  max_s=100), "a length above its bound (first at index 1)")


def test_decode_negative_length(checks_on):
    inp, w = _gqa()
    lens = torch.tensor([5, 9, -1], dtype=torch.int32, device=DEV)
    _expect_input_error(lambda: mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], lens, scale=w.scale),
                        "a negative length or start position (first at index 2)")


def test_decode_valid_lengths_unchanged(checks_on):
    inp, w = _gqa()
    lens = torch.tensor([5, 256, 0], dtype=torch.int32, device=DEV)
    a = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], lens, scale=w.scale)
    mk.set_device_checks(False)
    b = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], lens, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_fp8_and_mla_decode_lengths(checks_on):
    w = W.DecodeWorkload("checks_fp8", 6, 2, 8, 4, 96, 128, "bf16", lengths=(5, 5), sub=91)
    fi = W.fp8_decode_inputs(w, DEV)
    lens = torch.tensor([129, 3], dtype=torch.int32, device=DEV)             # 129 > max_s = 128
    _expect_input_error(lambda: mk.decode_gqa_fp8(fi["q"], fi["k_cache"], fi["v_cache"], fi["k_scale"],
                                                  fi["v_scale"], lens, scale=w.scale, max_s=128),
                        "a length above its bound (first at index 0)")
    wm = W.MlaWorkload("checks_mla", 6, 2, 16, 96, 128, 48, 96, 128, lengths=(5, 5), sub=92)
    mi = W.mla_inputs(wm, DEV)
    q_lat = mk.mla_absorb_query(mi["q_nope"], mi["w_uk"])
    lens = torch.tensor([3, 200], dtype=torch.int32, device=DEV)
    _expect_input_error(lambda: mk.decode_mla_absorbed(q_lat, mi["q_rope"], mi["c_cache"], mi["kr_cache"], lens,
                                                       wm.scale, max_s=128),
                        "a length above its bound (first at index 1)")


def test_prefill_offsets(checks_on):
    w = W.PrefillWorkload("checks_prefill", 6, 2, 8, 2, 128, lengths=(100, 60), sub=93)
    inp = W.prefill_inputs(w, DEV)
    q, k, v = inp["q"], inp["k"], inp["v"]
    bad = {
        "decreasing offsets (first at index 1)": [0, 100, 60],
        "offsets not starting at 0 (first at index 0)": [4, 100, 160],
        "the last offset above T (first at index 2)": [0, 100, 170],
        "a length above its bound (first at index 0)": [0, 120, 160],      # 120 > max_seqlen = 100
    }
    for rule, cu in bad.items():
        cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
        _expect_input_error(lambda: mk.prefill_gqa_causal(q, k, v, cu_t, 100, scale=w.scale), rule)
    ok = mk.prefill_gqa_causal(q, k, v, inp["cu_seqlens"], 100, scale=w.scale)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(ok).all())


def test_chunked_start_positions(checks_on):
    inp, w = _gqa(B=2, S_max=512)
    q = torch.randn((300, 8, 128), device=DEV).to(torch.bfloat16)
    cu = torch.tensor([0, 200, 300], dtype=torch.int32, device=DEV)
    for start, rule in (([100, 450], "start_pos + chunk length above max_kv (first at index 1)"),
                        ([-3, 10], "a negative length or start position (first at index 0)")):
        st = torch.tensor(start, dtype=torch.int32, device=DEV)
        _expect_input_error(lambda: mk.prefill_gqa_chunked(q, inp["k_cache"], inp["v_cache"], cu, st, 512,
                                                           scale=w.scale), rule)
    wm = W.MlaWorkload("checks_mla_chunk", 6, 2, 16, 96, 128, 48, 96, 512, lengths=(5, 5), sub=94)
    mi = W.mla_inputs(wm, DEV)
    ql = torch.randn((300, 16, 128), device=DEV).to(torch.bfloat16)
    qr = torch.randn((300, 16, 48), device=DEV).to(torch.bfloat16)
    st = torch.tensor([400, 0], dtype=torch.int32, device=DEV)               # 400 + 200 > max_kv = 512
    _expect_input_error(lambda: mk.prefill_mla_chunked(ql, qr, mi["c_cache"], mi["kr_cache"], cu, st, 512,
                                                       wm.scale), "start_pos + chunk length above max_kv")

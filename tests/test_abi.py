"""The C-ABI library loads, exports every entry point the header declares, and rejects bad
host-side arguments with the documented status before launching anything.

Runs without a GPU: every call here fails validation first, so no kernel is launched and
no device memory is touched (the pointers below are never dereferenced).
"""

import ctypes
import os
import re

import pytest

import mla_kv_cache_flash_b300 as mk

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mlakv.h")

OK, NULL, SHAPE, UNSUP, WS = 0, -1, -2, -3, -4
P = ctypes.c_void_p(1 << 20)   # aligned, non-NULL, never dereferenced
PU = ctypes.c_void_p((1 << 20) + 2)   # misaligned
N0 = ctypes.c_void_p(0)
S0 = ctypes.c_void_p(0)


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mk.lib_path):
        from mla_kv_cache_flash_b300 import build
        build.build()
    return mk.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("attn_decode_gqa", "attn_decode_mla_absorbed", "attn_prefill_gqa_causal",
                 "attn_merge_partials", "attn_last_error", "attn_check_status"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_only_the_abi_is_exported():
    out = os.popen(f"nm -D --defined-only {mk.lib_path}").read()
    ours = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    assert set(declared_functions()) <= set(ours)
    assert not [n for n in ours if "mlakv" in n], "internal symbols leaked into the dynamic table"


def test_version(L):
    assert "sm_103a" in mk.version()


def gqa(L, q=P, k=P, v=P, lens=P, out=P, B=2, Hq=8, Hkv=2, D=64, scale=0.125, S_max=128, max_S=128,
        dtype=0, n_split=0, ws=N0, ws_bytes=0):
    return L.attn_decode_gqa(q, k, v, lens, out, B, Hq, Hkv, D, scale, S_max, max_S, dtype, n_split,
                             ws, ws_bytes, S0)


@pytest.mark.parametrize("which", ["q", "k", "v", "lens", "out"])
def test_gqa_null_pointers(L, which):
    assert gqa(L, **{which: N0}) == NULL
    assert "non-NULL" in mk.last_error()


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(Hkv=0), dict(S_max=0), dict(max_S=-1),
                                dict(max_S=129), dict(Hq=32, Hkv=3), dict(Hq=32, Hkv=6), dict(n_split=-1),
                                dict(n_split=257), dict(scale=float("nan")), dict(scale=float("inf"))])
def test_gqa_bad_shapes(L, kw):
    assert gqa(L, **kw) == SHAPE


def test_gqa_divisibility_message(L):
    assert gqa(L, Hq=32, Hkv=3) == SHAPE
    assert "does not divide" in mk.last_error()


@pytest.mark.parametrize("kw", [dict(D=80), dict(D=256), dict(dtype=2), dict(dtype=3), dict(Hq=256, Hkv=1), dict(q=PU),
                                dict(k=PU), dict(out=PU)])
def test_gqa_unsupported(L, kw):
    assert gqa(L, **kw) == UNSUP


def test_gqa_workspace_checks(L):
    need = L.attn_decode_gqa_workspace_size(2, 8, 2, 64, 128, 0, 2)
    assert need > 0
    assert L.attn_decode_gqa_num_splits(2, 8, 2, 64, 128, 0, 2) == 2
    assert gqa(L, n_split=2) == WS
    assert gqa(L, n_split=2, ws=P, ws_bytes=need - 1) == WS
    assert gqa(L, n_split=2, ws=PU, ws_bytes=need) == WS
    # one split needs no workspace
    assert L.attn_decode_gqa_workspace_size(2, 8, 2, 64, 128, 0, 1) == 0


def test_gqa_split_plan_bounds(L):
    # never more splits than tiles of the longest sequence; an explicit count is honoured
    assert L.attn_decode_gqa_num_splits(1, 1, 1, 64, 1, 0, 0) == 1
    assert L.attn_decode_gqa_num_splits(1, 1, 1, 64, 0, 0, 0) == 1
    assert L.attn_decode_gqa_num_splits(2, 8, 2, 64, 128, 0, 7) == 7
    # bf16 caches: the persistent grid (one block per SM), capped at n_split x segments
    # (a segment: one sequence's tokens for a group of up to 4 KV heads)
    n = L.attn_decode_gqa_num_splits(1, 32, 1, 128, 8192, 1, 0)
    assert n >= 1
    assert L.attn_decode_gqa_num_splits(1, 32, 1, 128, 8192, 1, 3) == min(3, n)
    assert L.attn_decode_gqa_num_splits(2, 32, 32, 128, 8192, 1, 1) == min(2 * 8, n)
    assert L.attn_decode_gqa_num_splits(64, 32, 32, 128, 8192, 1, 0) >= 1
    assert L.attn_decode_gqa_num_splits(2, 8, 3, 64, 128, 0, 0) == SHAPE


def mla(L, ql=P, qr=P, c=P, kr=P, lens=P, out=P, B=2, Hq=16, r=128, dr=48, scale=1 / 12, S_max=64, max_S=64,
        n_split=0, ws=N0, ws_bytes=0):
    return L.attn_decode_mla_absorbed(ql, qr, c, kr, lens, out, B, Hq, r, dr, scale, S_max, max_S, n_split,
                                      ws, ws_bytes, S0)


@pytest.mark.parametrize("which", ["ql", "qr", "c", "kr", "lens", "out"])
def test_mla_null_pointers(L, which):
    assert mla(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(S_max=0), dict(max_S=65), dict(n_split=-2)])
def test_mla_bad_shapes(L, kw):
    assert mla(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(r=64), dict(dr=64), dict(Hq=8), dict(Hq=144), dict(c=PU)])
def test_mla_unsupported(L, kw):
    assert mla(L, **kw) == UNSUP


def test_mla_workspace(L):
    need = L.attn_decode_mla_workspace_size(2, 16, 128, 48, 4096, 4)
    assert need >= 2 * 16 * 4 * 128 * 4
    assert mla(L, S_max=4096, max_S=4096, n_split=4) == WS


def fp8(L, q=P, k=P, v=P, ks=P, vs=P, lens=P, out=P, B=2, Hq=8, Hkv=4, D=96, scale=0.1, S_max=128, max_S=128,
        n_split=1, ws=N0, ws_bytes=0):
    return L.attn_decode_gqa_fp8(q, k, v, ks, vs, lens, out, B, Hq, Hkv, D, scale, S_max, max_S, n_split, ws,
                                 ws_bytes, S0)


@pytest.mark.parametrize("which", ["q", "k", "v", "ks", "vs", "lens", "out"])
def test_fp8_null_pointers(L, which):
    assert fp8(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=8, Hkv=3), dict(max_S=129), dict(scale=float("inf"))])
def test_fp8_bad_shapes(L, kw):
    assert fp8(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(D=80), dict(ks=PU), dict(k=PU)])
def test_fp8_unsupported(L, kw):
    assert fp8(L, **kw) == UNSUP


def test_fp8_workspace(L):
    # the tensor-core fp8 plan: persistent blocks, three resident per SM (148 SMs without a
    # GPU), at most 32 per (sequence, KV head), each with two partial slots of G rows after
    # the counter region; n_split > 0 caps the blocks at n_split per (sequence, KV head)
    n = L.attn_decode_gqa_num_splits(2, 8, 4, 96, 4096, 2, 0)
    assert n == 32 * 2 * 4
    assert L.attn_decode_gqa_num_splits(32, 8, 4, 96, 4096, 2, 0) == 3 * 148
    assert L.attn_decode_gqa_num_splits(2, 8, 4, 96, 4096, 2, 5) == 5 * 2 * 4
    up = lambda x: (x + 255) // 256 * 256
    assert L.attn_decode_gqa_workspace_size(2, 8, 4, 96, 4096, 2, 0) == \
        (64 << 10) + up(2 * n * 2 * 96 * 4) + up(2 * n * 2 * 4)
    assert fp8(L, S_max=4096, max_S=4096, n_split=0) == WS


def chunked(L, q=P, k=P, v=P, cu=P, st=P, out=P, B=2, T=10, Hq=8, Hkv=4, D=96, scale=0.1, S_max=64, max_kv=64,
            dt=1, n_split=1, ws=N0, ws_bytes=0):
    return L.attn_prefill_gqa_chunked(q, k, v, cu, st, out, B, T, Hq, Hkv, D, scale, S_max, max_kv, dt, n_split, ws,
                                      ws_bytes, S0)


@pytest.mark.parametrize("which", ["q", "k", "v", "cu", "st", "out"])
def test_chunked_null_pointers(L, which):
    assert chunked(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(T=-1), dict(T=65536), dict(Hq=8, Hkv=3), dict(max_kv=65),
                                dict(scale=float("nan"))])
def test_chunked_bad_shapes(L, kw):
    assert chunked(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(D=80), dict(dt=2), dict(cu=PU), dict(out=PU)])
def test_chunked_unsupported(L, kw):
    assert chunked(L, **kw) == UNSUP


def test_chunked_empty_and_workspace(L):
    assert chunked(L, T=0) == OK
    assert chunked(L, max_kv=0) == OK
    assert L.attn_prefill_gqa_chunked_workspace_size(2, 10, 8, 4, 96, 64, 0, 1) == 0
    need = L.attn_prefill_gqa_chunked_workspace_size(2, 10, 8, 4, 96, 4096, 0, 4)
    assert need >= 10 * 8 * 4 * 96 * 4
    assert chunked(L, S_max=4096, max_kv=4096, n_split=4) == WS


def test_chunked_tensor_core_workspace(L):
    # bf16, D = 128 and 16 query heads per KV head: the tcgen05 form, whose workspace always
    # holds the arrival counters' region and the partial slots of one block per SM
    need = L.attn_prefill_gqa_chunked_workspace_size(2, 10, 32, 2, 128, 4096, 1, 0)
    assert need >= (64 << 10) + 2 * 148 * 64 * 128 * 4
    assert chunked(L, Hq=32, Hkv=2, D=128, dt=1, S_max=4096, max_kv=4096, n_split=0) == WS
    # the same shape over an fp32 cache stays on the CUDA-core form
    assert L.attn_prefill_gqa_chunked_workspace_size(2, 10, 32, 2, 128, 4096, 0, 1) == 0


def test_chunked_long_chunks_need_no_workspace(L):
    # bf16 at D = 128 with chunks of 128 new tokens or more on average: the tcgen05 prefill
    # kernel over the caches, no split and no workspace, for any n_split
    for hq, hkv in ((32, 2), (32, 8), (12, 4)):
        for n_split in (0, 1, 5):
            assert L.attn_prefill_gqa_chunked_workspace_size(2, 256, hq, hkv, 128, 4096, 1, n_split) == 0
    # one token short of 128 per sequence: the decode kernels again
    assert L.attn_prefill_gqa_chunked_workspace_size(2, 255, 32, 2, 128, 4096, 1, 0) > 0
    # fp32, or D below 128: never the prefill kernel
    assert L.attn_prefill_gqa_chunked_workspace_size(2, 256, 32, 8, 128, 4096, 0, 4) > 0
    assert L.attn_prefill_gqa_chunked_workspace_size(2, 256, 32, 8, 96, 4096, 1, 0) > 0


def test_mla_chunked_long_chunks_need_no_workspace(L):
    # chunks of 128 new tokens or more on average: the prefill kernel's MLA form, no workspace
    for hq in (16, 8, 3):
        for n_split in (0, 2):
            assert L.attn_prefill_mla_chunked_workspace_size(4, 512, hq, 4096, n_split) == 0
    assert L.attn_prefill_mla_chunked_workspace_size(4, 511, 16, 4096, 0) > 0


def mla_chunked(L, ql=P, qr=P, c=P, kr=P, cu=P, st=P, out=P, B=2, T=10, Hq=16, r=128, dr=48, scale=1 / 12,
                S_max=64, max_kv=64, n_split=1, ws=N0, ws_bytes=0):
    return L.attn_prefill_mla_chunked(ql, qr, c, kr, cu, st, out, B, T, Hq, r, dr, scale, S_max, max_kv, n_split,
                                      ws, ws_bytes, S0)


@pytest.mark.parametrize("which", ["ql", "qr", "c", "kr", "cu", "st", "out"])
def test_mla_chunked_null_pointers(L, which):
    assert mla_chunked(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(T=70000), dict(Hq=0), dict(max_kv=65), dict(scale=float("inf"))])
def test_mla_chunked_bad_shapes(L, kw):
    assert mla_chunked(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(r=64), dict(dr=64), dict(Hq=129), dict(kr=PU)])
def test_mla_chunked_unsupported(L, kw):
    assert mla_chunked(L, **kw) == UNSUP


def test_mla_chunked_empty_and_workspace(L):
    assert mla_chunked(L, T=0) == OK
    # 16 heads: the tcgen05 form, with its counter region and one block per SM
    assert L.attn_prefill_mla_chunked_workspace_size(2, 10, 16, 64, 1) >= (64 << 10) + 2 * 64 * 128 * 4
    assert L.attn_prefill_mla_chunked_workspace_size(2, 10, 16, 4096, 0) >= (64 << 10) + 2 * 148 * 64 * 128 * 4
    assert mla_chunked(L, S_max=4096, max_kv=4096, n_split=4) == WS
    assert mla_chunked(L) == WS


def absorb(L, qn=P, wuk=P, ql=P, B=2, Hq=16, dn=96, r=128):
    return L.attn_mla_absorb_query(qn, wuk, ql, B, Hq, dn, r, S0)


def apply_uv(L, ol=P, wuv=P, out=P, B=2, Hq=16, r=128, dv=96):
    return L.attn_mla_apply_uv(ol, wuv, out, B, Hq, r, dv, S0)


@pytest.mark.parametrize("which", ["qn", "wuk", "ql"])
def test_absorb_null_pointers(L, which):
    assert absorb(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(dn=0), dict(r=0)])
def test_absorb_bad_shapes(L, kw):
    assert absorb(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(r=48), dict(r=288), dict(dn=513), dict(wuk=PU)])
def test_absorb_unsupported(L, kw):
    assert absorb(L, **kw) == UNSUP


@pytest.mark.parametrize("which", ["ol", "wuv", "out"])
def test_apply_uv_null_pointers(L, which):
    assert apply_uv(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=-1), dict(r=0), dict(dv=0)])
def test_apply_uv_bad_shapes(L, kw):
    assert apply_uv(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(r=48), dict(r=288), dict(dv=257), dict(out=PU)])
def test_apply_uv_unsupported(L, kw):
    assert apply_uv(L, **kw) == UNSUP


def append(L, q=P, kn=P, vn=P, pos=P, cis=P, qo=P, kc=P, vc=P, lens=N0, B=2, Hq=8, Hkv=4, D=96, S_max=64, dt=1):
    return L.attn_kv_append_rope(q, kn, vn, pos, cis, qo, kc, vc, lens, B, Hq, Hkv, D, S_max, dt, S0)


def mla_append(L, qr=P, cn=P, krn=P, pos=P, cis=P, qo=P, cc=P, krc=P, lens=N0, B=2, Hq=16, r=128, dr=48, S_max=64):
    return L.attn_mla_append_rope(qr, cn, krn, pos, cis, qo, cc, krc, lens, B, Hq, r, dr, S_max, S0)


@pytest.mark.parametrize("which", ["q", "kn", "vn", "pos", "cis", "qo", "kc", "vc"])
def test_append_null_pointers(L, which):
    assert append(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(Hkv=0), dict(D=0), dict(S_max=0), dict(Hq=8, Hkv=3)])
def test_append_bad_shapes(L, kw):
    assert append(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(D=100), dict(D=6, dt=0), dict(dt=2), dict(kc=PU), dict(lens=PU)])
def test_append_unsupported(L, kw):
    assert append(L, **kw) == UNSUP


@pytest.mark.parametrize("which", ["qr", "cn", "krn", "pos", "cis", "qo", "cc", "krc"])
def test_mla_append_null_pointers(L, which):
    assert mla_append(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(r=0), dict(dr=0), dict(S_max=0)])
def test_mla_append_bad_shapes(L, kw):
    assert mla_append(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(r=100), dict(dr=50), dict(cc=PU)])
def test_mla_append_unsupported(L, kw):
    assert mla_append(L, **kw) == UNSUP


def prefill(L, q=P, k=P, v=P, cu=P, out=P, B=2, Hq=8, Hkv=2, D=128, scale=0.088, max_seqlen=64, T=100):
    return L.attn_prefill_gqa_causal(q, k, v, cu, out, B, Hq, Hkv, D, scale, max_seqlen, T, S0)


@pytest.mark.parametrize("which", ["q", "k", "v", "cu", "out"])
def test_prefill_null_pointers(L, which):
    assert prefill(L, **{which: N0}) == NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(Hkv=0), dict(Hq=8, Hkv=3), dict(max_seqlen=-1),
                                dict(T=-1), dict(scale=float("nan"))])
def test_prefill_bad_shapes(L, kw):
    assert prefill(L, **kw) == SHAPE


@pytest.mark.parametrize("kw", [dict(D=64), dict(D=96), dict(q=PU)])
def test_prefill_unsupported(L, kw):
    assert prefill(L, **kw) == UNSUP


def test_prefill_empty_is_a_no_op(L):
    assert prefill(L, T=0) == OK
    assert prefill(L, max_seqlen=0) == OK


def test_merge_checks(L):
    assert L.attn_merge_partials(N0, P, P, 4, 2, 64, S0) == NULL
    assert L.attn_merge_partials(P, P, P, 4, 0, 64, S0) == SHAPE
    assert L.attn_merge_partials(P, P, P, 4, 2, 66, S0) == UNSUP
    assert L.attn_merge_partials(P, P, P, -1, 2, 64, S0) == SHAPE


def test_tensor_core_plan(L):
    # MQA / wide groups at D=128 and MLA go to the tensor-core decode: 148 SMs (the plan
    # without a GPU assumes a 148-SM part); MQA keeps every SM streaming, MLA takes a whole
    # number of blocks per segment when that fills at least 85% of the resident blocks
    assert L.attn_decode_gqa_num_splits(64, 32, 1, 128, 8192, 1, 0) == 148       # every SM
    assert L.attn_decode_mla_num_splits(64, 16, 128, 48, 4096, 0) == 256          # 2 per SM, 4 per seq
    assert L.attn_decode_mla_num_splits(1, 16, 128, 48, 4096, 0) == 32            # one segment: 32 pieces
    assert L.attn_decode_mla_num_splits(8, 16, 128, 48, 4096, 0) == 256           # 32 per segment
    assert L.attn_decode_gqa_num_splits(64, 32, 8, 128, 8192, 1, 0) == 148        # register-MMA path
    # workspace: the fixed 64 KiB counter region (one counter per segment), then two partial
    # slots of N heads x 128 fp32 per block and their lse, each part 256-byte aligned
    up = lambda x: (x + 255) // 256 * 256
    region = 64 << 10
    n = 148
    assert L.attn_decode_gqa_workspace_size(64, 32, 1, 128, 8192, 1, 0) == \
        region + up(2 * n * 32 * 128 * 4) + up(2 * n * 32 * 4)
    n = 256
    assert L.attn_decode_mla_workspace_size(64, 16, 128, 48, 4096, 0) == \
        region + up(2 * n * 16 * 128 * 4) + up(2 * n * 16 * 4)


def test_workspace_counter_region(L):
    # every workspace that holds partials starts with the same 64 KiB counter region, so one
    # buffer serves calls of any shape: the fp32 path's partials lie after it too
    region = 64 << 10
    up = lambda x: (x + 255) // 256 * 256
    B, Hq, D, n = 2, 8, 64, 2
    assert L.attn_decode_gqa_workspace_size(B, Hq, 2, D, 128, 0, n) == \
        region + up(B * Hq * n * D * 4) + up(B * Hq * n * 4)
    # more segments than the region's 16384 counters: the region grows to hold them
    B, Hq, Hkv = 1024, 32, 32
    segs = B * Hkv
    need = L.attn_decode_gqa_workspace_size(B, Hq, Hkv, 128, 64, 1, 0)
    assert need >= up(segs * 4) > region


@pytest.mark.parametrize("cycles", [0, 999, 10**9 + 1])
def test_selftest_bounds(L, cycles):
    # validated before any launch
    assert L.attn_selftest_bounded_wait(cycles, S0) == SHAPE


def test_binding_signatures_cover_the_header():
    # the ctypes binding declares argument types for every entry point of the header
    assert set(declared_functions()) == set(mk._SIGNATURES)


def test_missing_library_fails_loudly(monkeypatch):
    # no library, no result: the binding raises instead of computing anything itself
    monkeypatch.setattr(mk, "_lib", None)
    monkeypatch.setattr(mk, "lib_path", os.path.join(os.path.dirname(mk.lib_path), "absent", "libmlakv.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        mk.lib()
    with pytest.raises(RuntimeError, match="no fallback"):
        mk.version()


def _kind(param):
    param = param.strip()
    if "*" in param or param.startswith("mlakv_stream_t"):
        return "ptr"
    if param.startswith("float"):
        return "float"
    if param.startswith("size_t"):
        return "size"
    if param.startswith("long long"):
        return "longlong"
    return "int"          # int, attn_dtype


_CTYPE_KIND = {ctypes.c_void_p: "ptr", ctypes.c_float: "float", ctypes.c_size_t: "size",
               ctypes.c_longlong: "longlong", ctypes.c_int: "int"}


def test_binding_argument_kinds_match_the_prototypes():
    # every ctypes argument list has the header prototype's length and kinds, in order
    text = re.sub(r"/\*.*?\*/", "", open(HEADER, encoding="utf-8").read(), flags=re.S)
    protos = dict(re.findall(r"\b(attn_\w+)\s*\(([^)]*)\)\s*;", text))
    assert set(protos) == set(mk._SIGNATURES)
    for name, args in protos.items():
        params = [] if args.strip() in ("", "void") else args.split(",")
        want = [_kind(p) for p in params]
        got = [_CTYPE_KIND[t] for t in mk._SIGNATURES[name][1]]
        assert got == want, name

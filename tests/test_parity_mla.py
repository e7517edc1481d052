"""MLA absorbed decode on the GPU against the fp64 CPU oracle (max |Δ| ≤ 3e-3).

The query absorption q_lat = W_UKᵀ q_nope happens before the library call (in fp32 from the
bf16 inputs, rounded to bf16); the kernel and the oracle see the same rounded q_lat. The
oracle's own absorbed = decompressed identity is pinned on the CPU in test_oracle_pins.
"""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from tests import mla_bounds as mb
from workloads import to_f64

pytestmark = pytest.mark.gpu

TOL = 3e-3
DEV = "cuda"


def absorb_on_device(q_nope, w_uk):
    return torch.einsum("hnr,bhn->bhr", w_uk.float(), q_nope.float()).to(torch.bfloat16).contiguous()


def _run(inp, scale, **kw):
    q_lat = absorb_on_device(inp["q_nope"], inp["w_uk"])
    out = mk.decode_mla_absorbed(q_lat, inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["seq_lens"], scale, **kw)
    torch.cuda.synchronize()
    return q_lat, out


def _ref(inp, q_lat, scale):
    return oracle.mla_decode_absorbed(to_f64(q_lat), to_f64(inp["q_rope"]), to_f64(inp["c_cache"]),
                                      to_f64(inp["kr_cache"]), inp["seq_lens"].cpu().numpy(), scale)


def test_minimind_mla_full():
    w = W.MINIMIND_MLA
    inp = W.mla_inputs(w, DEV)
    q_lat, out = _run(inp, w.scale)
    err = np.abs(out.cpu().double().numpy() - _ref(inp, q_lat, w.scale)).max()
    assert err <= TOL, err


@pytest.mark.parametrize("n_split", [0, 1, 3, 16])
@pytest.mark.parametrize("hq", [16, 32])
def test_ragged_and_splits(n_split, hq):
    lens = (0, 1, 63, 64, 65, 300, 1000)
    w = W.MlaWorkload("mla_ragged", 3, len(lens), hq, 96, 128, 48, 96, 1000, lengths=lens, sub=3)
    inp = W.mla_inputs(w, DEV)
    q_lat, out = _run(inp, w.scale, n_split=n_split)
    err = np.abs(out.cpu().double().numpy() - _ref(inp, q_lat, w.scale)).max()
    assert err <= TOL, err
    assert torch.all(out[0] == 0)


def test_single_token_is_c0():
    w = W.MlaWorkload("mla_one", 3, 2, 16, 96, 128, 48, 96, 8, lengths=(1, 1))
    inp = W.mla_inputs(w, DEV)
    _, out = _run(inp, w.scale)
    c0 = inp["c_cache"][:, 0].float()[:, None, :].expand(-1, 16, -1)
    assert torch.equal(out, c0)


def test_decompressed_output_close_to_naive():
    # kernel + W_UV applied in fp64 vs the oracle's decompress-then-attend path on the same
    # bf16 inputs: they differ by the bf16 rounding of the fp32 q_lat (bounded per score,
    # then per latent average) and the decode's own tolerance, each mapped through W_UV
    # (tests/mla_bounds.py states the derivation)
    w = W.MlaWorkload("mla_naive", 3, 4, 16, 96, 128, 48, 96, 256, lengths=(256, 100, 17, 200))
    inp = W.mla_inputs(w, DEV)
    q_lat, out = _run(inp, w.scale)
    o = oracle.apply_uv(out.cpu().double().numpy(), to_f64(inp["w_uv"]))
    ref = oracle.mla_decode_naive(to_f64(inp["q_nope"]), to_f64(inp["q_rope"]), to_f64(inp["c_cache"]),
                                  to_f64(inp["kr_cache"]), to_f64(inp["w_uk"]), to_f64(inp["w_uv"]),
                                  inp["seq_lens"].cpu().numpy(), w.scale)
    assert np.all(np.abs(o - ref) <= mb.full_step_tolerance(inp, w.scale, oracle))


@pytest.mark.parametrize("B", [1200, 3000])
def test_large_batches(B):
    """Past about 1000 sequences the per-sequence tables (8 bytes each in shared memory) leave
    room for one block per SM instead of two, so the persistent blocks of the split run in two
    waves; short ragged lengths, every output compared."""
    w = W.MlaWorkload("mla_large_b", 3, B, 16, 96, 128, 48, 96, 48, length_range=(0, 48), sub=7)
    inp = W.mla_inputs(w, DEV)
    q_lat, out = _run(inp, w.scale)
    mk.check_status()
    err = np.abs(out.cpu().double().numpy() - _ref(inp, q_lat, w.scale)).max()
    assert err <= TOL, err


def test_long_context():
    """MLA over 131072 and 70001 latent rows, every output compared."""
    w = W.MlaWorkload("mla_128k", 3, 2, 16, 96, 128, 48, 96, 131072, lengths=(131072, 70001), sub=8)
    inp = W.mla_inputs(w, DEV)
    q_lat, out = _run(inp, w.scale)
    mk.check_status()
    err = np.abs(out.cpu().double().numpy() - _ref(inp, q_lat, w.scale)).max()
    assert err <= TOL, err

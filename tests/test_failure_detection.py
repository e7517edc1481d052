"""Bounded waits: a wait that never completes makes its kernel give up, record the failure in
a device status word and return; the host learns of it from attn_check_status, and the GPU
context stays usable. The wait that runs out here is on an mbarrier nothing arrives on, with
a bound of 1e5 SM cycles (about 50 us); no memory outside the block is touched."""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    mk.check_status()                              # start from a clean status
    mk.selftest_bounded_wait(100_000)
    with pytest.raises(mk.MlakvError) as e:
        mk.check_status()
    assert e.value.code == mk.ATTN_ERR_TIMEOUT
    mk.check_status()                              # the flag was read and cleared
    # the context still runs kernels correctly
    w = W.DecodeWorkload("after_timeout", 0, 2, 8, 2, 128, 200, "bf16", lengths=(200, 33), sub=19)
    inp = W.decode_inputs(w, "cuda")
    out = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], inp["seq_lens"])
    mk.check_status()
    ref = oracle.decode_gqa(to_f64(inp["q"]), to_f64(inp["k_cache"]), to_f64(inp["v_cache"]),
                            inp["seq_lens"].cpu().numpy(), w.scale)
    assert float(np.abs(out.cpu().double().numpy() - ref).max()) <= 3e-3

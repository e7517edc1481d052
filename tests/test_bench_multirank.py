"""The N > 1 path of bench.py on the CPU: two gloo ranks. Each rank runs an independent
replica on its own sequences (inputs seeded per rank), the job's time is the slowest rank's
(maximum over ranks), and the reported value counts the units of every rank."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Wl:
    kind = "decode"
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_gqa_bf16.cu"
    call = "attn_decode_gqa call: "
    launch_note = ""
    name = "test"
    launches_per_step = 1

    def __init__(self):
        self.w = W.MINIMIND_GQA
        self.bytes_per_step = 1_000_000_000

    def describe(self):
        return {"workload": "test"}


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank inputs: the seed advances by 1000 per rank, as bench.py draws them
        w = W.MINIMIND_GQA
        inp = W.decode_inputs(w, "cpu", seed=w.seed + 1000 * rank)
        checksum = float(inp["k_cache"][:2, :8].float().sum())
        # rank r "took" (1 + r) / 10 seconds per step, and 0.5 + r seconds end to end
        secs, e2e = bench.max_over_ranks([(1.0 + rank) / 10, 0.5 + rank], torch.device("cpu"))
        t = {"seconds_per_call": secs, "calls_per_run": 10, "runs": 5, "timed_s": 5 * 10 * secs,
             "spread": (secs, secs), "clocks": None}
        peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1700.0}
        head = bench.summarize(_Wl(), t, peaks, "test", world)
        e2e_line = bench.e2e_line(_Wl(), e2e, 0, 0, world)
        out[rank] = (secs, e2e, head["value"], e2e_line["value"], checksum)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    (s0, e0, v0, ev0, c0), (s1, e1, v1, ev1, c1) = out[0], out[1]
    # both ranks agree on the slowest rank's times
    assert s0 == s1 == 0.2 and e0 == e1 == 1.5
    # whole-job throughput: world x bytes per step / slowest time per step
    assert v0 == v1 == pytest.approx(world * 1e9 / (2.0 / 10) / 1e9, rel=1e-6)
    assert ev0 == pytest.approx(world * 1e9 / 1.5 / 1e9, rel=1e-3)
    # the replicas stream different sequences
    assert c0 != c1


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]

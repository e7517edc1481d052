#!/usr/bin/env python
"""Benchmark of the KV-cache attention hot path on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Headline workload (default): the Llama-3-8B-shaped layer decode with 8 KV heads (GQA) —
B=64, Hq=32, Hkv=8, D=128, bf16 cache, 8192 cached tokens per sequence, one new query token
per sequence; a step is one ``attn_decode_gqa`` call over the whole batch. ``value`` =
algorithmic KV bytes read per step (each cached K/V element once) ÷ the device time per
step, in GB/s, with the inputs resident in HBM (the 2 GiB cache is 16× the L2; smaller
workloads cycle through enough distinct input sets to cover ≥ 4× the L2).

Timing: the calls are captured in a CUDA graph and replayed; each of 5 timed runs covers at
least ``--steps`` calls and at least 50 ms, timed with CUDA events on the launching stream;
the median run gives ``ms_per_step`` (``timing`` in the line says how many calls a run
held). Clocks are sampled during the runs.

The line also carries: ``roofline`` (the achieved GB/s against the measured HBM copy
bandwidth, and the DRAM traffic per launch from the committed ncu summary when the kernel
source is unchanged), ``e2e`` (the same metric through the Python API with the inputs copied
in from pinned host memory and the output copied back inside the timed region),
``cpu_baseline`` (the fp64 CPU oracle on the host cores, bounded sample), ``clocks``,
``gpu_launches`` and, last, ``also``: one short entry per other workload (the Llama layer
with 32 and 1 KV heads, the MiniMind GQA decode alone, with its cache append, over an fp8
cache and as a 4-token chunk, MLA decode alone, its full step and a 4-token chunk, and
causal prefill uniform and ragged), each with its own roofline fraction and oracle rate.

``--impl reference`` times the fp64 CPU oracle (the only reference this path has) on the
same workload and metric, on the host cores, and prints the same line with
``"impl": "reference"``. Under torchrun with N > 1 each rank runs an independent replica
on its own GPU and its own sequences (weak scaling, no collective on the data path);
rank 0 prints the aggregate.
"""

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "decode attn KV-read HBM GB/s (% of ~8 TB/s), tokens/s; prefill TFLOP/s"
NOMINAL_HBM_GBS = 8000.0
HEADLINE = "llama_hkv8"
MIN_RUN_S = 0.05          # each timed run lasts at least this long
N_RUNS = 5                # timed runs per workload; the median is reported
ORACLE_HOST_BYTES = 512 << 20   # fp32 host copies handed to the oracle, per workload
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ============================================================================ environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device):
    """Element-wise maximum of `values` (floats) over all ranks of the default process group
    (unchanged without one): the job's time is its slowest rank's. `device` holds the
    reduction buffer (the GPU for NCCL, the CPU for gloo)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


class ClockSampler:
    """Samples of the SM clock and the clock-event reasons taken while the timed region runs:
    NVML through pynvml when it is importable, else ``nvidia-smi --query-gpu ... -lms``."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, device_index, period_s=0.02):
        self.samples, self.reasons, self.max_mhz, self.error = [], set(), None, None
        self.period, self.stop_flag, self.thread, self.h, self.proc = period_s, threading.Event(), None, None, None
        props = torch.cuda.get_device_properties(device_index)
        try:
            self.bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        except Exception:
            self.bus = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            try:
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(self.bus.encode())
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception as e:
            self.error = f"pynvml: {e!r}; using nvidia-smi"
            self.h = None

    def _add_reasons(self, mask):
        for bit, name in self.REASONS.items():
            if mask & bit and bit != 0x1:
                self.reasons.add(name)

    def _run_nvml(self):
        while not self.stop_flag.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                self._add_reasons(self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h))
            except Exception:
                pass
            time.sleep(self.period)

    def _run_smi(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                self.samples.append(float(parts[0]))
                self.max_mhz = float(parts[1])
                self._add_reasons(int(parts[2], 16))
            except ValueError:
                pass

    def __enter__(self):
        if self.h is not None:
            self.thread = threading.Thread(target=self._run_nvml, daemon=True)
            self.thread.start()
            return self
        import subprocess
        cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", str(int(self.period * 1000))]
        if self.bus:
            cmd += ["-i", self.bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._run_smi, daemon=True)
            self.thread.start()
            time.sleep(0.3)    # let the first sample land before the timed work starts
        except Exception as e:
            self.error = f"{self.error}; nvidia-smi: {e!r}"
        return self

    def __exit__(self, *exc):
        self.stop_flag.set()
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
               "reasons": sorted(self.reasons), "samples": len(self.samples),
               "source": "nvml" if self.h is not None else "nvidia-smi"}
        if not self.samples:
            out["error"] = self.error or "no sample taken"
        return out


def source_sha(relpath):
    with open(os.path.join(ROOT, relpath), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_src, workload_name):
    """DRAM bytes per launch from a committed ncu summary, if its kernel source is unchanged.

    profiles/*.md lines of the form
      traffic: <workload> <kernel_src> <source_sha16> <bytes_per_launch>
    """
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = source_sha(kernel_src)
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        for line in open(os.path.join(pdir, fn), encoding="utf-8"):
            parts = line.strip().split()
            if len(parts) == 5 and parts[0] == "traffic:" and parts[1] == workload_name and parts[2] == kernel_src:
                if parts[3] == sha:
                    return float(parts[4])
    return None


# ============================================================================ workloads

def _f32(t):
    """Host fp32 copy of a tensor's exact values (bf16 widens exactly), for the oracle."""
    return t.detach().to("cpu", torch.float32).numpy()


def _host(t):
    return t.detach().cpu().numpy()


class DecodeGqa:
    kind = "decode"
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_gqa_bf16.cu"
    call = "attn_decode_gqa call: "
    launch_note = " (one launch, split segments merged in-kernel)"

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device = mk, w, device
        self.name = w.name
        self.sets = []
        first = W.decode_inputs(w, device, seed=w.seed + 1000 * rank)
        self.lens = first["seq_lens"].cpu().numpy()
        elt = 2 if w.dtype == "bf16" else 4
        self.bytes_per_step = int(self.lens.sum()) * 2 * w.n_kv_heads * w.head_dim * elt
        self.flops_per_step = 4 * w.head_dim * w.n_q_heads * int(self.lens.sum())
        cache_bytes = first["k_cache"].nbytes * 2
        n_sets = max(1, math.ceil(4 * l2_bytes / max(cache_bytes, 1)))
        self.sets.append(first)
        for i in range(1, n_sets):
            s = W.decode_inputs(w, device, seed=w.seed + 1000 * rank)
            self.sets.append(s)
        self.max_s = int(self.lens.max())
        self.out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device=device)
        code = mk.ATTN_BF16 if w.dtype == "bf16" else mk.ATTN_F32
        self.n_split = mk.decode_gqa_num_splits(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, self.max_s, code)
        nb = mk.decode_gqa_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, self.max_s, code)
        self.ws = torch.zeros(max(nb, 1), dtype=torch.uint8, device=device)
        # bf16 caches: one launch (split segments are merged inside it); fp32: decode + merge
        self.launches_per_step = 1 if w.dtype == "bf16" else 1 + (self.n_split > 1)
        g = w.n_q_heads // w.n_kv_heads
        if w.dtype == "bf16" and w.head_dim == 128 and g % 16 == 0:
            self.kernel_src = "mla_kv_cache_flash_b300/csrc/decode_tc.cu"
        self.l2_note = f"rotating {n_sets} distinct cache sets ({n_sets * cache_bytes / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def step(self, i):
        s = self.sets[i % len(self.sets)]
        self.mk.decode_gqa(s["q"], s["k_cache"], s["v_cache"], s["seq_lens"], out=self.out, scale=self.w.scale,
                           max_s=self.max_s, workspace=self.ws)

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q", "k_cache", "v_cache", "seq_lens")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self.mk.decode_gqa(dev_bufs["q"], dev_bufs["k_cache"], dev_bufs["v_cache"], dev_bufs["seq_lens"],
                           out=self.out, scale=self.w.scale, max_s=self.max_s, workspace=self.ws)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "decode"

    def _oracle_seqs(self, per_seq_bytes):
        """How many sequences (the first ones) the oracle gets: all of them, or as many as fit
        in ORACLE_HOST_BYTES of host copies (the workloads this cuts have equal lengths)."""
        return int(max(1, min(self.w.batch, ORACLE_HOST_BYTES // max(per_seq_bytes, 1))))

    def oracle_payload(self):
        """(host arrays, units, sequences covered) for the oracle; one unit = (sequence, KV head)."""
        s = self.sets[0]
        n = self._oracle_seqs(2 * s["k_cache"][0].numel() * 4)
        arrays = {"q": _f32(s["q"][:n]), "k": _f32(s["k_cache"][:n]), "v": _f32(s["v_cache"][:n]),
                  "lens": self.lens[:n]}
        return arrays, [(b, j) for b in range(n) for j in range(self.w.n_kv_heads)], n

    def unit_work(self, unit):
        elt = 2 if self.w.dtype == "bf16" else 4
        return int(self.lens[unit[0]]) * 2 * self.w.head_dim * elt

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "Hkv": w.n_kv_heads, "D": w.head_dim,
                "S_max": w.s_max, "lengths": (f"uniform[{w.length_range[0]},{w.length_range[1]}] seed {w.seed}"
                                              if w.length_range else f"all {int(self.lens[0])}"),
                "sum_lengths": int(self.lens.sum()), "n_split": self.n_split, "cache_dtype": w.dtype,
                "l2": self.l2_note}


class DecodeGqaStep(DecodeGqa):
    """A whole GQA decode step: the new token's q and k rotated and k, v written into the
    cache (attn_kv_append_rope), then the decode over the cache that holds it. Each sequence's
    new token is its last cached row (position = length − 1), so the decode reads the same
    bytes as the decode-only workload; the append's own bytes are added."""
    call = "attn_kv_append_rope + attn_decode_gqa; dominant: "

    def __init__(self, w, device, rank, l2_bytes):
        super().__init__(w, device, rank, l2_bytes)
        for i, s in enumerate(self.sets):
            new = W.append_inputs(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.s_max, device,
                                  seed=w.seed + 500 + i + 1000 * rank)
            s.update(new)
            s["pos"] = (s["seq_lens"] - 1).contiguous()
        B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
        self.bytes_per_step += B * (2 * Hq * D * 2 + 4 * Hkv * D * 2 + D * 4 + 8)
        self.q_rot = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.new_lens = torch.empty(B, dtype=torch.int32, device=device)
        self.launches_per_step = 2

    def _run(self, s):
        mk = self.mk
        mk.kv_append_rope(s["q"], s["k_new"], s["v_new"], s["pos"], s["freqs_cis"], s["k_cache"], s["v_cache"],
                          q_out=self.q_rot, new_lens=self.new_lens)
        mk.decode_gqa(self.q_rot, s["k_cache"], s["v_cache"], self.new_lens, out=self.out, scale=self.w.scale,
                      max_s=self.max_s, workspace=self.ws)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q", "k_new", "v_new", "pos", "freqs_cis", "k_cache", "v_cache")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "step"

    def oracle_payload(self):
        s = self.sets[0]
        n = self._oracle_seqs(2 * s["k_cache"][0].numel() * 4)
        arrays = {k: _f32(s[k][:n]) for k in ("q", "k_new", "v_new", "k_cache", "v_cache")}
        arrays.update(pos=_host(s["pos"][:n]), freqs_cis=_f32(s["freqs_cis"]))
        return arrays, [(b,) for b in range(n)], n

    def unit_work(self, unit):
        w = self.w
        append = 2 * w.n_q_heads * w.head_dim * 2 + 4 * w.n_kv_heads * w.head_dim * 2 + w.head_dim * 4 + 8
        return int(self.lens[unit[0]]) * 2 * w.n_kv_heads * w.head_dim * 2 + append

    def describe(self):
        return dict(super().describe(), workload=self.name,
                    launches="append the new token with RoPE at position length-1, then decode")


class DecodeGqaFp8(DecodeGqa):
    """The MiniMind decode batch over an E4M3 cache with per-row fp32 K and V scales.
    Algorithmic bytes: each live code once plus its row's scale."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_fp8.cu"
    call = "attn_decode_gqa_fp8 call: "
    launch_note = " (tensor-core fp8 decode over persistent blocks, shared segments merged in-kernel)"

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device, self.name = mk, w, device, w.name
        first = W.fp8_decode_inputs(w, device, seed=w.seed + 1000 * rank)
        self.lens = first["seq_lens"].cpu().numpy()
        self.bytes_per_step = int(self.lens.sum()) * 2 * w.n_kv_heads * (w.head_dim + 4)
        self.flops_per_step = 4 * w.head_dim * w.n_q_heads * int(self.lens.sum())
        cache_bytes = 2 * (first["k_cache"].nbytes + first["k_scale"].nbytes)
        n_sets = max(1, math.ceil(4 * l2_bytes / cache_bytes))
        self.sets = [first] + [W.fp8_decode_inputs(w, device, seed=w.seed + 1000 * rank) for _ in range(n_sets - 1)]
        self.max_s = int(self.lens.max())
        self.out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device=device)
        self.n_split = mk.decode_gqa_num_splits(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, self.max_s,
                                                mk.ATTN_FP8_E4M3)
        nb = mk.decode_gqa_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, self.max_s,
                                          mk.ATTN_FP8_E4M3)
        self.ws = torch.zeros(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 1      # two query heads per KV head: the one-launch tensor-core kernel
        self.l2_note = f"rotating {n_sets} distinct fp8 caches ({n_sets * cache_bytes / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def _run(self, s):
        self.mk.decode_gqa_fp8(s["q"], s["k_cache"], s["v_cache"], s["k_scale"], s["v_scale"], s["seq_lens"],
                               out=self.out, scale=self.w.scale, max_s=self.max_s, workspace=self.ws)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q", "k_cache", "v_cache", "k_scale", "v_scale", "seq_lens")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "fp8"

    def oracle_payload(self):
        s = self.sets[0]
        arrays = {"q": _f32(s["q"]), "k": _host(s["k_cache"]), "v": _host(s["v_cache"]),
                  "k_scale": _host(s["k_scale"]), "v_scale": _host(s["v_scale"]), "lens": self.lens}
        return arrays, [(b, j) for b in range(self.w.batch) for j in range(self.w.n_kv_heads)], self.w.batch

    def unit_work(self, unit):
        return int(self.lens[unit[0]]) * 2 * (self.w.head_dim + 4)

    def describe(self):
        return dict(super().describe(), cache_dtype="fp8_e4m3 + fp32 scale per row")


class DecodeChunked(DecodeGqa):
    """Chunks of 4 new tokens per sequence over the MiniMind caches (a speculative-decoding
    style step): each sequence's last 4 cached rows are its chunk, so row i sees
    length − 4 + i + 1 rows. Algorithmic bytes: each sequence's visible K/V once (as for the
    decode of the full length); the kernel reads them once per new token."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_gqa_bf16.cu"
    call = "attn_prefill_gqa_chunked call: "
    launch_note = (" (register-MMA decode kernel: 16/G new tokens x G heads per MMA tile, balanced over persistent"
                   " blocks, shared segments merged in-kernel)")
    n_new = 4

    def __init__(self, w, device, rank, l2_bytes):
        super().__init__(w, device, rank, l2_bytes)
        B, n = w.batch, self.n_new
        for i, s in enumerate(self.sets):
            g = torch.Generator(device=device).manual_seed(w.seed + 700 + i + 1000 * rank)
            s["q_chunk"] = torch.randn((B * n, w.n_q_heads, w.head_dim), generator=g, device=device).to(torch.bfloat16)
            s["cu_q"] = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=device)
            s["start_pos"] = (s["seq_lens"] - n).clamp_min(0).contiguous()
        self.out = torch.empty((B * n, w.n_q_heads, w.head_dim), dtype=torch.float32, device=device)
        lib = self.mk.lib()
        nb = int(lib.attn_prefill_gqa_chunked_workspace_size(B, B * n, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                             self.max_s, self.mk.ATTN_BF16, 0))
        self.ws = torch.zeros(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 1          # one launch; the workspace holds counters and partials

    def _run(self, s):
        self.mk.prefill_gqa_chunked(s["q_chunk"], s["k_cache"], s["v_cache"], s["cu_q"], s["start_pos"], self.max_s,
                                    out=self.out, scale=self.w.scale, workspace=self.ws)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_chunk", "k_cache", "v_cache", "cu_q", "start_pos")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "chunk"

    def oracle_payload(self):
        s = self.sets[0]
        arrays = {"q": _f32(s["q_chunk"]), "k": _f32(s["k_cache"]), "v": _f32(s["v_cache"]),
                  "cu_q": _host(s["cu_q"]), "start_pos": _host(s["start_pos"])}
        return arrays, [(b,) for b in range(self.w.batch)], self.w.batch

    def unit_work(self, unit):
        return int(self.lens[unit[0]]) * 2 * self.w.n_kv_heads * self.w.head_dim * 2

    def describe(self):
        return dict(super().describe(), workload=self.name, new_tokens_per_sequence=self.n_new,
                    launches="chunked prefill: 4 new tokens per sequence over its cache")


class DecodeMla(DecodeGqa):
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_tc.cu"
    call = "attn_decode_mla_absorbed call: "

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device, self.name = mk, w, device, w.name
        first = W.mla_inputs(w, device, seed=w.seed + 1000 * rank)
        self.lens = first["seq_lens"].cpu().numpy()
        row = (w.kv_lora_rank + w.rope_dim) * 2
        self.bytes_per_step = int(self.lens.sum()) * row
        self.flops_per_step = int(self.lens.sum()) * w.n_q_heads * (2 * (w.kv_lora_rank + w.rope_dim)
                                                                    + 2 * w.kv_lora_rank)
        cache_bytes = first["c_cache"].nbytes + first["kr_cache"].nbytes
        n_sets = max(1, math.ceil(4 * l2_bytes / cache_bytes))
        self.sets = []
        for i in range(n_sets):
            s = first if i == 0 else W.mla_inputs(w, device, seed=w.seed + 1000 * rank)
            s["q_lat"] = torch.einsum("hnr,bhn->bhr", s["w_uk"].float(), s["q_nope"].float()).to(torch.bfloat16).contiguous()
            self.sets.append(s)
        self.max_s = int(self.lens.max())
        self.out = torch.empty((w.batch, w.n_q_heads, w.kv_lora_rank), dtype=torch.float32, device=device)
        self.n_split = mk.decode_mla_num_splits(w.batch, w.n_q_heads, w.kv_lora_rank, w.rope_dim, self.max_s)
        nb = mk.decode_mla_workspace_size(w.batch, w.n_q_heads, w.kv_lora_rank, w.rope_dim, self.max_s)
        self.ws = torch.zeros(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 1
        self.l2_note = f"rotating {n_sets} distinct latent caches ({n_sets * cache_bytes / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def step(self, i):
        s = self.sets[i % len(self.sets)]
        self.mk.decode_mla_absorbed(s["q_lat"], s["q_rope"], s["c_cache"], s["kr_cache"], s["seq_lens"], self.w.scale,
                                    out_lat=self.out, max_s=self.max_s, workspace=self.ws)

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_lat", "q_rope", "c_cache", "kr_cache", "seq_lens")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        d = dev_bufs
        self.mk.decode_mla_absorbed(d["q_lat"], d["q_rope"], d["c_cache"], d["kr_cache"], d["seq_lens"], self.w.scale,
                                    out_lat=self.out, max_s=self.max_s, workspace=self.ws)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "mla"

    def oracle_payload(self):
        s = self.sets[0]
        arrays = {"q_lat": _f32(s["q_lat"]), "q_rope": _f32(s["q_rope"]), "c": _f32(s["c_cache"]),
                  "kr": _f32(s["kr_cache"]), "lens": self.lens}
        return arrays, [(b,) for b in range(self.w.batch)], self.w.batch

    def unit_work(self, unit):
        return int(self.lens[unit[0]]) * (self.w.kv_lora_rank + self.w.rope_dim) * 2

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "kv_lora_rank": w.kv_lora_rank,
                "rope_dim": w.rope_dim, "S": int(self.lens[0]), "n_split": self.n_split, "cache_dtype": "bf16",
                "l2": self.l2_note}


class DecodeMlaStep(DecodeMla):
    """The whole MLA decode step: W_UK absorbed into the query, the latent decode, W_UV on its
    output (three launches). Algorithmic bytes: the cache rows read plus both weight tensors."""
    call = "attn_mla_absorb_query + attn_decode_mla_absorbed + attn_mla_apply_uv; dominant: "

    def __init__(self, w, device, rank, l2_bytes):
        super().__init__(w, device, rank, l2_bytes)
        self.bytes_per_step += (self.sets[0]["w_uk"].nbytes + self.sets[0]["w_uv"].nbytes)
        self.out_lat = self.out
        self.out = torch.empty((w.batch, w.n_q_heads, w.v_head_dim), dtype=torch.float32, device=device)
        self.q_lat = torch.empty((w.batch, w.n_q_heads, w.kv_lora_rank), dtype=torch.bfloat16, device=device)
        self.launches_per_step = 3

    def _run(self, s):
        mk = self.mk
        mk.mla_absorb_query(s["q_nope"], s["w_uk"], q_lat=self.q_lat)
        mk.decode_mla_absorbed(self.q_lat, s["q_rope"], s["c_cache"], s["kr_cache"], s["seq_lens"], self.w.scale,
                               out_lat=self.out_lat, max_s=self.max_s, workspace=self.ws)
        mk.mla_apply_uv(self.out_lat, s["w_uv"], out=self.out)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_nope", "q_rope", "c_cache", "kr_cache", "w_uk", "w_uv",
                                                     "seq_lens")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "mla_step"

    def oracle_payload(self):
        s = self.sets[0]
        arrays = {k: _f32(s[k]) for k in ("q_nope", "q_rope", "w_uk", "w_uv")}
        arrays.update(c=_f32(s["c_cache"]), kr=_f32(s["kr_cache"]), lens=self.lens)
        return arrays, [(b,) for b in range(self.w.batch)], self.w.batch

    def unit_work(self, unit):
        s = self.sets[0]
        weights = (s["w_uk"].nbytes + s["w_uv"].nbytes) // self.w.batch
        return int(self.lens[unit[0]]) * (self.w.kv_lora_rank + self.w.rope_dim) * 2 + weights

    def describe(self):
        return dict(super().describe(), workload=self.name, nope_dim=self.w.nope_dim, v_head_dim=self.w.v_head_dim,
                    launches="absorb W_UK, latent decode, apply W_UV")


class MlaChunked(DecodeMla):
    """MLA chunked prefill, 4 new tokens per sequence over the MiniMind MLA latent caches
    (each sequence's last 4 rows are its chunk). Algorithmic bytes: each visible latent row
    once, as for the decode of the full length."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_tc.cu"
    call = "attn_prefill_mla_chunked call: "
    launch_note = (" (tcgen05 MLA decode kernel: 4 new tokens x 16 heads per block, balanced over persistent"
                   " blocks, shared segments merged in-kernel)")
    n_new = 4

    def __init__(self, w, device, rank, l2_bytes):
        super().__init__(w, device, rank, l2_bytes)
        B, n = w.batch, self.n_new
        for i, s in enumerate(self.sets):
            g = torch.Generator(device=device).manual_seed(w.seed + 800 + i + 1000 * rank)
            s["q_lat_chunk"] = torch.randn((B * n, w.n_q_heads, w.kv_lora_rank), generator=g,
                                           device=device).to(torch.bfloat16)
            s["q_rope_chunk"] = torch.randn((B * n, w.n_q_heads, w.rope_dim), generator=g,
                                            device=device).to(torch.bfloat16)
            s["cu_q"] = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=device)
            s["start_pos"] = (s["seq_lens"] - n).clamp_min(0).contiguous()
        self.out = torch.empty((B * n, w.n_q_heads, w.kv_lora_rank), dtype=torch.float32, device=device)
        nb = int(self.mk.lib().attn_prefill_mla_chunked_workspace_size(B, B * n, w.n_q_heads, self.max_s, 0))
        self.ws = torch.zeros(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 1          # one launch; the workspace holds counters and partials

    def _run(self, s):
        self.mk.prefill_mla_chunked(s["q_lat_chunk"], s["q_rope_chunk"], s["c_cache"], s["kr_cache"], s["cu_q"],
                                    s["start_pos"], self.max_s, self.w.scale, out_lat=self.out, workspace=self.ws)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_lat_chunk", "q_rope_chunk", "c_cache", "kr_cache", "cu_q",
                                                     "start_pos")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "mla_chunk"

    def oracle_payload(self):
        s = self.sets[0]
        arrays = {"q_lat": _f32(s["q_lat_chunk"]), "q_rope": _f32(s["q_rope_chunk"]), "c": _f32(s["c_cache"]),
                  "kr": _f32(s["kr_cache"]), "cu_q": _host(s["cu_q"]), "start_pos": _host(s["start_pos"])}
        return arrays, [(b,) for b in range(self.w.batch)], self.w.batch

    def describe(self):
        return dict(super().describe(), workload=self.name, new_tokens_per_sequence=self.n_new)


class Prefill:
    kind = "prefill"
    kernel_src = "mla_kv_cache_flash_b300/csrc/prefill.cu"
    call_name = "attn_prefill_gqa_causal"

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device, self.name = mk, w, device, w.name
        first = W.prefill_inputs(w, device, seed=w.seed + 1000 * rank)
        self.lens = first["lengths"]
        self.flops_per_step = sum(4 * w.head_dim * w.n_q_heads * int(s) * (int(s) + 1) // 2 for s in self.lens)
        io = first["q"].nbytes + first["k"].nbytes + first["v"].nbytes + first["q"].numel() * 4
        n_sets = max(1, math.ceil(4 * l2_bytes / io))
        self.sets = [first] + [W.prefill_inputs(w, device, seed=w.seed + 1000 * rank) for _ in range(n_sets - 1)]
        self.out = torch.empty((first["q"].shape[0], w.n_q_heads, w.head_dim), dtype=torch.float32, device=device)
        self.launches_per_step = 1
        self.bytes_per_step = io
        self.l2_note = f"rotating {n_sets} input sets ({n_sets * io / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def step(self, i):
        s = self.sets[i % len(self.sets)]
        self.mk.prefill_gqa_causal(s["q"], s["k"], s["v"], s["cu_seqlens"], s["max_seqlen"], out=self.out,
                                   scale=self.w.scale)

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q", "k", "v", "cu_seqlens")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self.mk.prefill_gqa_causal(dev_bufs["q"], dev_bufs["k"], dev_bufs["v"], dev_bufs["cu_seqlens"],
                                   self.sets[0]["max_seqlen"], out=self.out, scale=self.w.scale)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "prefill"

    def oracle_payload(self):
        """The first sequence of the batch (1 of 8): its packed rows, one unit per query head."""
        s = self.sets[0]
        n = int(self.lens[0])
        arrays = {"q": _f32(s["q"][:n]), "k": _f32(s["k"][:n]), "v": _f32(s["v"][:n]),
                  "cu": np.array([0, n], dtype=np.int64)}
        return arrays, [(0, h) for h in range(self.w.n_q_heads)], 1

    def unit_work(self, unit):
        n = int(self.lens[0])
        return 4 * self.w.head_dim * n * (n + 1) // 2

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "Hkv": w.n_kv_heads, "D": w.head_dim,
                "lengths": [int(x) for x in self.lens], "causal_flops": self.flops_per_step, "l2": self.l2_note}


class ChunkedPrefill(Prefill):
    """Chunked prefill of long chunks over existing caches: each sequence's last n_new cached
    rows are its new tokens (start_pos = S - n_new), so new row i sees start_pos + i + 1 rows.
    Algorithmic flops: 4·D per (new row, visible key) pair and query head (Q·Kᵀ and P·V)."""
    call_name = "attn_prefill_gqa_chunked (tcgen05 prefill kernel, K and V read from the caches)"
    n_new = 512

    def _make(self, seed):
        w, B, n = self.w, self.w.batch, self.n_new
        s = W.decode_inputs(w, self.device, seed=seed)
        del s["q"]
        g = torch.Generator(device=self.device).manual_seed(seed + 700)
        s["q_chunk"] = torch.randn((B * n, w.n_q_heads, w.head_dim), generator=g, device=self.device).to(torch.bfloat16)
        s["cu_q"] = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=self.device)
        s["start_pos"] = (s["seq_lens"] - n).contiguous()
        return s

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device, self.name = mk, w, device, w.name
        first = self._make(w.seed + 1000 * rank)
        B, n, D = w.batch, self.n_new, w.head_dim
        self.start = [int(x) for x in first["start_pos"].cpu()]
        self.lens = np.full(B, n)                       # new tokens per sequence
        self.flops_per_step = sum(self._seq_flops(b) for b in range(B))
        io = first["q_chunk"].nbytes + first["k_cache"].nbytes + first["v_cache"].nbytes + B * n * w.n_q_heads * D * 4
        n_sets = max(1, math.ceil(4 * l2_bytes / io))
        self.sets = [first] + [self._make(w.seed + 1000 * rank) for _ in range(n_sets - 1)]
        self.out = torch.empty((B * n, w.n_q_heads, D), dtype=torch.float32, device=device)
        nb = int(mk.lib().attn_prefill_gqa_chunked_workspace_size(B, B * n, w.n_q_heads, w.n_kv_heads, D, w.s_max,
                                                                  mk.ATTN_BF16, 0))
        if nb != 0:
            raise RuntimeError("long chunks are expected on the prefill kernel (no workspace)")
        self.launches_per_step = 1
        self.bytes_per_step = io
        self.l2_note = f"rotating {n_sets} input sets ({n_sets * io / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def _seq_flops(self, b):
        n, kv0 = self.n_new, self.start[b]
        return 4 * self.w.head_dim * self.w.n_q_heads * (n * kv0 + n * (n + 1) // 2)

    def _run(self, s):
        self.mk.prefill_gqa_chunked(s["q_chunk"], s["k_cache"], s["v_cache"], s["cu_q"], s["start_pos"], self.w.s_max,
                                    out=self.out, scale=self.w.scale)

    def step(self, i):
        self._run(self.sets[i % len(self.sets)])

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_chunk", "k_cache", "v_cache", "cu_q", "start_pos")}

    def e2e_step(self, host, dev_bufs, out_host):
        for k, t in host.items():
            dev_bufs[k].copy_(t, non_blocking=True)
        self._run(dev_bufs)
        out_host.copy_(self.out, non_blocking=True)

    oracle_kind = "chunk"

    def oracle_payload(self):
        """The first sequence of the batch: its chunk and its caches, one unit."""
        s, n = self.sets[0], self.n_new
        arrays = {"q": _f32(s["q_chunk"][:n]), "k": _f32(s["k_cache"][:1]), "v": _f32(s["v_cache"][:1]),
                  "cu_q": np.array([0, n], dtype=np.int64), "start_pos": _host(s["start_pos"][:1])}
        return arrays, [(0,)], 1

    def unit_work(self, unit):
        return self._seq_flops(unit[0])

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "Hkv": w.n_kv_heads, "D": w.head_dim,
                "S_max": w.s_max, "start_pos": self.start[0], "new_tokens_per_sequence": self.n_new,
                "causal_flops": self.flops_per_step, "l2": self.l2_note}


class MlaChunkedPrefill(ChunkedPrefill):
    """MLA chunked prefill of long chunks (W_UK absorbed) over existing latent caches: each
    sequence's last n_new latent rows belong to its new tokens. Algorithmic flops per (new
    row, visible latent row, head): 2·(r + dr) for the score and 2·r for P·c."""
    call_name = "attn_prefill_mla_chunked (tcgen05 prefill kernel, MLA form: latent tiles as keys and values)"

    def _make(self, seed):
        w, B, n = self.w, self.w.batch, self.n_new
        s = W.mla_inputs(w, self.device, seed=seed)
        for k in ("q_nope", "q_rope", "w_uk", "w_uv"):
            del s[k]
        g = torch.Generator(device=self.device).manual_seed(seed + 800)
        s["q_lat_chunk"] = torch.randn((B * n, w.n_q_heads, w.kv_lora_rank), generator=g,
                                       device=self.device).to(torch.bfloat16)
        s["q_rope_chunk"] = torch.randn((B * n, w.n_q_heads, w.rope_dim), generator=g,
                                        device=self.device).to(torch.bfloat16)
        s["cu_q"] = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=self.device)
        s["start_pos"] = (s["seq_lens"] - n).contiguous()
        return s

    def __init__(self, w, device, rank, l2_bytes):
        import mla_kv_cache_flash_b300 as mk
        self.mk, self.w, self.device, self.name = mk, w, device, w.name
        first = self._make(w.seed + 1000 * rank)
        B, n, r = w.batch, self.n_new, w.kv_lora_rank
        self.start = [int(x) for x in first["start_pos"].cpu()]
        self.lens = np.full(B, n)
        self.flops_per_step = sum(self._seq_flops(b) for b in range(B))
        io = sum(first[k].nbytes for k in ("q_lat_chunk", "q_rope_chunk", "c_cache", "kr_cache")) + B * n * w.n_q_heads * r * 4
        n_sets = max(1, math.ceil(4 * l2_bytes / io))
        self.sets = [first] + [self._make(w.seed + 1000 * rank) for _ in range(n_sets - 1)]
        self.out = torch.empty((B * n, w.n_q_heads, r), dtype=torch.float32, device=device)
        if int(mk.lib().attn_prefill_mla_chunked_workspace_size(B, B * n, w.n_q_heads, w.s_max, 0)) != 0:
            raise RuntimeError("long chunks are expected on the prefill kernel (no workspace)")
        self.launches_per_step = 1
        self.bytes_per_step = io
        self.l2_note = f"rotating {n_sets} input sets ({n_sets * io / 1e6:.0f} MB, L2 {l2_bytes / 1e6:.0f} MB)"

    def _seq_flops(self, b):
        w, n, kv0 = self.w, self.n_new, self.start[b]
        return (2 * (w.kv_lora_rank + w.rope_dim) + 2 * w.kv_lora_rank) * w.n_q_heads * (n * kv0 + n * (n + 1) // 2)

    def _run(self, s):
        self.mk.prefill_mla_chunked(s["q_lat_chunk"], s["q_rope_chunk"], s["c_cache"], s["kr_cache"], s["cu_q"],
                                    s["start_pos"], self.w.s_max, self.w.scale, out_lat=self.out)

    def host_inputs(self):
        s = self.sets[0]
        return {k: s[k].cpu().pin_memory() for k in ("q_lat_chunk", "q_rope_chunk", "c_cache", "kr_cache", "cu_q",
                                                     "start_pos")}

    oracle_kind = "mla_chunk"

    def oracle_payload(self):
        """The first sequence of the batch: its chunk and its latent caches, one unit."""
        s, n = self.sets[0], self.n_new
        arrays = {"q_lat": _f32(s["q_lat_chunk"][:n]), "q_rope": _f32(s["q_rope_chunk"][:n]),
                  "c": _f32(s["c_cache"][:1]), "kr": _f32(s["kr_cache"][:1]),
                  "cu_q": np.array([0, n], dtype=np.int64), "start_pos": _host(s["start_pos"][:1])}
        return arrays, [(0,)], 1

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "r": w.kv_lora_rank, "dr": w.rope_dim,
                "S_max": w.s_max, "start_pos": self.start[0], "new_tokens_per_sequence": self.n_new,
                "causal_flops": self.flops_per_step, "l2": self.l2_note}


WORKLOADS = {
    "minimind_gqa": lambda: (DecodeGqa, W.MINIMIND_GQA),
    "llama_hkv32": lambda: (DecodeGqa, W.LLAMA3_8B[32]),
    "llama_hkv8": lambda: (DecodeGqa, W.LLAMA3_8B[8]),
    "llama_hkv1": lambda: (DecodeGqa, W.LLAMA3_8B[1]),
    "mla": lambda: (DecodeMla, W.MINIMIND_MLA),
    "minimind_gqa_fp8": lambda: (DecodeGqaFp8, dataclasses.replace(W.MINIMIND_GQA, name=W.MINIMIND_GQA.name + "_fp8")),
    "minimind_gqa_chunk4": lambda: (DecodeChunked, dataclasses.replace(W.MINIMIND_GQA, name=W.MINIMIND_GQA.name + "_chunk4")),
    "minimind_gqa_step": lambda: (DecodeGqaStep, dataclasses.replace(W.MINIMIND_GQA, name=W.MINIMIND_GQA.name + "_with_append")),
    "mla_chunk4": lambda: (MlaChunked, dataclasses.replace(W.MINIMIND_MLA, name=W.MINIMIND_MLA.name + "_chunk4")),
    "mla_step": lambda: (DecodeMlaStep, dataclasses.replace(W.MINIMIND_MLA, name=W.MINIMIND_MLA.name + "_full_step")),
    "prefill": lambda: (Prefill, W.PREFILL_UNIFORM),
    "prefill_ragged": lambda: (Prefill, W.PREFILL_RAGGED),
    "prefill_chunk512": lambda: (ChunkedPrefill, W.LLAMA3_8B_CHUNK512),
    "mla_prefill_chunk512": lambda: (MlaChunkedPrefill, W.MINIMIND_MLA_CHUNK512),
}
# the largest decode and prefill configurations come last, so a log's tail keeps them
ALSO = ("minimind_gqa", "minimind_gqa_step", "minimind_gqa_fp8", "minimind_gqa_chunk4", "mla_chunk4", "mla_step",
        "prefill_chunk512", "mla_prefill_chunk512", "llama_hkv32", "llama_hkv1", "mla", "prefill", "prefill_ragged")


# ============================================================================ timing

def time_workload(wl, steps, warmup, stream, barrier, sampler_index):
    """Median device time per call of wl.step.

    The calls are captured in one CUDA graph of L calls (cycling through the workload's input
    sets, so host launch cost is off the clock), replayed R times per timed run with R chosen
    so that a run covers at least `steps` calls and lasts at least MIN_RUN_S; N_RUNS runs are
    timed with CUDA events on the launching stream, bracketed by a barrier and a device
    synchronisation, and the median run gives the time per call. Clocks are sampled during
    the runs."""
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    n_sets = len(getattr(wl, "sets", [0]))
    L = n_sets * max(1, 64 // n_sets) if wl.kind == "decode" else max(n_sets, 8 // n_sets * n_sets)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(L):
            wl.step(i)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.replay()      # warm the graph itself
    ev0.record(stream)
    g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    est = max(ev0.elapsed_time(ev1) / 1e3, 1e-6)
    reps = max(math.ceil(steps / L), math.ceil(MIN_RUN_S / est))
    per_call, total = [], 0.0
    with ClockSampler(sampler_index) as clk:
        for _ in range(N_RUNS):
            barrier()
            torch.cuda.synchronize()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
            t = ev0.elapsed_time(ev1) / 1e3
            total += t
            per_call.append(t / (reps * L))
    del g
    return {"seconds_per_call": statistics.median(per_call), "calls_per_run": reps * L, "runs": N_RUNS,
            "timed_s": total, "spread": (min(per_call), max(per_call)), "clocks": clk.summary()}


def time_e2e(wl, device, barrier, n=20):
    """The same workload end to end through the Python API: every call first copies its inputs
    from pinned host memory and ends by copying the output back and waiting for it."""
    host = wl.host_inputs()
    dev_bufs = {k: torch.empty_like(v, device=device) for k, v in host.items()}
    out_host = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
    for _ in range(3):
        wl.e2e_step(host, dev_bufs, out_host)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(n):
        wl.e2e_step(host, dev_bufs, out_host)
        torch.cuda.current_stream().synchronize()   # the result is read on the host each call
    wall = time.perf_counter() - t0
    barrier()
    res = {"seconds": wall / n, "h2d": sum(v.nbytes for v in host.values()), "d2h": out_host.nbytes}
    del dev_bufs, host
    return res


def summarize(wl, t, peaks, peak_src, world):
    per_step = t["seconds_per_call"]
    if wl.kind == "decode":
        achieved = wl.bytes_per_step / per_step / 1e9
        value, unit = achieved * world, "GB/s"
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic(wl.kernel_src, wl.name),
                "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS hbm_gbs)",
                "algorithmic_bytes_per_launch": wl.bytes_per_step,
                "kernel": wl.call + os.path.basename(wl.kernel_src) + wl.launch_note,
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}
        extra = {"tokens_per_s": round(wl.w.batch * world / per_step, 1),
                 "pct_of_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2)}
    else:
        achieved = wl.flops_per_step / per_step / 1e12
        value, unit = achieved * world, "TFLOP/s"
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": profiled_traffic(wl.kernel_src, wl.name),
                "peak_source": f"{peak_src} dense bf16 burst (MEASURED_PEAKS bf16_tflops)",
                "algorithmic_flops_per_launch": wl.flops_per_step, "kernel": wl.call_name}
        extra = {"tokens_per_s": round(float(np.sum(wl.lens)) * world / per_step, 1)}
    out = {"value": round(value, 2), "unit": unit, "ms_per_step": round(per_step * 1e3, 5), "roofline": roof,
           "gpu_launches": t["runs"] * t["calls_per_run"] * wl.launches_per_step, "config": wl.describe(),
           "clocks": t["clocks"],
           "timing": {"calls_per_run": t["calls_per_run"], "runs": t["runs"], "statistic": "median",
                      "ms_per_call_min_max": [round(x * 1e3, 5) for x in t["spread"]],
                      "timed_s": round(t["timed_s"], 3)}}
    out.update(extra)
    return out


def e2e_line(wl, seconds, h2d, d2h, world):
    """The e2e entry: the workload's metric over the slowest rank's end-to-end time per call."""
    if wl.kind == "decode":
        v, unit = wl.bytes_per_step / seconds / 1e9, "GB/s"
    else:
        v, unit = wl.flops_per_step / seconds / 1e12, "TFLOP/s"
    return {"value": round(v * world, 3), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(seconds * 1e3, 3)}


# ============================================================================ CPU oracle timing
#
# The oracle (the fp64 CPU definition the tests check the kernels against) timed on the host
# cores over the same inputs. The pool of worker processes is started with "spawn" before the
# first GPU call; each workload's host copies go to .npy files that the workers map read-only.

_MAPPED = {}


def _load(path):
    if path not in _MAPPED:
        _MAPPED.clear()
        with open(os.path.join(path, "meta.json")) as f:
            meta = json.load(f)
        arr = {k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r") for k in meta["arrays"]}
        arr["_meta"] = meta
        _MAPPED[path] = arr
    return _MAPPED[path]


def _oracle_unit(a, kind, unit, scale):
    import oracle
    if kind in ("decode", "fp8"):
        b, j = unit
        g = a["q"].shape[1] // a["k"].shape[2]
        s = int(a["lens"][b])
        if kind == "decode":
            k, v = a["k"][b, :s, j], a["v"][b, :s, j]
        else:
            k = oracle.dequantize(a["k"][b, :s, j], a["k_scale"][b, :s, j])
            v = oracle.dequantize(a["v"][b, :s, j], a["v_scale"][b, :s, j])
        oracle.attend(a["q"][b, j * g:(j + 1) * g], k, v, scale)
    elif kind == "step":
        b = unit[0]
        q_rot, kc, vc, lens = oracle.kv_append_rope(a["q"][b:b + 1], a["k_new"][b:b + 1], a["v_new"][b:b + 1],
                                                    a["pos"][b:b + 1], a["freqs_cis"], a["k_cache"][b:b + 1],
                                                    a["v_cache"][b:b + 1])
        oracle.decode_gqa(q_rot, kc, vc, lens, scale)
    elif kind in ("mla", "mla_step"):
        b = unit[0]
        s = int(a["lens"][b])
        if kind == "mla":
            q_lat = a["q_lat"][b]
        else:
            q_lat = oracle.absorb_query(a["q_nope"][b:b + 1], a["w_uk"])[0]
        q = np.concatenate([q_lat, a["q_rope"][b]], axis=1)
        k = np.concatenate([a["c"][b, :s], a["kr"][b, :s]], axis=1)
        o_lat = oracle.attend(q, k, a["c"][b, :s], scale)
        if kind == "mla_step":
            oracle.apply_uv(o_lat[None], a["w_uv"])
    elif kind in ("chunk", "mla_chunk"):
        b = unit[0]
        lo, hi = int(a["cu_q"][b]), int(a["cu_q"][b + 1])
        cu, start = np.array([0, hi - lo]), a["start_pos"][b:b + 1]
        if kind == "chunk":
            oracle.prefill_gqa_chunked(a["q"][lo:hi], a["k"][b:b + 1], a["v"][b:b + 1], cu, start, scale)
        else:
            oracle.mla_prefill_absorbed(a["q_lat"][lo:hi], a["q_rope"][lo:hi], a["c"][b:b + 1], a["kr"][b:b + 1],
                                        cu, start, scale)
    elif kind == "prefill":
        b, h = unit
        lo, hi = int(a["cu"][b]), int(a["cu"][b + 1])
        j = h // (a["q"].shape[1] // a["k"].shape[1])
        oracle.attend(a["q"][lo:hi, h], a["k"][lo:hi, j], a["v"][lo:hi, j], scale,
                      oracle.attention.causal_allowed(hi - lo, hi - lo))
    else:
        raise ValueError(kind)


def _oracle_task(job):
    path, units = job
    a = _load(path)
    meta = a["_meta"]
    for u in units:
        _oracle_unit(a, meta["kind"], tuple(u), meta["scale"])
    return len(units)


class OraclePool:
    """Worker processes (spawned, one per host core) that run oracle units."""

    def __init__(self):
        import multiprocessing as mp
        self.cores = len(os.sched_getaffinity(0))
        # one BLAS thread per worker: the workers already use every core
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        os.environ.update({k: "1" for k in saved})
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def rate(self, wl, budget_s, steps=None, warmup=0):
        """Oracle throughput over the workload's units (see each workload's oracle_payload):
        (value in the workload's unit, workers used, sample description, seconds per step).
        Without `steps`: as many whole passes over the units as fit in budget_s. With `steps`
        (the reference arm): each step a bounded sample of the units, sized so that warmup +
        steps fit in budget_s."""
        import shutil
        import tempfile
        arrays, units, n_seq = wl.oracle_payload()
        tmp = tempfile.mkdtemp(prefix="oracle_")
        try:
            for k, v in arrays.items():
                np.save(os.path.join(tmp, k + ".npy"), np.ascontiguousarray(v))
            with open(os.path.join(tmp, "meta.json"), "w") as f:
                json.dump({"kind": wl.oracle_kind, "scale": float(wl.w.scale), "arrays": sorted(arrays)}, f)
            order = [units[i] for i in np.random.default_rng(0).permutation(len(units))]
            # size the sample from the time of a few units in this process
            t0 = time.perf_counter()
            n_probe = min(len(order), 2)
            _oracle_task((tmp, order[:n_probe]))
            per_unit = (time.perf_counter() - t0) / n_probe
            self.pool.map(_oracle_task, [(tmp, [order[0]])] * self.cores)     # workers map the files
            scale_work = 1e9 if wl.kind == "decode" else 1e12
            if steps is None:
                passes = max(1, int(budget_s / max(per_unit * len(units) / self.cores, 1e-9)))
                sample = order * passes
                workers = min(self.cores, len(sample))
                t0 = time.perf_counter()
                self.pool.map(_oracle_task, [(tmp, sample[i::workers]) for i in range(workers)])
                wall = time.perf_counter() - t0
                work = passes * sum(wl.unit_work(u) for u in units)
                covered = "all" if n_seq == wl.w.batch else f"the first {n_seq} of the {wl.w.batch}"
                what = (f"{passes} pass(es) over {len(units)} units ({covered} sequences"
                        f"{', one unit per query head' if wl.oracle_kind == 'prefill' else ''}), fp64 oracle, "
                        f"{workers} worker processes")
                return work / wall / scale_work, workers, what, None
            per_step_budget = budget_s / max(1, steps + warmup)
            n_units = int(min(len(order), max(1, per_step_budget / per_unit * self.cores)))
            workers = min(self.cores, n_units)
            cursor = 0

            def one_step():
                nonlocal cursor
                sample = [order[(cursor + i) % len(order)] for i in range(n_units)]
                cursor += n_units
                self.pool.map(_oracle_task, [(tmp, sample[i::workers]) for i in range(workers)])
                return sum(wl.unit_work(u) for u in sample)

            for _ in range(warmup):
                one_step()
            t0 = time.perf_counter()
            work = sum(one_step() for _ in range(steps))
            wall = time.perf_counter() - t0
            what = (f"each step {n_units} of {len(units)} units of the workload's first {n_seq} sequence(s), "
                    f"fp64 oracle, {workers} worker processes")
            return work / wall / scale_work, workers, what, wall / steps
        finally:
            shutil.rmtree(tmp, ignore_errors=True)


# ============================================================================ main

# The line's `config` names the workload alone, identical for both arms; how this arm ran it
# (split count, the input sets that keep the timed calls out of L2, the replicas) is `plan`.
PLAN_KEYS = ("n_split", "l2", "parallelism")
L2_POLICY = "inputs larger than L2: distinct input sets, >= 4x L2 in total, cycled between timed calls"


def split_plan(cfg):
    cfg = dict(cfg)
    plan = {k: cfg.pop(k) for k in PLAN_KEYS if k in cfg}
    cfg["l2"] = L2_POLICY
    return cfg, plan


# The fields of one secondary line, in the order compact() lists them.
ALSO_FIELDS = ["workload", "value", "unit", "ms_per_step", "roofline_frac", "traffic_MB", "cpu", "sm_mhz",
               "reasons"]
# throttle reasons, abbreviated in the secondary lines
_REASON_ABBREV = {"sw_power_cap": "pc", "hw_slowdown": "hw", "hw_thermal_slowdown": "hwt", "sw_thermal_slowdown": "swt"}


def compact(name, s, cpu):
    """One secondary line as a list in ALSO_FIELDS order, kept short so that the whole list
    survives in the last 1500 characters of a log (the line ends with it)."""
    c = s["clocks"]
    traffic = s["roofline"]["traffic"]
    return [name, s["value"], s["unit"], s["ms_per_step"], s["roofline"]["frac"],
            round(traffic / 1e6, 2) if traffic is not None else None, cpu,
            round(c["sm_mhz"]) if c.get("sm_mhz") is not None else None,
            [_REASON_ABBREV.get(r, r) for r in (c.get("reasons") or [])]]


def main():
    ap = argparse.ArgumentParser(description="KV-cache attention benchmark (one JSON line)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-also", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baselines")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle budget for the headline line")
    ap.add_argument("--also-cpu-seconds", type=float, default=3.0, help="oracle budget per secondary line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    world, rank, local = dist_env()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 with torchrun")
    steps = args.steps
    peaks, peak_src = load_peaks()
    cls, w = WORKLOADS[args.workload]()

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle arm runs on the host only; inputs are generated on the CPU
        wl = _cpu_workload(cls, w)
        pool = OraclePool()
        try:
            value, cores, sample, per_step = pool.rate(wl, budget_s=120.0, steps=steps, warmup=args.warmup)
        finally:
            pool.close()
        unit = "GB/s" if wl.kind == "decode" else "TFLOP/s"
        cfg, _ = split_plan(wl.describe())
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world,
                "steps": steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg, "plan": {"l2": "host memory (the CPU oracle)", "parallelism": f"{cores} host processes"},
                "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    # the oracle's worker processes start before the first GPU call
    pool = OraclePool() if (rank == 0 and world == 1 and not args.no_cpu) else None
    try:
        return run_gpu(args, world, rank, local, steps, peaks, peak_src, cls, w, pool)
    finally:
        if pool is not None:
            pool.close()


def run_gpu(args, world, rank, local, steps, peaks, peak_src, cls, w, pool):
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        barrier = lambda: dist.barrier(device_ids=[local])  # noqa: E731
    else:
        barrier = lambda: None  # noqa: E731
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import mla_kv_cache_flash_b300 as mk
    mk.lib()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    stream = torch.cuda.Stream(device)

    with torch.cuda.stream(stream):
        wl = cls(w, device, rank, l2)
        t = time_workload(wl, steps, args.warmup, stream, barrier, device.index)
        e2e = time_e2e(wl, device, barrier) if hasattr(wl, "e2e_step") else None
    t["seconds_per_call"], e2e_s = max_over_ranks([t["seconds_per_call"], e2e["seconds"] if e2e else 0.0], device)
    head = summarize(wl, t, peaks, peak_src, world)
    if e2e:
        head["e2e"] = e2e_line(wl, e2e_s, e2e["h2d"], e2e["d2h"], world)
    cpu = None
    if pool is not None:
        value, cores, sample, _ = pool.rate(wl, args.cpu_seconds)
        cpu = {"value": round(value, 4), "unit": head["unit"], "cores": cores, "kind": "oracle", "sample": sample}
    del wl
    torch.cuda.empty_cache()

    also, launches = [], head["gpu_launches"]
    if not args.no_also and world == 1:
        for name in ALSO:
            if name == args.workload:
                continue
            c2, w2 = WORKLOADS[name]()
            try:
                with torch.cuda.stream(stream):
                    wl2 = c2(w2, device, rank, l2)
                    t2 = time_workload(wl2, steps, 3, stream, barrier, device.index)
                s2 = summarize(wl2, t2, peaks, peak_src, 1)
                launches += s2["gpu_launches"]
                cpu2 = None
                if pool is not None:
                    cpu2 = round(pool.rate(wl2, args.also_cpu_seconds)[0], 4)
                also.append(compact(name, s2, cpu2))
                del wl2
            except Exception as e:   # a secondary line must not cost the headline line
                also.append([name, "error", f"{type(e).__name__}: {e}"[:200]])
            torch.cuda.empty_cache()

    if rank == 0:
        cfg, plan = split_plan(head["config"])
        plan["parallelism"] = f"replicas x{world} (independent sequences per GPU)"
        line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": steps,
                "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": cfg, "plan": plan,
                "timing": head["timing"], "tokens_per_s": head.get("tokens_per_s"),
                "pct_of_8tbs": head.get("pct_of_8tbs"), "roofline": head["roofline"], "cpu_baseline": cpu,
                "e2e": head.get("e2e"), "gpu_launches": launches, "clocks": head["clocks"],
                "also_note": "also: one list per secondary line, fields as also_fields; traffic_MB = DRAM bytes "
                             "per launch from profiles/ (null if none), cpu = the fp64 oracle on this host in the "
                             "line's unit, sm_mhz and throttle reasons (pc = sw_power_cap) while timed; each line "
                             "is timed like the headline",
                "also_fields": ALSO_FIELDS,
                "also": also}
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _cpu_workload(cls, w):
    """Inputs for the oracle arm, generated on the host with the same recipe."""
    class HostOnly(cls):
        def __init__(self, w):
            self.w, self.name = w, w.name
            if issubclass(cls, DecodeMla):
                s = W.mla_inputs(w, "cpu")
                s["q_lat"] = torch.einsum("hnr,bhn->bhr", s["w_uk"].float(), s["q_nope"].float()).to(torch.bfloat16).contiguous()
            elif cls is Prefill:
                s = W.prefill_inputs(w, "cpu")
                self.lens = s["lengths"]
            else:
                s = W.decode_inputs(w, "cpu")
            self.sets = [s]
            if cls is not Prefill:
                self.lens = s["seq_lens"].numpy()
            self.n_split = None
            self.l2_note = "host memory"
            self.flops_per_step = sum(4 * w.head_dim * w.n_q_heads * int(x) * (int(x) + 1) // 2
                                      for x in self.lens) if cls is Prefill else None
    if cls not in (DecodeGqa, DecodeMla, Prefill):
        raise SystemExit("the oracle arm covers the single-call decode and prefill workloads")
    return HostOnly(w)


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Benchmark of the KV-cache attention hot path on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Headline workload (default): MiniMind-shaped GQA decode — B=32, Hq=8, Hkv=4, D=96, bf16
cache, one new query token per sequence, cache lengths uniform in [512, 2048] from the
seed. A step is one ``attn_decode_gqa`` call (one balanced split-KV decode launch that also
merges the segments it splits) over the whole batch. ``value`` = algorithmic KV bytes read per step (each cached K/V
element of the live lengths once) ÷ the device time per step, in GB/s, with the inputs
resident in HBM; the timed steps cycle through enough distinct cache sets that they
cannot be served from L2 (≥ 4 × the L2 size in total).

The line also carries: ``roofline`` (the decode call's achieved GB/s against the measured
HBM copy bandwidth), ``e2e`` (same metric through the Python API with pinned host inputs
copied in and the output copied back inside the timed region), ``cpu_baseline`` (the fp64
CPU oracle on the host cores, bounded sample), ``clocks`` (NVML samples taken during the
timed region), ``gpu_launches`` and ``also`` (the other workloads: Llama-3-8B-shaped decode
with Hkv 32/8/1, MLA absorbed decode, causal prefill, each with its own roofline).

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

    def oracle_units(self):
        return [(b, j) for b in range(self.w.batch) for j in range(self.w.n_kv_heads)]

    def unit_bytes(self, unit):
        b, _ = unit
        elt = 2 if self.w.dtype == "bf16" else 4
        return int(self.lens[b]) * 2 * self.w.head_dim * elt

    def host_arrays(self):
        s = self.sets[0]
        return {"q": s["q"].float().cpu().numpy(), "k": s["k_cache"].float().cpu().numpy(),
                "v": s["v_cache"].float().cpu().numpy(), "lens": self.lens, "scale": self.w.scale}

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

    def describe(self):
        return dict(super().describe(), workload=self.name,
                    launches="append the new token with RoPE at position length-1, then decode")


class DecodeGqaFp8(DecodeGqa):
    """The MiniMind decode batch over an E4M3 cache with per-row fp32 K and V scales.
    Algorithmic bytes: each live code once plus its row's scale."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_gqa_fma.cu"
    call = "attn_decode_gqa_fp8 call: "
    launch_note = " (CUDA-core decode, then the merge launch when the plan splits)"

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
        self.launches_per_step = 1 + (self.n_split > 1)
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

    def describe(self):
        return dict(super().describe(), cache_dtype="fp8_e4m3 + fp32 scale per row")


class DecodeChunked(DecodeGqa):
    """Chunks of 4 new tokens per sequence over the MiniMind caches (a speculative-decoding
    style step): each sequence's last 4 cached rows are its chunk, so row i sees
    length − 4 + i + 1 rows. Algorithmic bytes: each sequence's visible K/V once (as for the
    decode of the full length); the kernel reads them once per new token."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/decode_gqa_fma.cu"
    call = "attn_prefill_gqa_chunked call: "
    launch_note = " (CUDA-core decode, then the merge launch when the plan splits)"
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
                                                             self.max_s, 0))
        self.ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 2 if nb else 1

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

    def oracle_units(self):
        return [(b, 0) for b in range(self.w.batch)]

    def unit_bytes(self, unit):
        return int(self.lens[unit[0]]) * (self.w.kv_lora_rank + self.w.rope_dim) * 2

    def host_arrays(self):
        s = self.sets[0]
        return {"q_lat": s["q_lat"].float().cpu().numpy(), "q_rope": s["q_rope"].float().cpu().numpy(),
                "c": s["c_cache"].float().cpu().numpy(), "kr": s["kr_cache"].float().cpu().numpy(),
                "lens": self.lens, "scale": self.w.scale}

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

    def describe(self):
        return dict(super().describe(), workload=self.name, nope_dim=self.w.nope_dim, v_head_dim=self.w.v_head_dim,
                    launches="absorb W_UK, latent decode, apply W_UV")


class MlaChunked(DecodeMla):
    """MLA chunked prefill, 4 new tokens per sequence over the MiniMind MLA latent caches
    (each sequence's last 4 rows are its chunk). Algorithmic bytes: each visible latent row
    once, as for the decode of the full length."""
    kernel_src = "mla_kv_cache_flash_b300/csrc/prefill_chunked_mla.cu"
    call = "attn_prefill_mla_chunked call: "
    launch_note = " (CUDA-core decode form, then the merge launch when the plan splits)"
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
        self.ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=device)
        self.launches_per_step = 2 if nb else 1

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

    def describe(self):
        return dict(super().describe(), workload=self.name, new_tokens_per_sequence=self.n_new)


class Prefill:
    kind = "prefill"
    kernel_src = "mla_kv_cache_flash_b300/csrc/prefill.cu"

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

    def describe(self):
        w = self.w
        return {"workload": w.name, "B": w.batch, "Hq": w.n_q_heads, "Hkv": w.n_kv_heads, "D": w.head_dim,
                "lengths": [int(x) for x in self.lens], "causal_flops": self.flops_per_step, "l2": self.l2_note}


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
}
DEFAULT_STEPS = {"minimind_gqa": 60000, "minimind_gqa_step": 60000, "minimind_gqa_fp8": 60000,
                 "minimind_gqa_chunk4": 20000, "llama_hkv32": 400, "llama_hkv8": 2000, "llama_hkv1": 10000,
                 "mla": 40000, "mla_step": 40000, "mla_chunk4": 8000, "prefill": 2000, "prefill_ragged": 1500}


# ============================================================================ timing

def time_device(run, steps, warmup, graph_len, stream):
    """Device time of `steps` calls of run(i): CUDA graphs of `graph_len` calls replayed back to
    back (so host launch cost is off the clock), CUDA events on the launching stream."""
    for i in range(warmup):
        run(i)
    torch.cuda.synchronize()
    graph_len = max(1, min(graph_len, steps))
    reps, rem = divmod(steps, graph_len)
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        for i in range(graph_len):
            run(i)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                run(i)
    g_full.replay()  # warm the graph itself
    torch.cuda.synchronize()
    return reps, g_full, g_rem


def timed_region(reps, g_full, g_rem, stream, barrier):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / 1e3


def run_workload(cls, w, device, rank, steps, warmup, l2, stream, barrier, want_e2e):
    wl = cls(w, device, rank, l2)
    graph_len = len(getattr(wl, "sets", [0])) * max(1, 256 // max(1, len(getattr(wl, "sets", [0]))))
    if wl.kind == "prefill":
        graph_len = min(graph_len, 8)
    reps, g_full, g_rem = time_device(wl.step, steps, warmup, graph_len, stream)
    with ClockSampler(device.index) as clk:
        t = timed_region(reps, g_full, g_rem, stream, barrier)
    res = {"wl": wl, "seconds": t, "clocks": clk.summary()}
    del g_full, g_rem
    if want_e2e and hasattr(wl, "e2e_step"):
        host = wl.host_inputs()
        dev_bufs = {k: torch.empty_like(v, device=device) for k, v in host.items()}
        out_host = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
        n_e2e = 20
        for _ in range(3):
            wl.e2e_step(host, dev_bufs, out_host)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(n_e2e):
            wl.e2e_step(host, dev_bufs, out_host)
            torch.cuda.current_stream().synchronize()   # the result is read on the host each step
        end.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier()
        res["e2e_seconds"] = wall / n_e2e
        res["e2e_h2d"] = sum(v.nbytes for v in host.values())
        res["e2e_d2h"] = out_host.nbytes
    return res


def summarize(res, steps, peaks, peak_src, world):
    wl = res["wl"]
    per_step = res["seconds"] / steps
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
                "algorithmic_flops_per_launch": wl.flops_per_step, "kernel": "attn_prefill_gqa_causal"}
        extra = {"tokens_per_s": round(float(np.sum(wl.lens)) * world / per_step, 1)}
    out = {"value": round(value, 2), "unit": unit, "ms_per_step": round(per_step * 1e3, 5), "roofline": roof,
           "gpu_launches": steps * wl.launches_per_step, "config": wl.describe(), "clocks": res["clocks"]}
    out.update(extra)
    if res.get("e2e_seconds"):
        e = res["e2e_seconds"]
        ev = (wl.bytes_per_step / e / 1e9) if wl.kind == "decode" else (wl.flops_per_step / e / 1e12)
        out["e2e"] = {"value": round(ev * world, 3), "unit": unit, "h2d_bytes_per_step": res["e2e_h2d"],
                      "d2h_bytes_per_step": res["e2e_d2h"], "ms_per_step": round(e * 1e3, 3)}
    return out


# ============================================================================ CPU oracle timing

def _oracle_worker_init(path):
    global _ARR
    _ARR = dict(np.load(path, allow_pickle=False))


def _oracle_decode_units(units):
    import oracle
    a = _ARR
    done = 0
    if "q_lat" in a:
        for b, _ in units:
            s = int(a["lens"][b])
            q = np.concatenate([a["q_lat"][b], a["q_rope"][b]], axis=1)
            k = np.concatenate([a["c"][b, :s], a["kr"][b, :s]], axis=1)
            oracle.attend(q, k, a["c"][b, :s], float(a["scale"]))
            done += 1
        return done
    g = a["q"].shape[1] // a["k"].shape[2]
    for b, j in units:
        s = int(a["lens"][b])
        oracle.attend(a["q"][b, j * g:(j + 1) * g], a["k"][b, :s, j], a["v"][b, :s, j], float(a["scale"]))
        done += 1
    return done


def cpu_oracle_rate(wl, budget_s, steps=None, warmup=0):
    """Time the fp64 oracle on the host cores over a bounded sample of the workload's units
    (one unit = one sequence and KV head). Returns (value in GB/s of KV read, cores used,
    sample description, seconds per step or None)."""
    import multiprocessing as mp
    import tempfile
    global _ARR
    cores = len(os.sched_getaffinity(0))
    arrays = {k: np.asarray(v) for k, v in wl.host_arrays().items()}
    units = wl.oracle_units()
    order = [units[i] for i in np.random.default_rng(0).permutation(len(units))]
    _ARR = arrays
    t0 = time.perf_counter()
    _oracle_decode_units(order[:min(8, len(order))])
    per_unit = (time.perf_counter() - t0) / min(8, len(order))
    tmp = tempfile.NamedTemporaryFile(suffix=".npz", delete=False)
    tmp.close()
    np.savez(tmp.name, **arrays)
    ctx = mp.get_context("spawn")
    try:
        with ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(tmp.name,)) as pool:
            pool.map(_oracle_decode_units, [[order[0]]] * cores)   # workers up and loaded
            if steps is None:
                passes = max(1, int(budget_s / max(per_unit * len(units) / cores, 1e-9)))
                sample = order * passes
                t0 = time.perf_counter()
                pool.map(_oracle_decode_units, [sample[i::cores] for i in range(cores)])
                wall = time.perf_counter() - t0
                nbytes = passes * sum(wl.unit_bytes(u) for u in units)
                return (nbytes / wall / 1e9, cores,
                        f"{passes} full pass(es) over all {len(units)} (sequence, kv-head) units, fp64 oracle.attend, "
                        f"{cores} worker processes", None)
            per_step_budget = budget_s / max(1, steps + warmup)
            n_units = int(min(len(order), max(1, per_step_budget / per_unit * cores)))
            workers = min(cores, n_units)
            cursor = 0

            def one_step():
                nonlocal cursor
                sample = [order[(cursor + i) % len(order)] for i in range(n_units)]
                cursor += n_units
                if workers == 1:
                    _oracle_decode_units(sample)
                else:
                    pool.map(_oracle_decode_units, [sample[i::workers] for i in range(workers)])
                return sum(wl.unit_bytes(u) for u in sample)

            for _ in range(warmup):
                one_step()
            t0 = time.perf_counter()
            nbytes = sum(one_step() for _ in range(steps))
            wall = time.perf_counter() - t0
    finally:
        os.unlink(tmp.name)
    what = "all" if n_units == len(units) else f"{n_units} of the"
    return (nbytes / wall / 1e9, workers,
            f"each step {what} {len(units)} (sequence, kv-head) units of the workload, fp64 oracle.attend, "
            f"{workers} worker processes", wall / steps)


# ============================================================================ main

def main():
    ap = argparse.ArgumentParser(description="KV-cache attention benchmark (one JSON line)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="minimind_gqa")
    ap.add_argument("--no-also", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 with torchrun")
    steps = args.steps or DEFAULT_STEPS[args.workload]
    peaks, peak_src = load_peaks()
    cls, w = WORKLOADS[args.workload]()

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle arm runs on the host only; inputs are generated on the CPU
        wl = _cpu_workload(cls, w)
        value, cores, sample, per_step = cpu_oracle_rate(wl, budget_s=120.0, steps=steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
                "steps": steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": wl.describe(),
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

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
        res = run_workload(cls, w, device, rank, steps, args.warmup, l2, stream, barrier, want_e2e=True)
    res["seconds"], res["e2e_seconds"] = max_over_ranks([res["seconds"], res.get("e2e_seconds", 0.0)], device)
    head = summarize(res, steps, peaks, peak_src, world)

    also = []
    if not args.no_also and world == 1:
        for name in ("minimind_gqa_step", "minimind_gqa_fp8", "minimind_gqa_chunk4", "llama_hkv32", "llama_hkv8",
                     "llama_hkv1", "mla", "mla_step", "mla_chunk4", "prefill", "prefill_ragged"):
            if name == args.workload:
                continue
            c2, w2 = WORKLOADS[name]()
            try:
                with torch.cuda.stream(stream):
                    r2 = run_workload(c2, w2, device, rank, max(3, DEFAULT_STEPS[name] // 4), 3, l2, stream,
                                      barrier, want_e2e=False)
                s2 = summarize(r2, max(3, DEFAULT_STEPS[name] // 4), peaks, peak_src, 1)
                also.append({"workload": w2.name, "value": s2["value"], "unit": s2["unit"],
                             "ms_per_step": s2["ms_per_step"], "roofline": s2["roofline"],
                             "tokens_per_s": s2.get("tokens_per_s"), "clocks": s2["clocks"],
                             "config": s2["config"]})
                del r2
            except Exception as e:   # a secondary line must not cost the headline line
                also.append({"workload": w2.name, "error": f"{type(e).__name__}: {e}"})
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and not isinstance(
            res["wl"], (DecodeMlaStep, DecodeGqaStep, DecodeGqaFp8, DecodeChunked, MlaChunked)):
        value, cores, sample, _ = cpu_oracle_rate(res["wl"], args.cpu_seconds)
        cpu = {"value": round(value, 4), "unit": head["unit"], "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": steps,
                "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": dict(head["config"], parallelism=f"replicas x{world} (independent sequences per GPU)"),
                "tokens_per_s": head.get("tokens_per_s"), "pct_of_8tbs": head.get("pct_of_8tbs"),
                "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head.get("e2e"),
                "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "also": also}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _cpu_workload(cls, w):
    """Inputs for the oracle arm, generated on the host with the same recipe."""
    class HostOnly(cls):
        def __init__(self, w):
            self.w, self.name = w, w.name
            if cls is DecodeMla:
                s = W.mla_inputs(w, "cpu")
                s["q_lat"] = torch.einsum("hnr,bhn->bhr", s["w_uk"].float(), s["q_nope"].float()).to(torch.bfloat16).contiguous()
            else:
                s = W.decode_inputs(w, "cpu")
            self.sets = [s]
            self.lens = s["seq_lens"].numpy()
            self.n_split = None
            self.l2_note = "host memory"
    if cls in (Prefill, DecodeMlaStep, DecodeGqaStep, DecodeGqaFp8, DecodeChunked, MlaChunked):
        raise SystemExit("the oracle arm covers the single-call decode workloads")
    return HostOnly(w)


if __name__ == "__main__":
    sys.exit(main())

"""bench.py's workload classes build on the CPU with the byte counts their roofline lines
state (the GPU timing itself runs only on a GPU)."""

import pytest

import bench


def _make(name):
    cls, w = bench.WORKLOADS[name]()
    return cls(w, "cpu", 0, 1), w


def test_step_with_append_counts_the_cache_and_the_new_token():
    wl, w = _make("minimind_gqa_step")
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    cache = int(wl.lens.sum()) * 2 * Hkv * D * 2
    assert wl.bytes_per_step == cache + B * (2 * Hq * D * 2 + 4 * Hkv * D * 2 + D * 4 + 8)
    assert wl.launches_per_step == 2
    s = wl.sets[0]
    assert (s["pos"] == s["seq_lens"] - 1).all()


def test_fp8_counts_codes_and_row_scales():
    wl, w = _make("minimind_gqa_fp8")
    assert wl.bytes_per_step == int(wl.lens.sum()) * 2 * w.n_kv_heads * (w.head_dim + 4)
    assert wl.sets[0]["k_cache"].dtype.itemsize == 1
    assert wl.describe()["workload"].endswith("_fp8")


def test_chunked_counts_each_visible_row_once():
    wl, w = _make("minimind_gqa_chunk4")
    assert wl.bytes_per_step == int(wl.lens.sum()) * 2 * w.n_kv_heads * w.head_dim * 2
    s = wl.sets[0]
    assert s["q_chunk"].shape == (w.batch * 4, w.n_q_heads, w.head_dim)
    assert s["cu_q"].tolist() == list(range(0, w.batch * 4 + 1, 4))
    assert ((s["start_pos"] + 4) == s["seq_lens"]).all()


def test_mla_full_step_counts_cache_and_weights():
    wl, w = _make("mla_step")
    cache = int(wl.lens.sum()) * (w.kv_lora_rank + w.rope_dim) * 2
    weights = 2 * w.n_q_heads * w.nope_dim * w.kv_lora_rank * 2
    assert wl.bytes_per_step == cache + weights
    assert wl.launches_per_step == 3


def test_mla_chunked_counts_each_visible_latent_row_once():
    wl, w = _make("mla_chunk4")
    assert wl.bytes_per_step == int(wl.lens.sum()) * (w.kv_lora_rank + w.rope_dim) * 2
    s = wl.sets[0]
    assert s["q_lat_chunk"].shape == (w.batch * 4, w.n_q_heads, w.kv_lora_rank)
    assert ((s["start_pos"] + 4) == s["seq_lens"]).all()


@pytest.mark.parametrize("name", ["minimind_gqa_step", "minimind_gqa_fp8", "minimind_gqa_chunk4", "mla_step",
                                  "mla_chunk4"])
def test_multi_launch_lines_have_no_oracle_arm(name):
    cls, w = bench.WORKLOADS[name]()
    with pytest.raises(SystemExit):
        bench._cpu_workload(cls, w)


@pytest.mark.parametrize("name", ["minimind_gqa", "minimind_gqa_step", "minimind_gqa_fp8", "minimind_gqa_chunk4",
                                  "mla", "mla_step", "mla_chunk4", "prefill"])
def test_oracle_leg_runs_every_kind_and_counts_the_line_work(name, tmp_path):
    # the CPU baseline beside each line: the oracle runs one unit of the workload from the
    # files the worker processes map, and the units' work adds up to the line's own count
    import json
    import numpy as np
    wl, w = _make(name)
    arrays, units, n_seq = wl.oracle_payload()
    for k, v in arrays.items():
        np.save(tmp_path / (k + ".npy"), np.ascontiguousarray(v))
    (tmp_path / "meta.json").write_text(json.dumps({"kind": wl.oracle_kind, "scale": w.scale,
                                                    "arrays": sorted(arrays)}))
    assert bench._oracle_task((str(tmp_path), [units[-1]])) == 1
    work = sum(wl.unit_work(u) for u in units)
    if wl.kind == "prefill":
        s0 = int(wl.lens[0])
        assert work == 4 * w.head_dim * w.n_q_heads * s0 * (s0 + 1) // 2
    else:
        assert n_seq == w.batch
        assert work == wl.bytes_per_step


def test_long_chunk_lines_count_each_visible_pair():
    # new row i of a 512-token chunk after 3584 cached rows sees 3585 + i keys: Σ = 512·3584 +
    # 512·513/2 pairs a sequence, 4·D flops a pair and query head (GQA), 2·(r + dr) + 2·r (MLA)
    pairs = 512 * 3584 + 512 * 513 // 2
    wl, w = _make("prefill_chunk512")
    assert wl.start == [3584] * w.batch
    assert wl.flops_per_step == w.batch * 4 * w.head_dim * w.n_q_heads * pairs
    assert wl.sets[0]["q_chunk"].shape == (w.batch * 512, w.n_q_heads, w.head_dim)
    assert wl.sets[0]["cu_q"].tolist() == list(range(0, w.batch * 512 + 1, 512))
    wm, m = _make("mla_prefill_chunk512")
    assert wm.flops_per_step == m.batch * (2 * (m.kv_lora_rank + m.rope_dim) + 2 * m.kv_lora_rank) * m.n_q_heads * pairs
    assert wm.sets[0]["q_rope_chunk"].shape == (m.batch * 512, m.n_q_heads, m.rope_dim)


@pytest.mark.parametrize("name", ["prefill_chunk512", "mla_prefill_chunk512"])
def test_long_chunk_oracle_leg(name, tmp_path):
    # the CPU baseline's unit (the first sequence's whole chunk) runs from the mapped files and
    # counts that sequence's flops
    import json
    import numpy as np
    wl, w = _make(name)
    arrays, units, n_seq = wl.oracle_payload()
    assert units == [(0,)] and n_seq == 1
    for k, v in arrays.items():
        np.save(tmp_path / (k + ".npy"), np.ascontiguousarray(v))
    (tmp_path / "meta.json").write_text(json.dumps({"kind": wl.oracle_kind, "scale": w.scale,
                                                    "arrays": sorted(arrays)}))
    assert bench._oracle_task((str(tmp_path), units)) == 1
    assert wl.unit_work((0,)) * w.batch == wl.flops_per_step

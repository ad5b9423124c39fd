"""CPU checks of the measurement code in bench.py: the DRAM-traffic lookup
honours the captured source's hash, and the decode step's algorithmic bytes
and launch counts follow the workloads' shapes."""
import json
import os

import pytest

import bench
from transformer_attention_gb300 import workloads as WL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _traffic_table():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_for_returns_the_committed_bytes_while_the_source_matches(monkeypatch):
    table = _traffic_table()
    assert table
    for kernel, rows in table.items():
        for workload, e in rows.items():
            monkeypatch.setattr(bench, "source_hash", lambda path, h=e["source_sha256_16"]: h)
            assert bench.traffic_for(kernel, workload) == e["dram_bytes_per_launch"]
    assert bench.traffic_for("attention", "no_such_workload") is None
    assert bench.traffic_for("no_such_kernel", "1b_global") is None


def test_traffic_for_follows_the_current_sources():
    for kernel, rows in _traffic_table().items():
        for workload, e in rows.items():
            src = os.path.join(ROOT, "transformer_attention_gb300", "csrc", e["source"])
            live = bench.source_hash(src) == e["source_sha256_16"]
            assert bench.traffic_for(kernel, workload) == (e["dram_bytes_per_launch"] if live
                                                           else None)


def test_traffic_for_is_null_once_the_source_changed(monkeypatch):
    monkeypatch.setattr(bench, "source_hash", lambda path: "0" * 16)
    assert bench.traffic_for("attention", "1b_global") is None


@pytest.mark.parametrize("name", ["27b_global_decode", "4b_local_decode"])
def test_decode_work_bytes(name):
    w = WL.WORKLOADS[name]
    work, launches = bench.decode_work(w, 152)
    KVD, HD = w.H_kv * w.d_h, w.H * w.d_h
    end = w.cache_len - w.T
    # every visible slot's K' and V once: a global layer sees the whole
    # cache, a local one its window plus the new tokens
    visible = end + w.T if w.window == 0 else min(w.window + w.T - 1, end + w.T)
    kv = w.B * visible * KVD * 2 * 2
    assert work["attention"] == kv + 2 * w.M * HD * 2 + w.B * (end + w.T) * 4
    # the projections read Wq, Wkv and Wo once
    weights = (HD * w.D + 2 * KVD * w.D + w.D * HD) * 2
    assert weights < work["linear"] < 1.01 * weights
    # Q|KV projection, QK prologue (which also writes the cache and scans a
    # local layer's cache span), O projection; attention: the split kernel
    # and its merge
    assert launches["linear"] == 3
    assert launches["attention"] == 2


def test_host_cpu_names_the_cores_and_the_model():
    h = bench.host_cpu()
    assert h["nproc"] == os.cpu_count() and h["nproc"] >= 1
    assert isinstance(h["cpu_model"], str) and h["cpu_model"]


def test_default_workload_is_the_largest_single_gpu_layer():
    # the 27B-shaped global layer: the most attention work of the layer workloads
    w = WL.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert (w.B, w.T, w.D, w.H, w.H_kv, w.d_h) == (1, 131072, 5376, 32, 16, 128)
    assert w.attn_type == "global" and w.rope_scale == 8.0


def test_algorithmic_flops_of_the_4b_local_and_27b_global_layers():
    """Attention over unmasked pairs plus the projections, as tabulated for
    the 4B-local (0.541 + 2.062 TF) and 27B-global (140.7 + 17.3 TF) layers."""
    w = WL.WORKLOADS["4b_local"]
    f = bench.algorithmic_flops(w, [w.T] * w.B, w.B * w.T)
    assert abs(f - (0.541e12 + 2.062e12)) / f < 2e-3
    w = WL.WORKLOADS["27b_global"]
    f = bench.algorithmic_flops(w, [w.T], w.T)
    assert abs(f - (140.7e12 + 17.3e12)) / f < 2e-3
    # a block adds its feed-forward GEMMs, a model its read-out
    b = WL.small(WL.WORKLOADS["4b_block"], B=1, T=100)
    base = WL.small(WL.WORKLOADS["4b_local"], B=1, T=100)
    extra = bench.algorithmic_flops(b, [100], 100) - bench.algorithmic_flops(base, [100], 100)
    assert extra == 2.0 * 100 * 2 * b.d_ff * b.D + 2.0 * 100 * b.D * b.d_ff

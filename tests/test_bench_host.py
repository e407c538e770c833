"""Host-side checks of bench.py (no GPU): the workload table resolves every
name to the shape the metric is quoted on, and the DRAM-traffic record is
reported only for the kernel sources its counters were taken on."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_workload_is_the_dense_bf16_config():
    w = bench.get_workload("dense")
    assert (w.dtype, w.B, w.H, w.N, w.d, w.causal) == ("bf16", 4, 16, 8448, 128, False)
    # 4 B H N^2 d
    assert w.flops() == pytest.approx(4 * 4 * 16 * 8448 ** 2 * 128)


def test_fp8_workload_and_causal_halving():
    w = bench.get_workload("fp8")
    assert (w.dtype, w.B, w.H, w.N, w.d, w.causal) == ("fp8", 4, 16, 8192, 128, False)
    c = bench.get_workload("causal:2048:16:128")
    assert (c.B, c.H, c.N, c.d, c.causal) == (8, 16, 2048, 128, True)
    assert c.flops() == pytest.approx(4 * 8 * 16 * 2048 ** 2 * 128 / 2)


@pytest.mark.parametrize("name", ["dense", "tiny", "fp8", "fp8_d64", "varlen", "gqa", "paged",
                                  "bwd", "bwd_causal", "causal:512:32:64"])
def test_every_workload_name_resolves(name):
    w = bench.get_workload(name)
    assert w.flops() > 0


def test_unknown_workload_is_an_error():
    with pytest.raises(SystemExit):
        bench.get_workload("no-such-workload")


def test_traffic_record_follows_the_kernel_sources(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec, "no traffic record"
    for name, entry in rec.items():
        assert entry["bytes"] > 0 and entry["kernel"] and entry["how"].startswith("ncu ")
    # counters taken on these sources: reported; on other sources: null
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: next(iter(rec.values()))["source_sha"])
    name, entry = next(iter(rec.items()))
    assert bench.traffic_record(name) == entry["bytes"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.traffic_record(name) is None
    assert bench.traffic_record("no-such-workload") is None


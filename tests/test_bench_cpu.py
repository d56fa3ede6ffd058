"""bench.py host logic that needs no GPU: the DRAM-traffic table, the
workload description and the argument defaults."""
import sys

import bench


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    t = bench.TRAFFIC[("qwen3", 1)]
    # as if the sources were the captured ones
    monkeypatch.setattr(bench, "kernel_src_hash", lambda: t["src"])
    # scaled to the timed steps' mean unique-expert count
    assert bench.traffic_per_launch("qwen3", 1, t["unique"]) == t["bytes"]
    assert bench.traffic_per_launch("qwen3", 1, 2 * t["unique"]) == 2 * t["bytes"]
    # no capture of this workload: no number
    assert bench.traffic_per_launch("qwen3", 3, 20.0) is None
    # sources changed since the capture: no number
    monkeypatch.setattr(bench, "kernel_src_hash", lambda: "0" * 16)
    assert bench.traffic_per_launch("qwen3", 1, 8.0) is None


def test_traffic_exceeds_the_algorithmic_bytes_only_slightly():
    import moe_synth as ms
    shape = ms.SHAPES["qwen3"]
    for (name, n), t in bench.TRAFFIC.items():
        algorithmic = t["unique"] * shape.plane_bytes + 2 * n * shape.D * 2
        assert algorithmic <= t["bytes"] <= 1.05 * algorithmic, (name, n)


def test_default_arguments_are_the_headline_workload(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert (a.gpus, a.shape, a.n_tokens, a.kind, a.impl, a.stack) == (1, "qwen3", 1, "independent", "ours", 0)
    assert a.warmup >= 3 and a.replicas * 339_738_624 > 8 * 129 * 2 ** 20  # replicas defeat the L2
    cfg = bench.workload_config(a)
    assert cfg["E"] == 128 and cfg["top_k"] == 8 and cfg["D"] == 2048 and cfg["Dff"] == 768
    assert "n_tokens=1" in cfg["workload"]

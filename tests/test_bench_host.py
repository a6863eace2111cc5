"""Host logic of bench.py that needs no GPU: the workloads' stack depth and routing, and the
committed DRAM traffic it reports next to a roofline."""
import json

import pytest

import bench
from quantized_routed_expert_softmax_gb300 import synth


def test_supplied_routing_workloads():
    for name in ("zipf", "zipf_nvfp4"):
        w = synth.WORKLOADS[name]
        assert bench.routed(w)
        # a step's routed experts must not sit in L2 at the next step: 4 layers x 8 experts
        # of 6.3 MB (Q8_0) is about 200 MB, above the 129 MB L2
        assert bench.default_layers(w) == bench.ZIPF_LAYERS >= 4
        assert "routing" in bench.workload_config(w, 1, bench.default_layers(w))
    for name in ("gemma", "nemotron", "minimax"):
        w = synth.WORKLOADS[name]
        assert not bench.routed(w)
        assert bench.default_layers(w) == w.layers
        assert "routing" not in bench.workload_config(w, 1, w.layers)


def _write_traffic(tmp_path, monkeypatch, entries):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(entries))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def test_measured_traffic_scales_a_stack_entry_with_the_depth(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha(("decode.cu",))
    _write_traffic(tmp_path, monkeypatch, {
        "gemma_T1": {"bytes": 3000, "layers": 30, "sources": ["decode.cu"], "source_sha1_12": sha},
        "gemma_T512": {"bytes": 777, "sources": ["decode.cu"], "source_sha1_12": sha},
    })
    # the kernel sources are read from the real package, not from tmp_path
    monkeypatch.setattr(bench, "kernel_source_sha", lambda files=(): sha)
    assert bench.measured_traffic("gemma", 1, 30) == 3000
    assert bench.measured_traffic("gemma", 1, 2) == 200
    assert bench.measured_traffic("gemma", 512, 30) == 777    # a per-layer launch: no scaling
    assert bench.measured_traffic("gemma", 4, 30) is None     # no capture for this workload
    assert bench.measured_traffic("zipf", 1, 4) is None


def test_measured_traffic_is_null_once_the_kernel_changed(tmp_path, monkeypatch):
    _write_traffic(tmp_path, monkeypatch, {
        "gemma_T1": {"bytes": 3000, "layers": 30, "sources": ["decode.cu"], "source_sha1_12": "000000000000"},
    })
    monkeypatch.setattr(bench, "kernel_source_sha", lambda files=(): "123456789abc")
    assert bench.measured_traffic("gemma", 1, 30) is None


def test_single_core_baseline_restores_the_thread_count():
    import oracle
    w = synth.WORKLOADS["tiny"]
    cache = {}
    step_s, n, threads, _ = bench.oracle_sample(w, 16, 1, max_units=3, time_budget_s=1.0, warmup_units=1,
                                                cache=cache)
    assert n >= 1 and step_s > 0 and 0 in cache      # the layer's experts were quantised once
    one = bench.single_core_baseline(w, 16, 1, threads, cache)
    assert one["cores"] == 1 and one["value"] > 0, one
    assert oracle.num_threads() == threads


def test_single_core_baseline_records_a_failure(monkeypatch):
    import oracle
    threads = oracle.num_threads()

    def boom(*a, **k):
        raise RuntimeError("planted")
    monkeypatch.setattr(bench, "oracle_sample", boom)
    got = bench.single_core_baseline(synth.WORKLOADS["tiny"], 16, 1, threads, {})
    assert got == {"error": "RuntimeError: planted"}
    assert oracle.num_threads() == threads

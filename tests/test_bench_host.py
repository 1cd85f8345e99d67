"""Host-side logic of bench.py on CPU: which bf16 peak a timed GEMM is divided by, the DRAM traffic
record keyed by the kernel sources' hash, and the algorithmic work per stage."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from mixture_experts_routing_moe_gb300 import workloads as W  # noqa: E402

PK = {"hbm_gbs": 6788.3, "bf16_tflops": 1884.4, "bf16_tflops_sustained": 1693.4}


def test_burst_peak_for_a_short_region_at_max_clock():
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(PK, clocks, 0.19) == (1884.4, "burst")


@pytest.mark.parametrize("clocks,region", [
    ({"sm_mhz": 1650.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, 0.19),  # clock dropped
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, 3.0),                 # long region
    (None, 0.19),                                                                   # no samples
])
def test_sustained_peak_otherwise(clocks, region):
    assert bench.tensor_peak(PK, clocks, region) == (1693.4, "sustained")


def test_traffic_record_is_used_only_for_the_recorded_sources(tmp_path, monkeypatch):
    rec = {"kernel_source_sha256": bench.kernel_source_sha256(),
           "launches": {"moe_experts_tc2<gate/up>": {"skewed": {"bytes_per_launch": 123456789}}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("moe_experts_tc2<gate/up>", "skewed") == 123456789
    assert bench.recorded_traffic("moe_experts_tc2<gate/up>", "prefill") is None
    assert bench.recorded_traffic("moe_experts_tc2<down>", "skewed") is None
    rec["kernel_source_sha256"] = "0" * 64            # the kernels changed since the capture
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("moe_experts_tc2<gate/up>", "skewed") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic("moe_experts_tc2<gate/up>", "skewed") is None


def test_committed_traffic_record_is_well_formed():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    assert len(rec["kernel_source_sha256"]) == 64
    for kernel, by_wl in rec["launches"].items():
        for wl, e in by_wl.items():
            assert e["bytes_per_launch"] > 0 and wl in W.WORKLOADS, (kernel, wl)


def test_stage_work_of_the_skewed_layer():
    wl = W.WORKLOADS["skewed"]
    w = bench.stage_work(wl, 176)
    R = wl.T * wl.top_k
    assert w["gate_up_gemm"]["flops"] == 4 * R * wl.H * wl.I
    assert w["down_gemm"]["flops"] == 2 * R * wl.I * wl.H
    # x_d rows + gate and up of the routed experts + a
    assert w["gate_up_gemm"]["bytes"] == 2 * (R * wl.H + 2 * 176 * wl.I * wl.H + R * wl.I)
    assert w["route"]["bytes"] == wl.T * wl.E * 2 + R * 6

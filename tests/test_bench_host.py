"""Host-side pieces of the benchmark harness (no GPU): the FLOP counts behind
`value` and `roofline.achieved`, the digest gate on the committed DRAM
traffic, and the clock sampler's reason decoding (NVML replaced by a fake)."""
import importlib.util
import json
import os
import time

import numpy as np
import pytest

from attention_forward_11_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mask_count(Sq, Skv, causal):
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    if causal == 1:
        vis = j <= i + (Skv - Sq)
    elif causal == 2:
        vis = j <= i
    else:
        vis = np.ones((Sq, Skv), dtype=bool)
    return int(vis.sum())


class W:
    def __init__(self, B, Sq, Skv, Hq, Hkv, D, causal):
        self.B, self.Sq, self.Skv, self.Hq, self.Hkv, self.D, self.causal = B, Sq, Skv, Hq, Hkv, D, causal


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("Sq,Skv", [(1, 1), (5, 9), (9, 5), (128, 128), (200, 333), (333, 200)])
def test_visible_pairs_equal_the_mask_count(bench, Sq, Skv, causal):
    w = W(2, Sq, Skv, 4, 2, 128, causal)
    assert bench.visible_pairs(w) == _mask_count(Sq, Skv, causal)
    assert bench.exact_flops(w) == 4 * 128 * 2 * 4 * _mask_count(Sq, Skv, causal)


def test_metric_counts_of_the_benchmark_workloads(bench):
    # 4 * B * Hq * Sq * Skv * D, halved when causal (the metric's own rule)
    head = inputs.WORKLOADS["mha_causal_4x16x4096"]
    assert bench.metric_flops(head) == 274877906944
    assert bench.exact_flops(head) == 274945015808  # exact (query row, key) pairs: 4096 * 4097 / 2 per head
    assert bench.exact_flops(head) == 4 * 128 * 4 * 16 * (4096 * 4097 // 2)
    chunk = inputs.WORKLOADS["chunked_prefill_gqa_64x8_512x32768"]
    assert bench.metric_flops(chunk) == 4 * 64 * 512 * 32768 * 128 // 2
    # bottom-right: row i sees Skv - Sq + i + 1 keys
    assert bench.exact_flops(chunk) == 4 * 128 * 64 * sum(32768 - 512 + i + 1 for i in range(512))
    long_ = inputs.WORKLOADS["long_sharp_1x16x16384"]
    assert bench.metric_flops(long_) == bench.exact_flops(long_) == 4 * 16 * 16384 * 16384 * 128


def test_committed_traffic_matches_the_kernel_source(bench):
    """profiles/traffic.json is read only while its digest matches the forward
    kernel's sources; the committed summary must have been taken on them."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    digest = bench.kernel_source_digest()
    for name, rec in d.items():
        assert rec["kernel_source_digest"] == digest, name
        if "dram_bytes_read" in rec:
            assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert bench.load_traffic(name) == rec["dram_bytes_per_launch"]
    assert bench.load_traffic("no_such_workload") is None


def test_traffic_is_dropped_when_the_kernel_changes(bench, monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0000000000000000")
    assert bench.load_traffic("mha_causal_4x16x4096") is None


class _FakeNvml:
    """Stands in for libnvidia-ml: fixed SM clock and clock-event reason bits."""

    def __init__(self, mhz, reasons):
        self.mhz, self.bits = mhz, reasons

    def nvmlDeviceGetClockInfo(self, handle, kind, out):
        out._obj.value = self.mhz
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle, out):
        out._obj.value = self.bits
        return 0


@pytest.mark.parametrize("bits,expected", [
    (0x1, []),                                               # idle only: not reported
    (0x4, ["sw_power_cap"]),
    (0x8 | 0x40, ["hw_slowdown", "hw_thermal_slowdown"]),
    (0x20 | 0x1, ["sw_thermal_slowdown"]),
])
def test_clock_sampler_reports_reasons_and_median(bench, bits, expected):
    s = bench.ClockSampler(0, period_s=0.001)
    s.nvml, s.handle, s.max_mhz = _FakeNvml(1965, bits), None, 2070
    with s:
        time.sleep(0.02)
    out = s.summary()
    assert out["sm_mhz"] == 1965 and out["sm_max_mhz"] == 2070 and out["samples"] > 0
    assert out["reasons"] == expected


def test_clock_sampler_without_nvml(bench):
    s = bench.ClockSampler(0)
    s.nvml = None
    with s:
        pass
    assert s.summary()["samples"] == 0


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) needs no
    GPU: one JSON line with the keys the harness contract names."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_causal", "--steps", "3", "--warmup", "3", "--ref-step-seconds", "0.2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_causal"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_link_bound_takes_the_slowest_direction(bench):
    link = {"h2d": 200.0, "d2h": 100.0, "both": 250.0}
    b = bench.link_bound(link, 200e9 * 1e-3, 50e9 * 1e-3, 1e12)   # 1 ms up, 0.5 ms down, 1 ms both
    assert abs(b["min_ms_per_step"] - 1.0) < 1e-9
    assert abs(b["max_tflops"] - 1000.0) < 1e-6
    link = {"h2d": 200.0, "d2h": 200.0, "both": 250.0}
    b = bench.link_bound(link, 100e6, 100e6, 1e12)                  # both directions at once bind
    assert abs(b["min_ms_per_step"] - 0.8) < 1e-9


def test_numpy_point_counts_the_visible_pairs(bench):
    tf, dt = bench.numpy_fp64_rate(inputs.WORKLOADS["tiny_causal"])
    assert tf > 0 and dt > 0

"""The benchmark's host-side bookkeeping on CPU: the clock record's summary
(which samples count, which clock-event reasons are reported) and the DRAM
traffic record that the roofline quotes only while the GEMM source matches."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _poller(samples, max_mhz=2032.0):
    p = bench.NvmlPoller.__new__(bench.NvmlPoller)
    p.samples, p.max_mhz = list(samples), max_mhz
    return p


def test_nvml_summary_reports_median_minimum_and_reasons():
    power_cap, hw_slow = 0x4, 0x8
    s = _poller([(2032.0, 0), (1900.0, power_cap), (1950.0, 0), (1800.0, power_cap | hw_slow)]).summary()
    assert s["samples"] == 4 and s["sm_mhz"] == 1925.0 and s["sm_min_mhz"] == 1800.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert _poller([]).summary() is None


def test_clock_sampler_prefers_nvml_and_keeps_both_sources():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    # nvidia-smi lines: index, sm, max sm, power, active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    c.lines = ["0, 1990, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2000, 2032, 910.0, 0x0, Not Active, Active, Not Active, Not Active",
               "0, 2010, 2032, 915.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    c.start, c.stop = 1, 3                       # only the timed region's samples count
    c.nvml = _poller([(2032.0, 0)] * 5)
    s = c.summary()
    assert s["source"].startswith("NVML") and s["samples"] == 5
    assert s["nvidia_smi"]["samples"] == 2 and s["nvidia_smi"]["sm_mhz"] == 2005.0
    # a reason either source saw during the region is reported; the one outside it is not
    assert s["reasons"] == ["hw_thermal_slowdown"]
    c.nvml = _poller([])
    s = c.summary()
    assert s["source"].startswith("nvidia-smi") and s["samples"] == 2


def test_traffic_record_applies_only_to_the_source_it_was_taken_with(tmp_path, monkeypatch):
    """A copy of the tree: the record counts while the GEMM code is unchanged,
    survives comment edits, and is dropped once a line of code changes."""
    import hashlib
    import shutil
    csrc = tmp_path / "mixture_experts_layer_90_b300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gemm.cu", "common.cuh"):
        shutil.copy(os.path.join(ROOT, "mixture_experts_layer_90_b300", "csrc", f), csrc / f)
    h = hashlib.sha1()
    for f in ("gemm.cu", "common.cuh"):
        for ln in open(csrc / f, encoding="utf-8"):
            code = ln.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.md").write_text(f"`gemm1_swiglu: 123456789 {h.hexdigest()[:12]}`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("gemm1_swiglu") == 123456789.0
    assert bench.profiled_traffic("gemm2") is None
    with open(csrc / "gemm.cu", "a", encoding="utf-8") as fh:
        fh.write("// a comment changes nothing\n")
    assert bench.profiled_traffic("gemm1_swiglu") == 123456789.0
    with open(csrc / "gemm.cu", "a", encoding="utf-8") as fh:
        fh.write("static int changed_code = 1;\n")
    assert bench.profiled_traffic("gemm1_swiglu") is None

"""The benchmark's host-side accounting (no GPU).

The algorithmic bytes are checked against the sizes of the tensors the workload
generator actually makes (inputs read once, outputs and final states written
once), the useful flops against the page's count with the feature width the
method uses (273 features for the Taylor map), and the workload descriptions
against the configurations.  The clock record (median under load, throttle
reasons) and the choice of roofline peaks are checked on fake inputs.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _small(name, **over):
    c = dict(workloads.CONFIGS[name])
    c.update(B=1, T=256, **over)
    return c


def test_feature_dim():
    assert bench.feature_dim(workloads.CONFIGS["taylor_linear_attention_bf16"]) == 1 + 16 + 256
    assert bench.feature_dim(workloads.CONFIGS["linear_attention_bf16"]) == 64
    assert bench.feature_dim(workloads.CONFIGS["msr_retention_bf16"]) == 128


def test_alg_bytes_are_the_tensors_once():
    for name in ("linear_attention_bf16", "gated_retention_bf16", "taylor_linear_attention_bf16",
                 "msr_retention_bf16"):
        c = _small(name)
        x = workloads.make_inputs(c)
        B, H, T, dv = c["B"], c["H"], c["T"], c["dv"]
        df = bench.feature_dim(c)
        read = sum(t.numel() * t.element_size() for t in (x["q"], x["k"], x["v"]))
        if c.get("gate"):
            read += x["log_a"].numel() * x["log_a"].element_size()
        out = torch.empty((B, H, T, dv), dtype=x["v"].dtype)
        state = torch.empty((B, H, df, dv), dtype=torch.float32)
        z = torch.empty((B, H, df), dtype=torch.float32) if c["normalize"] else None
        written = out.numel() * out.element_size() + state.numel() * 4 + (z.numel() * 4 if z is not None else 0)
        assert bench.alg_bytes(c) == read + written, name


def test_alg_flops_use_the_feature_width():
    c = workloads.CONFIGS["taylor_linear_attention_bf16"]
    per_token = 4 * 273 * c["dv"] + bench.C_REF * (273 + c["dv"])
    assert bench.alg_flops(c) == c["B"] * c["H"] * c["T"] * per_token
    h = workloads.CONFIGS["linear_attention_bf16"]
    assert bench.alg_flops(h) == h["B"] * h["H"] * h["T"] * (4 * 64 * 64 + bench.C_REF * 128)


def test_descriptions_name_the_feature_map():
    d = bench.describe("taylor_linear_attention_bf16", workloads.CONFIGS["taylor_linear_attention_bf16"])
    assert "Taylor" in d and "273 features" in d and "normalised" in d
    d = bench.describe("linear_attention_bf16", workloads.CONFIGS["linear_attention_bf16"])
    assert "phi=elu+1" in d
    d = bench.describe("gated_retention_bf16", workloads.CONFIGS["gated_retention_bf16"])
    assert "per-token decay" in d and "phi=identity" in d


def test_headline_is_bound_by_bytes_and_taylor_sits_at_the_ridge():
    """Arithmetic intensity (useful flops per algorithmic byte) against the ridge of a
    GB300 (about 1.9 PFLOP/s over 6.8 TB/s, 280 flop/B): the headline far below it,
    the Taylor workload within a few percent of it."""
    ridge = 1.9e15 / 6.8e12
    h = workloads.CONFIGS["linear_attention_bf16"]
    t = workloads.CONFIGS["taylor_linear_attention_bf16"]
    assert bench.alg_flops(h) / bench.alg_bytes(h) < 0.2 * ridge
    ratio = bench.alg_flops(t) / bench.alg_bytes(t) / ridge
    assert 0.9 < ratio < 1.1
    assert np.isfinite(ratio)


def test_clock_summary_takes_the_median_under_load_and_every_reason():
    """The clock record: idle samples (under a quarter of the peak power) stay out of
    the median, and a throttle reason seen in any sample is reported."""
    s = bench.ClockSampler(0)
    s.out = "\n".join([
        "0, 900, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2040, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbled line",
        "0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    c = s.summary()
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 4
    assert c["reasons"] == ["sw_power_cap"]
    s.out = "0, 1500, 2070, 1200.0, 0x8, Active, Not Active, Active, Not Active"
    assert bench.ClockSampler.summary(s)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.out = ""
    assert s.summary() is None


def test_peaks_come_from_the_measured_file(tmp_path, monkeypatch):
    """The roofline's denominators: the measured file when present (sustained falling
    back to burst), else the stated fallback figures."""
    import json
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.5,
                                                              "bf16_tflops": 2000.0}))
    p = bench.peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 7000.5
    assert p["bf16_tflops_sustained"] == 2000.0

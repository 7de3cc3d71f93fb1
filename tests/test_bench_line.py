"""The bench's JSON line, assembled on CPU from fake measurements.

The line is built by one pure function (bench.assemble_line); these tests
give it made-up timings, clock samples and extended-block entries and check
that every key of the bench contract comes out, with the arithmetic the
docstrings state, and that the line is valid JSON.
"""

import json

import bench
from scaled_dot_product_07_gb300 import workloads as W

PEAKS = {"hbm_gbs": 6683.2, "bf16_tflops": 1940.8, "bf16_tflops_sustained": 1728.1}


def _timings(steps=20):
    return {"total_ms": 1.8 * steps, "fwd_ms": 0.41, "bwd_ms": 1.36, "fwd_kernel_ms": 0.405,
            "bwd_main_ms": 1.20}


def test_line_has_every_contract_key():
    w = W.WORKLOADS["decoder_long"]
    clocks = bench.summarize_clocks([(0.0, 1900.0, 2070.0, 900.0, set()),
                                     (0.1, 1950.0, 2070.0, 950.0, {"sw_power_cap"})], "nvml")
    sustained = {"steps": 1600, "ms_per_step": 1.85, "tflops": 1040.0, "clocks": clocks}
    extras = {"graph_step": {"ms": 1.7}}
    e2e = {"value": 590.0, "unit": "TFLOP/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 8,
           "copies_declared": True}
    cpu = {"value": 0.034, "unit": "TFLOP/s", "cores": 16, "kind": "oracle", "sample": "x"}
    line = bench.assemble_line(w, 1, 20, 5, _timings(), PEAKS, "measured", clocks, sustained,
                               extras, e2e, cpu)
    json.loads(json.dumps(line))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline", "sustained",
                "extended", "roofline_fwd", "roofline_bwd_hbm"):
        assert key in line, key
    assert line["metric"] == bench.METRIC
    assert line["dtype"] == "bf16" and line["unit"] == "TFLOP/s"
    assert line["config"]["workload"].startswith("decoder_long B8 H16 Sq4096 Sk4096 D128 causal")
    f, b = bench.flops(w)
    assert abs(line["value"] - (f + b) / 1.8e-3 / 1e12) < 1e-9
    r = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r
    assert r["bound"] == "tensor" and r["peak"] == PEAKS["bf16_tflops"]
    assert abs(r["achieved"] - b / 1.2e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert line["sustained"]["peak"] == PEAKS["bf16_tflops_sustained"]
    assert abs(line["sustained"]["frac"] - 1040.0 / 1728.1) < 1e-12
    hbm = line["roofline_bwd_hbm"]
    assert hbm["achieved"] > 0 and hbm["peak"] == PEAKS["hbm_gbs"]
    assert line["gpu_launches"] == 4 * 20
    assert line["cpu_baseline"]["cores"] == 16


def test_hbm_figure_is_null_when_the_difference_is_not_positive():
    w = W.WORKLOADS["decoder_long"]
    t = _timings()
    t["bwd_main_ms"] = t["bwd_ms"] + 0.001  # event noise
    line = bench.assemble_line(w, 1, 20, 5, t, PEAKS, "measured",
                               bench.summarize_clocks([], "nvml"))
    assert line["roofline_bwd_hbm"]["achieved"] is None
    assert line["roofline_bwd_hbm"]["frac"] is None
    json.dumps(line)


def test_fallback_peaks_are_used_without_the_measured_file():
    w = W.WORKLOADS["decoder_long"]
    line = bench.assemble_line(w, 2, 10, 3, _timings(10), bench.FALLBACK_PEAKS, "fallback",
                               bench.summarize_clocks([], None))
    assert line["roofline"]["peak"] == bench.FALLBACK_PEAKS["bf16_tflops"]
    assert "fallback" in line["roofline"]["peak_source"]
    # weak scaling: two ranks, each with the whole workload
    f, b = bench.flops(w)
    assert abs(line["value"] - 2 * (f + b) / 1.8e-3 / 1e12) < 1e-9
    assert line["clocks"]["reasons"] == ["no clock source"]


def test_clock_window_keeps_only_its_samples_and_flags_throttling():
    s = bench.ClockSampler(0)
    s.source = "nvml"
    s.samples = [(0.5, 2070.0, 2070.0, 200.0, set()),
                 (1.0, 1800.0, 2070.0, 1000.0, {"sw_power_cap"}),
                 (1.5, 1700.0, 2070.0, 1100.0, {"sw_power_cap"}),
                 (2.5, 1000.0, 2070.0, 1100.0, {"hw_slowdown"})]
    c = s.window(0.9, 2.0)
    assert c["samples_under_load"] == 2
    assert c["sm_mhz"] == 1750.0 and c["sm_min_mhz"] == 1700.0
    assert c["reasons"] == ["sw_power_cap"] and c["rejected"] is False
    c2 = s.window(0.9, 3.0)
    assert c2["rejected"] is True and "hw_slowdown" in c2["reasons"]


def test_philox_alu_bound_of_the_decoder_forward():
    """One Philox group per four visible pairs; the integer bound is the
    busier of the ALU pipe (64 lane-operations per clock per SM) and the
    FMA-heavy pipe's wide multiplies (32 per clock per SM), and the pass's
    roofline the larger of that and its tensor bound."""
    w = W.make_workload("decoder_long", dropout_p=0.1)
    groups = 4096 * 4097 // 2 * 8 * 16 / 4
    r = bench.philox_alu_bound(w, "fwd", 2000.0, 1.35, 0.41, 1940.8)
    assert r["groups"] == groups
    alu_ms = groups * bench.PHILOX_OPS["fwd"]["alu"] / (64 * 152 * 2000e6) * 1e3
    mul_ms = groups * bench.PHILOX_OPS["fwd"]["mul_wide"] / (32 * 152 * 2000e6) * 1e3
    assert mul_ms > alu_ms  # 20 wide multiplies at half rate outweigh 28 ALU operations
    assert abs(r["alu_bound_ms"] - mul_ms) < 1e-12
    # the backward forms its round keys and quad nibbles: the ALU pipe is busier
    rb = bench.philox_alu_bound(w, "bwd", 2000.0, 2.0, 1.36, 1940.8)
    assert abs(rb["alu_bound_ms"] - groups * 56 / (64 * 152 * 2000e6) * 1e3) < 1e-12
    alu_ms = mul_ms
    tensor_ms = bench.flops(w)[0] / 1940.8e12 * 1e3
    assert abs(r["tensor_bound_ms"] - tensor_ms) < 1e-12
    assert r["bound"] == "alu" and abs(r["frac"] - max(alu_ms, tensor_ms) / 1.35) < 1e-12
    assert abs(r["dropout_extra_ms"] - 0.94) < 1e-12


def test_stored_bits_line():
    """The dropout pair with the keep bits carried in a buffer: its step is
    the two passes, beside the pair that draws them twice, and its backward
    is read against the tensor peak alone."""
    w = W.make_workload("decoder_long", dropout_p=0.1)
    r = bench.stored_bits_line(w, 1.5, 1.46, 1.31, 2.03, 268435456, 1940.8)
    assert abs(r["step_ms"] - 2.96) < 1e-12 and abs(r["step_ms_redrawn"] - 3.34) < 1e-12
    b = bench.flops(w)[1]
    assert abs(r["bwd_tflops"] - b / 1.46e-3 / 1e12) < 1e-9
    assert abs(r["bwd_frac"] - r["bwd_tflops"] / 1940.8) < 1e-12
    assert r["bits_bytes"] == 268435456

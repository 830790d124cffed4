"""Host-side pieces of bench.py that need no GPU: the clock summary, the check
that a stored ncu traffic figure belongs to the current kernel sources, and
the NVML sampler's failure on a machine without a driver (bench then falls
back to nvidia-smi)."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _row(sm, power=500.0, hw="Not Active", hw_thermal="Not Active", sw_thermal="Not Active",
         sw_power="Not Active"):
    return dict(sm=sm, max=2070.0, power=power, hw=hw, hw_thermal=hw_thermal,
                sw_thermal=sw_thermal, sw_power=sw_power)


def test_clock_summary_median_and_reasons():
    rows = [_row(2070.0), _row(1800.0, sw_power="Active"), _row(1900.0)]
    s = bench.ClockSampler.summary(rows)
    assert s["sm_mhz"] == 1900.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    s = bench.ClockSampler.summary([_row(1500.0, hw="Active", hw_thermal="Active")])
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_summary_raw_reason_mask():
    """The OR of the raw masks is kept, and bits outside the four the timing
    rules act on are named (HW power brake, idle, ...)."""
    rows = [_row(2070.0), _row(2070.0), _row(2070.0)]
    rows[1]["mask"] = 0x80
    rows[2]["mask"] = 0x1 | 0x4
    rows[2]["sw_power"] = "Active"
    s = bench.ClockSampler.summary(rows)
    assert s["reasons"] == ["sw_power_cap"]
    assert s["reasons_mask"] == "0x85"
    assert s["other_reasons"] == ["gpu_idle", "hw_power_brake_slowdown"]
    s = bench.ClockSampler.summary([_row(2070.0)])  # rows without a mask
    assert s["reasons_mask"] == "0x0" and s["other_reasons"] == []


def test_clock_summary_memory_clock_range():
    rows = [_row(2070.0), _row(2070.0)]
    rows[0]["mem"], rows[1]["mem"] = 3996.0, 3200.0
    s = bench.ClockSampler.summary(rows)
    assert s["mem_mhz_min"] == 3200.0 and s["mem_mhz_max"] == 3996.0
    assert "mem_mhz_min" not in bench.ClockSampler.summary([_row(2070.0)])


def test_clock_summary_without_samples():
    s = bench.ClockSampler.summary([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []


def test_stored_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "tensor_core_dense_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cuh").write_text("// kernel v1\n")
    (csrc / "h.cuh").write_text("// helper\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha(["k.cuh", "h.cuh"])
    (tmp_path / "profiles" / "p.md").write_text(
        "# profile\n\nsource_files: `k.cuh h.cuh`\n"
        f"source_sha256: `{sha}`\ntraffic_bytes_per_launch: 12345\n")
    assert bench.stored_traffic("p.md") == 12345
    (csrc / "k.cuh").write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.stored_traffic("p.md") is None
    assert bench.stored_traffic("missing.md") is None


def test_committed_profile_is_parsed():
    """The committed headline summary carries a hash and a traffic figure
    (whether they still match the sources is what the bench line reports)."""
    text = open(os.path.join(ROOT, "profiles", "gemm_tn2_bf16_4096.md")).read()
    assert "source_sha256:" in text and "traffic_bytes_per_launch:" in text
    t = bench.stored_traffic()
    assert t is None or t > 0


def test_nvml_sampler_fails_cleanly_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises((OSError, AttributeError)):
        bench.NvmlSampler("GPU-00000000-0000-0000-0000-000000000000")


def test_isa_peak_arithmetic():
    # 8,192 BF16 FLOP/clk/SM x 152 SMs x 2.07 GHz; FP8 twice that
    assert bench.isa_peak_tflops(152, 2070.0) == pytest.approx(2577.5, abs=0.1)
    assert bench.isa_peak_tflops(152, 2070.0, fp8=True) == pytest.approx(5155.1, abs=0.1)
    assert bench.isa_peak_tflops(152, None) is None


def test_peak_fractions_by_input_type():
    """Every FP8 workload (per tensor, block-scaled, microscaled) is measured
    against the FP8 rates, the BF16 ones against the BF16 rates."""
    for name in ("fp8_4096", "fp8_block_4096", "fp8_skinny_128", "mxfp8_4096"):
        o = bench.add_peak_fractions({"workload": name, "tflops": 2577.5}, 1000.0, 152, 2070.0)
        assert "frac_of_bf16_peak" not in o
        assert o["frac_of_fp8_peak"] == pytest.approx(2577.5 / (1000.0 * bench.FP8_OVER_BF16), abs=1e-4)
        assert o["frac_of_isa_peak_at_clock"] == pytest.approx(0.5, abs=1e-4)
    for name in ("bf16_4096", "bf16_mlp", "bf16_skinny_16"):
        o = bench.add_peak_fractions({"workload": name, "tflops": 2577.5}, 1000.0, 152, 2070.0)
        assert "frac_of_fp8_peak" not in o
        assert o["frac_of_bf16_peak"] == pytest.approx(2.5775, abs=1e-4)
        assert o["frac_of_isa_peak_at_clock"] == pytest.approx(1.0, abs=1e-4)


def test_cpu_baseline_config_tiles_and_extrapolation():
    import synth.workloads as W
    w = W.make("bf16_256")
    r = bench.cpu_baseline_config(w, 0.01, 2)
    assert r["tiles"] == 1 and r["tile"] == "whole output"
    assert r["full_output_s_extrapolated"] == pytest.approx(r["wall_s"], rel=0.05, abs=0.05)
    w = W.make("fp8_skinny_16", N=8192, K=256)
    r = bench.cpu_baseline_config(w, 0.0, 3)   # one batch: one tile per core
    assert r["tiles"] == 3
    # the fixed set leads with the first and the last tile
    tiles = W.sample_tiles(16, 1024, n=8)
    assert tiles[0][:2] == (0, 0) and tiles[1][:2] == (0, 1024 - 128)

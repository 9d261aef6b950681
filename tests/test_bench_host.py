"""Host logic of bench.py (no GPU): the algorithmic bytes and FLOPs the roofline
fractions divide by, the lookup of profiled DRAM traffic, the peak selection and the
whole-job rate."""
import json
import os

import pytest

import bench
import synthetic as syn


def test_step_bytes_and_flops_match_the_workload_table():
    """Per-step bytes and FLOPs of the 27B workloads against the table of the hot-path
    scope (readout 1.842 / 1.914 GB, verify 6.1 / 97.2 MB, 12.9 / 205.8 GFLOP)."""
    b1 = bench.step_bytes(syn.CONFIGS["27b_b1"], 1)
    assert round((b1["fc"] + b1["lm_head"] + b1["chain"]) / 1e9, 3) == 1.842
    assert round(b1["verify"] / 1e6, 1) == 6.1
    assert round(bench.step_flops(syn.CONFIGS["27b_b1"]) / 1e9, 1) == 12.9
    b16 = bench.step_bytes(syn.CONFIGS["27b_b16"], 1)
    assert round((b16["fc"] + b16["lm_head"] + b16["chain"]) / 1e9, 3) == 1.914
    assert round(b16["verify"] / 1e6, 1) == 97.2
    assert round(bench.step_flops(syn.CONFIGS["27b_b16"]) / 1e9, 1) == 205.8
    # the LM-head term alone: each weight byte once, h read, the fp32 logits written
    assert b1["lm_head"] == 1_560_150_528
    assert b1["total"] == b1["fc"] + b1["lm_head"] + b1["chain"] + b1["verify"]
    # greedy verify draws nothing: no resample rows
    assert bench.step_bytes(syn.CONFIGS["27b_b1"], 0)["verify"] == 8 * 151936 * 4


def test_fp8_step_bytes_halve_the_weight_stream():
    b = bench.step_bytes(syn.CONFIGS["27b_b1"], 1)
    b8 = bench.step_bytes(syn.CONFIGS["27b_b1_fp8"], 1)
    V, H = 151936, 5120
    # one byte per weight plus a fp32 scale per row, instead of two bytes per weight
    assert b["lm_head"] - b8["lm_head"] == V * H - V * 4 - 2 * 7 * H


def _write_profile(root, workload, traffic, src_text, sha=None):
    import hashlib
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "kernel.cu"), "w") as f:
        f.write(src_text)
    if sha is None:
        sha = hashlib.sha256(src_text.encode()).hexdigest()[:16]
    with open(os.path.join(root, "profiles", "gemm_tcgen05_lm_head_%s.md" % workload), "w") as f:
        f.write("# capture\n\n| metric | value |\n|---|---|\n| x | 1 |\n\n")
        f.write("traffic_bytes_per_launch: %d\nsource: kernel.cu\nsource_sha256_16: %s\n" % (traffic, sha))


def test_profiled_traffic_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write_profile(str(tmp_path), "w1", 123456789, "kernel source\n")
    assert bench.profiled_traffic("w1") == 123456789
    assert bench.profiled_traffic("missing") is None
    with open(os.path.join(str(tmp_path), "kernel.cu"), "a") as f:
        f.write("// edited\n")
    assert bench.profiled_traffic("w1") is None


def test_committed_profiles_name_a_source_and_a_hash():
    for w in ("27b_b1", "27b_b16", "27b_b1_fp8", "flash_b4"):
        path = os.path.join(bench.ROOT, "profiles", "gemm_tcgen05_lm_head_%s.md" % w)
        text = open(path).read()
        assert "traffic_bytes_per_launch:" in text and "source_sha256_16:" in text


def test_measured_peaks_fall_back_when_no_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, bench.FALLBACK_BF16_TFLOPS, "fallback")
    with open(os.path.join(str(tmp_path), "MEASURED_PEAKS.json"), "w") as f:
        json.dump({"gb300": {"hbm_gbs": 7123.0, "bf16_tflops": 2001.0,
                             "bf16_tflops_sustained": 1700.0}}, f)
    hbm, tflops, src = bench.measured_peaks()
    assert (hbm, tflops, src) == (7123.0, 2001.0, "measured")


@pytest.mark.parametrize("units,world,secs,rate", [(100, 1, 2.0, 50.0), (100, 4, 2.0, 200.0)])
def test_whole_job_rate_counts_every_rank(units, world, secs, rate):
    assert bench.whole_job_rate(units, world, secs) == rate


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, lines):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    cs.fh = open(cs.path, "a")
    cs.proc = _FakeProc()
    return cs


def test_clock_sampler_reports_median_clock_and_throttle_reasons(tmp_path):
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1390.2, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1001.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line",
            "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    out = _sampler_with(tmp_path, rows).stop()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    hot = ["0, 1500, 2070, 1400.0, 0x48, Active, Not Active, Active, Not Active"] * 3
    assert _sampler_with(tmp_path, hot).stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler_with(tmp_path, ["nothing parseable"]).stop() is None

"""Host-side arithmetic of bench.py's JSON line (no GPU): the algorithmic flops
and compulsory bytes per step that the roofline fraction divides by, the bound
it picks, and where the per-launch DRAM traffic comes from."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from persistent_step_megakernel_gb300 import synthetic as S  # noqa: E402


def test_step_flops_count_every_gemm():
    # C5: 4 forward, 4 weight-grad and 3 input-grad GEMMs of 4096^3 (layer 1 has no input grad)
    assert S.CONFIGS["c5"].flops() == 11 * 2 * 4096 ** 3
    # C2: 64 x (256*512 + 512*512 + 512*128) per GEMM kind; 2 flops per MAC
    macs = 64 * (256 * 512 + 512 * 512 + 512 * 128)
    assert S.CONFIGS["c2"].flops() == 2 * (3 * macs - 64 * 256 * 512)


def test_compulsory_bytes_of_the_headline_step():
    # bf16 parameters read and written, x and y read, the loss written
    params = 256 * 512 + 512 * 512 + 512 * 128 + 512 + 512 + 128
    want = 2 * (2 * params + 64 * 256 + 64 * 128 + 1)
    assert S.CONFIGS["c2"].compulsory_bytes() == want


@pytest.fixture
def peaks_dir(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_roofline_picks_the_binding_resource(peaks_dir):
    c5, c2 = S.CONFIGS["c5"], S.CONFIGS["c2"]
    r = bench.roofline(c5, 1e-3, None)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0 and r["peak_source"] == "measured"
    assert r["achieved"] == pytest.approx(c5.flops() / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    r = bench.roofline(c2, 50e-6, 12345)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 12345
    assert r["achieved"] == pytest.approx(c2.compulsory_bytes() / 50e-6 / 1e9)
    assert r["roofline_us"] == pytest.approx(c2.compulsory_bytes() / 7000e9 * 1e6)


def test_traffic_is_taken_only_from_a_summary_of_the_same_kernel_source(peaks_dir, monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "abc123")
    path = peaks_dir / "profiles" / f"{bench.KERNEL}_c2.md"
    path.write_text("# summary\n\nsource_sha: abc123\ndram_bytes_per_launch: 1160960\n")
    assert bench.traffic_from_profiles("c2") == 1160960
    path.write_text("# summary\n\nsource_sha: 0000\ndram_bytes_per_launch: 1160960\n")
    assert bench.traffic_from_profiles("c2") is None          # stale counters are not reported
    assert bench.traffic_from_profiles("c4") is None          # no summary at all


def test_sampled_oracle_rate_scales_to_whole_steps():
    # a bounded sample of whole steps: the rate is reported per whole step
    value, frac, threads = bench.oracle_sampled(S.CONFIGS["c1"], 0.5, steps=2, warmup=1)
    assert value > 0 and 0 < frac <= 1 and threads >= 1


def test_back_to_back_batches_follow_the_step_size():
    assert bench.batch_steps_for(S.CONFIGS["c5"]) == 20
    assert bench.batch_steps_for(S.CONFIGS["c2"]) == 100


def test_clock_summary_uses_busy_samples_and_keeps_every_reason():
    c = bench.Clocks(0)
    c.lines = ["2070, 2070, 500.1, Not Active, Not Active, Not Active, Active, 95",
               "1900, 2070, 300.0, Not Active, Not Active, Not Active, Not Active, 0",
               "2055, 2070, 640.0, Not Active, Not Active, Not Active, Not Active, 90"]
    s = c.summary()
    assert s["sm_mhz"] == 2062.5 and s["sm_max_mhz"] == 2070 and s["samples"] == 3 and s["samples_busy"] == 2
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 640.0
    c.lines = ["1900, 2070, 300.0, Not Active, Not Active, Not Active, Not Active, 0"]
    assert c.summary()["sm_mhz"] == 1900                     # no busy sample: all samples

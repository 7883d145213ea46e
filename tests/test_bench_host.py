"""Host logic of bench.py (no GPU): the roofline's recorded DRAM traffic is
used only while the kernel sources match the capture, the clock samplers
decode throttle reasons (a run that saw a thermal or hardware slowdown is
rejected on these names), and the metric's arithmetic follows its closed
forms."""
import json
import os
import shutil
import statistics
import threading
import types

import pytest

import bench
import mla_inputs as mi


def _write_profile(root, name, sha, bytes_):
    d = os.path.join(root, "profiles")
    os.makedirs(d, exist_ok=True)
    with open(os.path.join(d, name), "w") as f:
        f.write("some kernel on some workload\n")
        f.write(f"kernel_source_sha: {sha}\n")
        f.write(f"dram_bytes_per_launch: {bytes_}\n")
        f.write("(a note line: with a colon)\n")


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write_profile(str(tmp_path), "fwd_kernel_config2_ncu.txt", "abc123", "39517440.0")
    _write_profile(str(tmp_path), "bwd_kernel_config2_ncu.txt", "abc123", "not-a-number")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kind="fwd": "abc123")
    assert bench.profiled_traffic(2, "fwd") == 39517440.0
    assert bench.profiled_traffic(2, "bwd") is None          # malformed figure
    assert bench.profiled_traffic(3, "fwd") is None          # no capture of that workload
    assert bench.profiled_traffic(3, "idx") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kind="fwd": "def456")
    assert bench.profiled_traffic(2, "fwd") is None          # sources changed since the capture


def test_kernel_source_hash_tracks_each_family(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "serving_sparse_mla_gb300", "csrc")
    dst = os.path.join(str(tmp_path), "serving_sparse_mla_gb300", "csrc")
    os.makedirs(dst)
    for name in {n for names in bench.KERNEL_SOURCES.values() for n in names}:
        shutil.copy(os.path.join(src, name), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert before == {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}   # deterministic
    with open(os.path.join(dst, "bwd_kernel.cuh"), "a") as f:
        f.write("\n// edit\n")
    after = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert after["bwd"] != before["bwd"]
    assert after["fwd"] == before["fwd"] and after["idx"] == before["idx"]
    with open(os.path.join(dst, "ptx.cuh"), "a") as f:
        f.write("\n// edit\n")
    final = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert all(final[k] != after[k] for k in bench.KERNEL_SOURCES)


def _nvml_with_samples(samples, max_mhz=2070):
    s = object.__new__(bench.NvmlClockSampler)
    s.ok = True
    s.samples = list(samples)
    s.max_mhz = max_mhz
    s._run, s._stop = threading.Event(), threading.Event()
    s.thread = types.SimpleNamespace(join=lambda timeout=None: None)
    return s


def test_nvml_sampler_decodes_reasons():
    got = _nvml_with_samples([(2070, 300.0, 0x0), (2055, 320.0, 0x4), (1980, 340.0, 0x4 | 0x40)]).stop()
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert got["sm_mhz"] == 2055 and got["sm_max_mhz"] == 2070 and got["samples"] == 3
    assert got["power_w_median"] == 320.0
    got = _nvml_with_samples([(2070, 200.0, 0x8), (2070, 200.0, 0x20)]).stop()
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _nvml_with_samples([(2070, 200.0, 0x1 | 0x2 | 0x100)]).stop()["reasons"] == []   # idle / app clocks
    assert _nvml_with_samples([]).stop() is None


def test_smi_sampler_parses_its_csv(tmp_path):
    path = os.path.join(str(tmp_path), "clocks.csv")
    rows = ["0, 2070, 2070, 310.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 2040, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, [N/A], 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1500, 2070, 1400.0, 0x0000000000000040, Not Active, Active, Not Active, Active",
            "garbage"]
    with open(path, "w") as f:
        f.write("\n".join(rows) + "\n")
    s = bench.ClockSampler(0, str(tmp_path))
    s.path = path
    s.fh = open(os.devnull, "w")
    s.proc = types.SimpleNamespace(terminate=lambda: None, wait=lambda timeout=None: 0, kill=lambda: None)
    got = s.stop()
    assert got["samples"] == 3
    assert got["sm_mhz"] == statistics.median([2070, 2040, 1500]) and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_metric_arithmetic_closed_forms():
    c1 = bench.workload(1)
    assert bench.valid_entries(c1) == 2080
    assert bench.step_flops(c1) == 2.0 * 64 * 8 * 2048 * (576 + 512)
    # whole-job rate: units of all ranks over the slowest rank's time
    assert bench.whole_job_tflops(2e12, 10, 4, 1000.0) == pytest.approx(80.0)
    dec = mi.decode_case(703, 4, 6, 8, 500, 3000, topk=512, poison=False)
    assert bench.step_flops(dec) == 2.0 * 4 * 6 * 8 * 512 * 1088
    assert bench.workload(2, tokens=300).q.shape == (300, 8, 576)
    assert bench.workload(3, tokens=256).q.shape == (256, 64, 576)
    with pytest.raises(SystemExit):
        bench.workload(5, tokens=100)


def test_peaks_file_or_fallback(tmp_path, monkeypatch):
    d, kind = bench.load_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and d["hbm_gbs"] > 0 and d["bf16_tflops"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d, kind = bench.load_peaks()
    assert kind == "fallback" and d == bench.FALLBACK_PEAKS
    with open(os.path.join(str(tmp_path), "MEASURED_PEAKS.json"), "w") as f:
        json.dump({"hbm_gbs": 1.0, "bf16_tflops": 2.0}, f)
    assert bench.load_peaks() == ({"hbm_gbs": 1.0, "bf16_tflops": 2.0}, "measured")

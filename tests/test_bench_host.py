"""Host-side pieces of bench.py on CPU: the clock and throttle-reason sampler
against a stand-in NVML, the peak lookup, and the rule that a profile's
traffic figure counts only when it was taken from the current kernel
sources."""
import ctypes
import json
import os

import pytest
import torch

import bench


class _FakeNvml:
    """Read-only NVML calls the sampler makes; clocks and reason bits are
    played back in order."""

    def __init__(self, clocks, reasons, max_mhz=2070):
        self.clocks, self.reasons, self.max_mhz, self.i = list(clocks), list(reasons), max_mhz, 0

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, handle):
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, index, handle):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, kind, out):
        out._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetClockInfo(self, handle, kind, out):
        out._obj.value = self.clocks[min(self.i, len(self.clocks) - 1)]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle, out):
        out._obj.value = self.reasons[min(self.i, len(self.reasons) - 1)]
        self.i += 1
        return 0


class _Props:
    uuid = "0000-fake"


def _sampler(monkeypatch, clocks, reasons):
    fake = _FakeNvml(clocks, reasons)
    monkeypatch.setattr(ctypes, "CDLL", lambda *a, **k: fake)
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda i: _Props())
    s = bench.ClockSampler(0, interval_s=0.0)
    assert s.ok and s.max_mhz == 2070
    return s, fake


def test_clock_sampler_reports_median_and_reasons(monkeypatch):
    s, fake = _sampler(monkeypatch, [2070, 2070, 1900, 2070, 2070], [0, 0x4, 0, 0x8, 0])
    for _ in range(5):
        s._sample()
    s._thread = type("NoThread", (), {"join": lambda self: None})()   # sampled by hand above
    out = s.stop()
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 5
    assert out["reasons"] == ["sw_power_cap", "hw_slowdown"]


def test_clock_sampler_thread_collects_samples(monkeypatch):
    s, fake = _sampler(monkeypatch, [1500] * 1000, [0x40] * 1000)
    s.start()
    import time
    time.sleep(0.05)
    out = s.stop()
    assert out["samples"] >= 1 and out["sm_mhz"] == 1500
    assert out["reasons"] == ["hw_thermal_slowdown"]


def test_clock_sampler_without_nvml_reports_nothing(monkeypatch):
    def no_lib(*a, **k):
        raise OSError("no NVML")
    monkeypatch.setattr(ctypes, "CDLL", no_lib)
    s = bench.ClockSampler(0)
    assert not s.ok
    s.start()
    assert s.stop() is None


def test_measured_peak_and_fallback(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6791.7}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (6791.7, "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_profile_traffic_only_for_current_sources(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "pa_decode_w.md").write_text(
        "x\nsource_sha256: abcdef0123456789\ntraffic_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abcdef0123456789")
    assert bench.profile_name("w") == "pa_decode_w"
    assert bench.profile_traffic(bench.profile_name("w")) == 12345
    monkeypatch.setattr(bench, "source_digest", lambda: "0000000000000000")
    assert bench.profile_traffic("pa_decode_w") is None      # kernels changed since the capture
    assert bench.profile_traffic("pa_decode_missing") is None


def test_profile_names_follow_the_configuration():
    assert bench.profile_name("long_ctx_fp8", 512) == "pa_decode_long_ctx_fp8_p512"
    assert bench.profile_name("qwen7b_fp16", 0, 8) == "pa_attention_qwen7b_fp16_q8"
    assert bench.profile_name("qwen7b_fp16") == "pa_decode_qwen7b_fp16"
    assert bench.profile_name("qwen7b_fp16", simt=True) == "pa_decode_qwen7b_fp16_simt"


def test_committed_profiles_name_their_digest_and_traffic():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = [n for n in os.listdir(os.path.join(root, "profiles")) if n.startswith(("pa_decode_", "pa_attention_"))]
    assert names
    for n in names:
        txt = open(os.path.join(root, "profiles", n)).read()
        assert "source_sha256:" in txt and "traffic_bytes_per_launch:" in txt, n


def test_source_digest_follows_code_not_comments():
    a = "int f(int x) {  // doubles\n    return 2 * x; /* fast */\n}\n"
    b = "// a header line\nint f(int x) {\n    return 2 * x;\n}\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)

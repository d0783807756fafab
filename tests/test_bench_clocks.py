"""The clock record of the timed region, parsed from nvidia-smi's CSV samples
(a stand-in process here, no GPU): median SM clock, the maximum, and every
throttle reason seen active in any sample; and the peaks the roofline divides by."""
import bench


class _FakeSmi:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _record(lines):
    s = bench.ClockSampler(None)
    s.proc = _FakeSmi("\n".join(lines) + "\n")
    return s.stop()


def test_median_clock_and_no_reason():
    rows = ["0, %d, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, "
            "Not Active" % mhz for mhz in (2070, 2040, 2070, 1995, 2070)]
    rec = _record(rows)
    assert rec["sm_mhz"] == 2070 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == [] and rec["samples"] == 5


def test_reasons_seen_in_any_sample_are_reported():
    rows = ["0, 2070, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1800, 2070, 1400.0, 0x48, Not Active, Active, Not Active, Active",
            "garbage line",
            "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    rec = _record(rows)
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["samples"] == 2 and rec["sm_mhz"] == (2070 + 1800) / 2


def test_without_nvidia_smi():
    s = bench.ClockSampler(None)
    rec = s.stop()
    assert rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]


def test_measured_peaks_or_fallback(tmp_path):
    import json
    good = tmp_path / "peaks.json"
    good.write_text(json.dumps({"hbm_gbs": 6792.1, "bf16_tflops": 1930.6,
                                "bf16_tflops_sustained": 1716.1, "chip": "GB300"}))
    peaks, kind = bench.measured_peaks(str(good))
    assert kind == "measured" and peaks["hbm_gbs"] == 6792.1
    partial = tmp_path / "partial.json"
    partial.write_text(json.dumps({"hbm_gbs": 6792.1}))
    for path in (partial, tmp_path / "missing.json"):
        peaks, kind = bench.measured_peaks(str(path))
        assert kind == "fallback" and peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert bench.measured_peaks(str(bad))[1] == "fallback"

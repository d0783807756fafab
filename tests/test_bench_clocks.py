"""The clock record of the timed region, parsed from nvidia-smi's CSV samples
(a stand-in process here, no GPU): median SM clock, the maximum, and every
throttle reason seen active in any sample."""
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

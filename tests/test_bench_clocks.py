"""bench.py's clock sampling, on CPU against a stand-in NVML library and canned nvidia-smi lines.

The bench reports the median SM clock and every throttle reason seen while the timed region
ran; a run with a thermal or hardware slowdown is rejected, so the reason bits must map to
the right names and samples outside the region must not count.
"""
import os
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeNvml:
    """Answers the read-only queries the sampler makes; the clock and reason mask are settable."""

    def __init__(self, uuid="GPU-1234", mhz=2070, max_mhz=2070, mask=0, event_reasons_name=True):
        self.uuid = uuid
        self.mhz, self.max_mhz, self.mask = mhz, max_mhz, mask
        self.inits = self.shutdowns = 0
        if event_reasons_name:
            self.nvmlDeviceGetCurrentClocksEventReasons = self._reasons
        else:
            self.nvmlDeviceGetCurrentClocksThrottleReasons = self._reasons

    def nvmlInit_v2(self):
        self.inits += 1
        return 0

    def nvmlShutdown(self):
        self.shutdowns += 1
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        if uuid.decode() != self.uuid:
            return 13  # NVML_ERROR_NOT_FOUND
        ref._obj.value = 0x1000
        return 0

    def nvmlDeviceGetClockInfo(self, handle, clock, ref):
        assert clock == 1  # NVML_CLOCK_SM
        ref._obj.value = self.mhz
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, clock, ref):
        assert clock == 1
        ref._obj.value = self.max_mhz
        return 0

    def _reasons(self, handle, ref):
        ref._obj.value = self.mask
        return 0


def test_reason_bits_map_to_names():
    assert bench.nvml_reason_names(0) == set()
    assert bench.nvml_reason_names(0x1) == set()  # idle is not a throttle reason
    assert bench.nvml_reason_names(0x4) == {"sw_power_cap"}
    assert bench.nvml_reason_names(0x8 | 0x40) == {"hw_slowdown", "hw_thermal_slowdown"}
    assert bench.nvml_reason_names(0x20) == {"sw_thermal_slowdown"}


@pytest.mark.parametrize("event_name", [True, False])
def test_nvml_sampler_collects_many_samples_in_a_short_region(event_name):
    lib = FakeNvml(mhz=2040, max_mhz=2070, mask=0x4, event_reasons_name=event_name)
    s = bench.NvmlClockSampler("GPU-1234", lib=lib, period_s=0.001)
    s.start()
    time.sleep(0.01)
    t0 = time.time()
    time.sleep(0.03)
    t1 = time.time()
    lib.mask = 0x20  # after the region: must not be reported
    time.sleep(0.01)
    out = s.stop(t0, t1)
    assert lib.shutdowns == 1
    assert out["samples"] >= 5
    assert out["sm_mhz"] == 2040 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["source"].startswith("nvml")


def test_nvml_sampler_refuses_an_unknown_device():
    lib = FakeNvml(uuid="GPU-aaaa")
    with pytest.raises(OSError):
        bench.NvmlClockSampler("GPU-bbbb", lib=lib)
    assert lib.shutdowns == 1


def test_nvidia_smi_lines_parse_and_window():
    lines = [
        (1.0, "2070, 2070, 900.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"),
        (2.0, "1980, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active"),
        (3.0, "2010, 2070, 1380.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active"),
        (4.0, "1500, 2070, 1400.0, 0x0000000000000040, Not Active, Active, Not Active, Not Active"),
        (2.5, "garbage"),
    ]
    out = bench.summarise_clock_samples(bench.ClockSampler.parse(lines), 1.5, 3.5, "nvidia-smi")
    assert out["samples"] == 2
    assert out["sm_mhz"] == pytest.approx(1995.0)
    assert out["reasons"] == ["sw_power_cap"]
    out = bench.summarise_clock_samples(bench.ClockSampler.parse(lines), 3.5, 4.5, "nvidia-smi")
    assert out["reasons"] == ["hw_thermal_slowdown"]
    assert bench.summarise_clock_samples([], 0.0, 1.0, "x") is None

"""Host logic of bench.py's clock sampling (no GPU): NVML reason bits, and the summary of the
samples taken inside the timed region, driven by a fake reader."""
import time

import bench


def test_decode_reasons():
    assert bench.decode_reasons(0) == []
    assert bench.decode_reasons(0x1 | 0x2 | 0x10 | 0x100) == []  # idle, app clocks, sync boost, display
    assert bench.decode_reasons(0x4) == ["sw_power_cap"]
    assert bench.decode_reasons(0x8 | 0x40) == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.decode_reasons(0x20 | 0x80) == ["hw_power_brake_slowdown", "sw_thermal_slowdown"]


class FakeReader:
    """Stands in for NvmlReader: clocks and reasons follow a script, one entry per read."""

    def __init__(self, script):
        self.script = script
        self.i = 0

    def read(self):
        r = self.script[min(self.i, len(self.script) - 1)]
        self.i += 1
        return dict(r)


def _run(sampler, before_s, inside_s):
    sampler.start()
    time.sleep(before_s)
    sampler.mark_start()
    time.sleep(inside_s)
    sampler.mark_stop()
    return sampler.stop()


def test_summary_of_samples_inside_the_region():
    quiet = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w": 300.0, "reasons": 0}
    capped = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "power_w": 1400.0, "reasons": 0x4}
    s = bench.ClockSampler(0, reader=FakeReader([quiet] * 10 + [capped] * 10000), period_s=0.001)
    out = _run(s, 0.05, 0.05)
    assert out["source"].startswith("nvml")
    assert out["samples"] > 5
    assert out["sm_mhz"] == 1800.0  # every sample inside the region is a capped one
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 1400.0


def test_unreadable_reader_gives_no_samples():
    class Broken:
        def read(self):
            return None
    s = bench.ClockSampler(0, reader=Broken(), period_s=0.001)
    out = _run(s, 0.01, 0.01)
    assert out["samples"] == 0 and out["sm_mhz"] is None and out["reasons"] == []

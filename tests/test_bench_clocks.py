"""bench.py's clock sampler on CPU: the NVML polling loop against a fake
library (read-only calls only), and the summary the bench line carries."""
import threading

import bench


class _FakeNvml:
    """Answers the three read-only queries the sampler makes."""

    def __init__(self, clocks, reasons):
        self.clocks = list(clocks)
        self.reasons = list(reasons)
        self.i = 0
        self.shutdown = False
        self.done = threading.Event()

    def nvmlDeviceGetClockInfo(self, h, kind, ref):
        assert kind == 1   # SM clock
        ref._obj.value = self.clocks[min(self.i, len(self.clocks) - 1)]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, ref):
        ref._obj.value = self.reasons[min(self.i, len(self.reasons) - 1)]
        self.i += 1
        if self.i >= len(self.clocks):
            self.done.set()
        return 0

    def nvmlShutdown(self):
        self.shutdown = True
        return 0


def test_nvml_loop_collects_clocks_and_reasons():
    fake = _FakeNvml([2070, 2070, 1537, 2070], [0, 0x4, 0x4 | 0x40, 0])
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.period_s = 0.001
    cs.samples = []
    cs._stop = threading.Event()
    t = threading.Thread(target=cs._nvml_loop,
                         args=(fake, None, fake.nvmlDeviceGetCurrentClocksEventReasons))
    t.start()
    assert fake.done.wait(10)
    cs._stop.set()
    t.join(10)
    assert fake.shutdown
    assert [x for x, _ in cs.samples[:4]] == [2070.0, 2070.0, 1537.0, 2070.0]
    assert cs.samples[1][1] == ["sw_power_cap"]
    assert cs.samples[2][1] == ["sw_power_cap", "hw_thermal_slowdown"]
    s = bench.ClockSampler.summary(cs.samples[:4], 2070.0, "nvml", "00000000:41:00.0")
    assert s["sm_mhz"] == 2070.0 and s["sm_mhz_min"] == 1537.0 and s["samples"] == 4
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert s["gpu_pci"] == "00000000:41:00.0"


def test_summary_without_samples():
    assert bench.ClockSampler.summary([], None, "nvml", None) is None

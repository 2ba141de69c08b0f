"""Host logic of the benchmark's clock record: the NVML clock-event reason bits
map to the names nvidia-smi prints, and the summary takes the median SM clock
and the union of the reasons seen.  No GPU and no NVML are needed."""
import sys

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reason_bits():
    assert bench.nvml_reason_names(0) == []
    assert bench.nvml_reason_names(0x1) == []            # idle: not a throttle
    assert bench.nvml_reason_names(0x4) == ["sw_power_cap"]
    assert bench.nvml_reason_names(0x8) == ["hw_slowdown"]
    assert bench.nvml_reason_names(0x80) == ["hw_slowdown"]  # power brake
    assert bench.nvml_reason_names(0x40 | 0x20) == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.nvml_reason_names(0x1FF) == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                                              "sw_thermal_slowdown"]


def test_summary():
    s = bench.clock_summary([(2070.0, 2070.0, []), (1980.0, 2070.0, ["sw_power_cap"]),
                             (2070.0, 2070.0, [])], "nvml")
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "source": "nvml"}
    e = bench.clock_summary([], None)
    assert e["reasons"] == ["unsampled"] and e["samples"] == 0


def test_sampler_keeps_only_the_marked_window():
    class FakeNvml:
        max_mhz = 2070.0

        def __init__(self):
            self.n = 0

        def read(self):
            self.n += 1
            return 1500.0 + self.n, 0x4

    c = bench.Clocks(0)
    c.nvml = FakeNvml()
    c.stop = False
    import threading
    import time
    t = threading.Thread(target=c._poll, daemon=True)
    t.start()
    time.sleep(0.02)
    assert c.samples == []          # nothing before begin()
    c.begin()
    time.sleep(0.02)
    c.end()
    n = len(c.samples)
    time.sleep(0.02)
    c.stop = True
    t.join(timeout=2)
    assert n > 0 and len(c.samples) <= n + 1
    assert all(s[2] == ["sw_power_cap"] and s[1] == 2070.0 for s in c.samples)


def test_nvidia_smi_fallback_parses_its_lines():
    class FakeProc:
        stdout = iter(["2070, 2070, Not Active, Not Active, Not Active, Not Active\n",
                       "1965, 2070, Not Active, Not Active, Not Active, Active\n",
                       "garbage\n",
                       "[N/A], 2070, Not Active, Not Active, Not Active, Not Active\n",
                       "2070, 2070, Active, Not Active, Not Active, Not Active\n"])

    c = bench.Clocks(0)
    c.proc = FakeProc()
    c._read()
    s = bench.clock_summary(c.samples, "nvidia-smi")
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]

"""bench.py's clock sampler against a fake NVML (CPU only): only the samples
taken inside the timed window count, the clock event reasons are decoded from
their bits, the device is found by UUID (else by index), and a missing NVML
is reported instead of raising."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class FakeNvml:
    """Answers like NVML: return code 0 and the value through the pointer.
    Inside [hot0, hot1] the GPU reads as loaded (1980 MHz, power cap active,
    700 W), outside it as idle and hot (345 MHz, thermal slowdown, 90 W)."""

    def __init__(self, hot0, hot1, uuid=b"GPU-fake"):
        self.hot0, self.hot1, self.uuid = hot0, hot1, uuid
        self.open = 0
        self.handles = []

    def _hot(self):
        return self.hot0 <= time.perf_counter() <= self.hot1

    def nvmlInit_v2(self):
        self.open += 1
        return 0

    def nvmlShutdown(self):
        self.open -= 1
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ph):
        if uuid != self.uuid:
            return 13  # not found
        ph._obj.value = 0x1000
        self.handles.append("uuid")
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, index, ph):
        ph._obj.value = 0x2000 + index.value
        self.handles.append("index")
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, p):
        p._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, p):
        assert kind.value == bench.NVML_CLOCK_SM
        p._obj.value = 1980 if self._hot() else 345
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, p):
        p._obj.value = 0x4 if self._hot() else 0x40
        return 0

    def nvmlDeviceGetPowerUsage(self, h, p):
        p._obj.value = 700000 if self._hot() else 90000
        return 0


class FakeNvmlWithDriver(FakeNvml):
    def nvmlSystemGetDriverVersion(self, buf, length):
        buf.value = b"580.159"
        return 0


def _run(lib, uuid):
    a = time.perf_counter() + 0.02
    lib.hot0, lib.hot1 = a, a + 0.08
    s = bench.NvmlSampler(uuid, 3, lib, period_s=0.0005)
    assert s.start()
    while time.perf_counter() < lib.hot1 + 0.02:
        time.sleep(0.005)
    return s.stop(lib.hot0 + 0.01, lib.hot1 - 0.01)


def test_only_samples_inside_the_window_count():
    lib = FakeNvml(0, 0)
    res = _run(lib, "GPU-fake")
    assert res["samples"] >= 10
    assert res["sm_mhz"] == 1980.0 and res["sm_max_mhz"] == 2070.0
    assert res["reasons"] == ["sw_power_cap"]          # the thermal bit was set outside only
    assert res["reason_bits_seen"] == "0x4" and res["sm_min_mhz"] == 1980.0
    assert res["power_w_max"] == 700.0
    assert lib.handles == ["uuid"] and lib.open == 0   # NVML closed again


def test_device_found_by_index_when_the_uuid_is_unknown():
    lib = FakeNvml(0, 0, uuid=b"GPU-other")
    res = _run(lib, "GPU-fake")
    assert lib.handles == ["index"] and res["sm_mhz"] == 1980.0


def test_driver_version_when_nvml_has_it():
    lib = FakeNvmlWithDriver(0, 0)
    s = bench.NvmlSampler("GPU-fake", 0, lib)
    assert s.start()
    s.stop(0.0, 0.0)
    assert s.driver == "580.159"
    s = bench.NvmlSampler("GPU-fake", 0, FakeNvml(0, 0))   # no such call: no version
    assert s.start()
    s.stop(0.0, 0.0)
    assert s.driver is None


def test_missing_nvml_is_reported_not_raised():
    assert bench.NvmlSampler("GPU-x", 0, None).start() is False

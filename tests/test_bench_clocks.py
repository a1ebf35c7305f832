"""The bench's clock samplers (CPU): NVML polling against a fake NVML, the
nvidia-smi line parser, and the summary both feed into the JSON line."""

import itertools
import time

import bench


class FakeNvml:
    """Read-only NVML calls with canned answers (return 0 = NVML_SUCCESS)."""

    def __init__(self, clocks, reasons):
        self.clocks = itertools.cycle(clocks)
        self.reasons = reasons
        self.shut = False

    def nvmlInit_v2(self):
        return 0

    def nvmlShutdown(self):
        self.shut = True
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        return 13  # NVML_ERROR_NOT_FOUND: fall back to the index

    def nvmlDeviceGetHandleByIndex_v2(self, index, ref):
        ref._obj.value = 4096 + index.value
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, kind, ref):
        assert kind.value == 1  # NVML_CLOCK_SM
        ref._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, handle, kind, ref):
        assert kind.value == 1
        ref._obj.value = next(self.clocks)
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle, ref):
        ref._obj.value = self.reasons
        return 0


class Dev:
    index = 0


def _run(sampler, n=3, limit_s=5.0):
    """Run the sampler until it has n samples (or limit_s passes)."""
    t0 = time.perf_counter()
    with sampler:
        while len(sampler.samples) < n and time.perf_counter() - t0 < limit_s:
            time.sleep(0.005)
    return sampler.summary()


def test_nvml_sampler_median_and_reasons():
    fake = FakeNvml([2070, 2070, 1980], 0x1 | 0x4)  # GPU idle (ignored) + SW power cap
    out = _run(bench.NvmlClockSampler(Dev(), period_s=0.001, lib=fake))
    assert fake.shut
    assert out["samples"] >= 3 and out["source"] == "nvml"
    assert out["sm_max_mhz"] == 2070
    assert out["sm_mhz"] in (2070, 1980)
    assert out["reasons"] == ["sw_power_cap"]


def test_nvml_sampler_throttle_bits():
    fake = FakeNvml([1200], 0x8 | 0x20 | 0x40)
    out = _run(bench.NvmlClockSampler(Dev(), period_s=0.001, lib=fake), n=1)
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_nvml_sampler_poll_from_the_caller():
    """A short timed region samples from the waiting thread too: each poll adds
    one sample, whatever the sampling thread has done."""
    fake = FakeNvml([2070, 1980], 0x4)
    s = bench.NvmlClockSampler(Dev(), period_s=10.0, lib=fake)  # the thread samples once
    with s:
        n0 = len(s.samples)
        for _ in range(4):
            s.poll()
        assert len(s.samples) >= n0 + 4
    out = s.summary()
    assert out["samples"] >= 4 and out["reasons"] == ["sw_power_cap"]
    bench.ClockSampler(0).poll()  # nvidia-smi samples on its own; poll is a no-op


def test_nvidia_smi_parser_and_empty_summary():
    c = bench.ClockSampler(0)
    c.lines = ["2070, 2070, Not Active, Not Active, Not Active, Active",
               "1995, 2070, Active, Not Active, Not Active, Not Active",
               "[N/A], 2070, Not Active, Not Active, Not Active, Not Active",
               "garbled"]
    out = c.summary()
    assert out["samples"] == 2 and out["source"] == "nvidia-smi"
    assert out["sm_mhz"] == (2070 + 1995) / 2 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.clock_summary([], "nvml")["sm_mhz"] is None

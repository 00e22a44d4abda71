"""bench.py's clock record on CPU, with a stand-in for the NVML reader: the
samples taken while the timed region runs give the median SM clock, the
maximum, the sample count, and the clock-event reasons that the timing rules
watch, by name.  Needs no GPU."""
import time

import bench


class FakeNvml:
    """Returns a fixed list of (SM MHz, reason bits) samples, then repeats the
    last one."""

    def __init__(self, samples, max_mhz=2070):
        self.samples = list(samples)
        self.max_mhz = max_mhz
        self.closed = False

    def sample(self):
        return self.samples.pop(0) if len(self.samples) > 1 else self.samples[0]

    def max_sm(self):
        return self.max_mhz

    def close(self):
        self.closed = True


def run_sampler(monkeypatch, samples, hold_s=0.01):
    fake = FakeNvml(samples)
    monkeypatch.setattr(bench, "_Nvml", lambda index: fake)
    with bench.ClockSampler(0) as c:
        time.sleep(hold_s)
    return c.summary(), fake


def test_clean_run_has_no_reasons(monkeypatch):
    s, fake = run_sampler(monkeypatch, [(2070, 0x0), (2070, 0x1), (2070, 0x0)])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["samples"] >= 3  # one before, the loop's, one after
    assert s["reasons"] == []  # GPU idle (bit 0) is not a throttle reason
    assert fake.closed


def test_reason_bits_are_named(monkeypatch):
    # nvml.h clock-event reasons: sw power cap 0x4, hw slowdown 0x8,
    # sw thermal 0x20, hw thermal 0x40; sync boost 0x10 is not watched
    s, _ = run_sampler(monkeypatch, [(1800, 0x4), (1900, 0x8 | 0x10), (2000, 0x20), (2070, 0x40)])
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert 1800.0 <= s["sm_mhz"] <= 2070.0


def test_median_of_the_samples(monkeypatch):
    s, _ = run_sampler(monkeypatch, [(1000, 0), (2000, 0), (2000, 0)], hold_s=0.0)
    assert s["sm_mhz"] == 2000.0


def test_falls_back_when_nvml_cannot_load(monkeypatch):
    def no_nvml(index):
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")

    monkeypatch.setattr(bench, "_Nvml", no_nvml)
    with bench.ClockSampler(0) as c:
        pass
    s = c.summary()
    # no GPU here: nvidia-smi is absent or prints nothing, so no record at all
    assert s is None or s["source"].startswith("nvidia-smi")

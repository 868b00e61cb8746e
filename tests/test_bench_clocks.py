"""bench.py's clock record (no GPU): the nvidia-smi CSV sampled during the
timed region is reduced to the median SM clock under load, the maximum
clock and the throttle reasons that were active at any sample."""
import bench


class FakeSmi:
    def __init__(self, text):
        self.text = text
        self.terminated = False

    def terminate(self):
        self.terminated = True

    def communicate(self, timeout=None):
        return self.text, ""


def sampler(text):
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.p = FakeSmi(text)
    return c


def test_median_max_and_reasons():
    csv = "\n".join([
        "0, 1965, 2070, 850.10, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1210.55, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1190.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    c = sampler(csv)
    r = c.stop()
    assert c.p.terminated
    assert r["sm_mhz"] == 2010.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3


def test_hardware_slowdown_is_reported():
    csv = "0, 1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active\n"
    r = sampler(csv).stop()
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_no_nvidia_smi():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.p = None
    r = c.stop()
    assert r["sm_mhz"] is None and r["reasons"] == ["nvidia-smi unavailable"]


def test_clocks_rejected():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clocks_rejected(ok) is None
    assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"], sm_mhz=1500.0)) is None
    assert bench.clocks_rejected(dict(ok, reasons=["hw_thermal_slowdown"])) == "throttled: hw_thermal_slowdown"
    assert "with no reason" in bench.clocks_rejected(dict(ok, sm_mhz=1200.0))
    # nvidia-smi missing: nothing to judge by
    assert bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}) is None

"""Host-side helpers of bench.py (no GPU): the source fingerprint that keys the recorded
DRAM-traffic capture to the kernel code it was taken on, and the NVML clock record (driven
by a fake NVML library that answers queries from a script)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("// a comment\nint f(int x) {  // trailing note\n\n  return x + 1;\n}\n\n")
    assert b.code_hash(str(a)) == b.code_hash(str(c))


def test_code_hash_sees_code_changes(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert b.code_hash(str(a)) != b.code_hash(str(c))


def test_traffic_only_for_the_captured_batch():
    b = _bench()
    # the capture holds for the benchmark batch only; any other T reports no traffic
    assert b.traffic_per_launch(4096) is None
    assert b.traffic_per_launch(b.TRAFFIC_CAPTURE["T"]) in (None, b.TRAFFIC_CAPTURE["bytes"])


class FakeNvml:
    """Answers the NVML queries the sampler makes; records the UUID it was asked for.
    Every query fills the output argument through its ctypes reference."""

    def __init__(self, clocks, powers_mw, reasons, max_mhz=2070, uuids=("GPU-abc",)):
        self.clocks, self.powers, self.reasons = list(clocks), list(powers_mw), list(reasons)
        self.i = 0
        self.max_mhz = max_mhz
        self.uuids = uuids
        self.asked_uuid = None
        self.shutdown = False
        self.settings_changed = False      # no setter is ever called

    @staticmethod
    def _set(ref, v):
        ref._obj.value = v

    def nvmlInit_v2(self):
        return 0

    def nvmlShutdown(self):
        self.shutdown = True
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        self.asked_uuid = uuid.decode()
        return 0 if self.asked_uuid in self.uuids else 13

    def nvmlDeviceGetCount_v2(self, ref):
        self._set(ref, 1)
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, i, ref):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, kind, ref):
        assert kind == 1                    # NVML_CLOCK_SM
        self._set(ref, self.max_mhz)
        return 0

    def _next(self, seq):
        return seq[min(self.i, len(seq) - 1)]

    def nvmlDeviceGetClockInfo(self, dev, kind, ref):
        assert kind == 1
        self._set(ref, self._next(self.clocks))
        return 0

    def nvmlDeviceGetPowerUsage(self, dev, ref):
        self._set(ref, self._next(self.powers))
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, ref):
        self._set(ref, self._next(self.reasons))
        self.i += 1                         # one sample = clock, power, reasons
        return 0


def test_nvml_sampler_summary_from_fake_queries():
    import time
    b = _bench()
    fake = FakeNvml(clocks=[1500, 1560, 1620, 1580, 1510], powers_mw=[900000, 1200000, 1300000],
                    reasons=[0x0, 0x4, 0x4, 0x0, 0x0])
    s = b.NvmlSampler("abc", period_s=0.002, lib=fake)      # torch's uuid has no "GPU-"
    assert s.ok and fake.asked_uuid == "GPU-abc"
    time.sleep(0.05)
    rec = s.stop()
    assert fake.shutdown and not fake.settings_changed
    assert rec["source"] == "nvml" and rec["samples"] >= 5
    assert rec["samples_under_load"] == rec["samples"]
    assert sum(rec["sm_mhz_bins"].values()) == rec["samples"]
    assert set(rec["sm_mhz_bins"]) <= {"1500-1599", "1600-1699"}
    assert rec["sm_max_mhz"] == 2070 and rec["sm_mhz_min"] == 1500
    assert rec["reasons"] == ["sw_power_cap"]
    assert rec["power_w_max"] == 1300.0


def test_nvml_reason_bits_and_unknown_device():
    b = _bench()
    rows = [dict(t=0.0, sm=1400.0, power=500.0, reasons=0x8 | 0x20),
            dict(t=0.01, sm=1450.0, power=600.0, reasons=0x40 | 0x80)]
    rec = b.NvmlSampler.summarize(rows, 2070.0, 0.01)
    assert rec["reasons"] == ["hw_power_brake_slowdown", "hw_slowdown", "hw_thermal_slowdown",
                              "sw_thermal_slowdown"]
    assert rec["sm_mhz"] == 1425.0 and rec["sm_mhz_bins"] == {"1400-1499": 2}
    assert b.NvmlSampler.summarize([], 2070.0, 0.01) is None
    # a UUID NVML does not know, with several GPUs visible: no sampler (nvidia-smi is used)
    fake = FakeNvml([1500], [100000], [0], uuids=("GPU-other",))
    fake.nvmlDeviceGetCount_v2 = lambda ref: (FakeNvml._set(ref, 4), 0)[1]
    s = b.NvmlSampler("abc", lib=fake)
    assert not s.ok and fake.shutdown

"""The bench's clock record: NVML is sampled from a background thread every millisecond while
the timed region runs. The main thread enqueues the timed calls in Python and holds the
interpreter lock between them, so the sampler must still get its turns over a region of a
few milliseconds. NVML is replaced by a fake here (CPU only)."""
import sys
import time

import bench


class _FakeNVML:
    def nvmlDeviceGetClockInfo(self, handle, kind, ref):
        ref._obj.value = 2070
        return 0

    def nvmlDeviceGetPowerUsage(self, handle, ref):
        ref._obj.value = 500000
        return 0

    def nvmlShutdown(self):
        return 0


def _fake_open(self):
    self.nvml, self.handle, self.max_mhz = _FakeNVML(), None, 2070
    self.reasons_fn = lambda handle, ref: 0
    return True


def test_sampler_gets_turns_while_the_main_thread_is_busy(monkeypatch):
    monkeypatch.setattr(bench.ClockSampler, "_open_nvml", _fake_open)
    before = sys.getswitchinterval()
    with bench.ClockSampler(device=None) as cs:
        end = time.perf_counter() + 0.05
        n = 0
        while time.perf_counter() < end:  # pure Python: holds the interpreter lock
            n += 1
        cs.mark()
    s = cs.summary()
    # 50 ms at one sample a millisecond; the default 5 ms switch interval allows about 10
    assert s["samples"] >= 20, s
    assert s["sync_samples"] == 1 and s["sm_mhz"] == 2070 and s["reasons"] == []
    assert sys.getswitchinterval() == before  # restored on exit

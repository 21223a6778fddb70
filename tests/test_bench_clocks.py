"""The bench's clock record (CPU): the nvidia-smi sampler parsed from a fake
process that prints lines in nvidia-smi's csv format, so no GPU is needed."""
import os
import threading
import time

import bench


class FakeSmi:
    """Prints one csv line every 20 ms until terminated.  Line i reports
    `sm(i)` MHz and, when `cap(i)`, sw_power_cap active."""

    def __init__(self, sm, cap):
        r, w = os.pipe()
        self.stdout = os.fdopen(r, "r")
        self._w = os.fdopen(w, "w")
        self._stop = threading.Event()
        self._rc = None

        def run():
            i = 0
            while not self._stop.is_set():
                reason = "Active" if cap(i) else "Not Active"
                self._w.write(f"0, {sm(i)}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {reason}\n")
                self._w.flush()
                i += 1
                time.sleep(0.02)
            self._w.close()

        self._t = threading.Thread(target=run, daemon=True)
        self._t.start()

    def poll(self):
        return self._rc

    def terminate(self):
        self._stop.set()
        self._rc = 0

    def wait(self, timeout=None):
        self._t.join(timeout)
        return 0

    def kill(self):
        self.terminate()


def run_sampler(monkeypatch, sm, cap, before=0.2, region=0.2, after=0.2):
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: FakeSmi(sm, cap))
    with bench.ClockSampler(0) as clk:
        time.sleep(before)
        clk.mark_start()
        time.sleep(region)
        clk.mark_end()
        time.sleep(after)
    return clk.summary()


def test_clock_summary_under_load(monkeypatch):
    s = run_sampler(monkeypatch, sm=lambda i: 1980 if i % 4 == 0 else 2070, cap=lambda i: i == 3)
    assert s["sm_mhz"] == 2070 and s["sm_min_mhz"] == 1980 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] >= 10
    # about region / 20 ms lines fall inside the marked region
    assert 3 <= s["samples_in_timed_region"] <= s["samples"]


def test_clock_summary_without_nvidia_smi(monkeypatch):
    def missing(*a, **k):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", missing)
    with bench.ClockSampler(0) as clk:
        pass
    assert clk.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}

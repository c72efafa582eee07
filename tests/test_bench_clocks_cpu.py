"""bench.py's clock record: nvidia-smi samples are kept only when they fall
inside the timed window, throttle reasons are collected from those samples,
and with no sample inside the window every sample counts (flagged)."""

import datetime
import time

import bench


class _FakeSmi:
    """Stands in for the nvidia-smi subprocess: lines at given offsets (s) from now."""

    def __init__(self, rows):
        now = datetime.datetime.now()
        self.out = "\n".join(
            f"{(now + datetime.timedelta(seconds=dt)).strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, "
            f"{mhz}, 2032, 700.0, 0x0, {hw}, Not Active, Not Active, {cap}"
            for dt, mhz, hw, cap in rows)

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _sampler(rows):
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi(rows)
    return s


def test_only_samples_inside_the_window_count():
    rows = [(-0.30, 1000, "Not Active", "Not Active"),   # idle, before the window
            (0.01, 1965, "Not Active", "Active"),
            (0.02, 1965, "Not Active", "Active"),
            (0.50, 1200, "Active", "Not Active")]        # after the window
    t = time.time()
    c = _sampler(rows).stop(t, t + 0.1)
    assert c["in_timed_window"] and c["samples"] == 2
    assert c["sm_mhz"] == 1965.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside


def test_no_sample_inside_uses_all_and_says_so():
    rows = [(-0.30, 1000, "Not Active", "Not Active"), (0.50, 2032, "Active", "Not Active")]
    t = time.time()
    c = _sampler(rows).stop(t, t + 0.1)
    assert not c["in_timed_window"] and c["samples"] == 2
    assert c["reasons"] == ["hw_slowdown"]


def test_unavailable_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop(0.0, 1.0)["reasons"] == ["nvidia-smi unavailable"]

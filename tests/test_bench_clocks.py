"""bench.py's clock summary on CPU, from a sample file written as the NVML
sampling process writes it ("max MHz" first, then "monotonic_s mhz watts
reasons" lines): the median and the throttle reasons over the timed region,
and the nearest samples when the region is too short to hold enough."""

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _summary(tmp_path, samples, t_start, t_end):
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.period, c.error = 0.0002, None
    c.path = str(tmp_path / "clocks.txt")
    c.proc = _Done()
    c.t_start, c.t_end = t_start, t_end
    with open(c.path, "w") as f:
        f.write("max 2070\n")
        for t, mhz, w, r in samples:
            f.write("%.6f %d %.3f %d\n" % (t, mhz, w, r))
    return c.stop()


def test_samples_inside_the_region(tmp_path):
    power_cap = [bit for bit, name in bench.CLOCK_REASONS if name == "sw_power_cap"][0]
    s = [(10.0 + 0.001 * i, 2070 if i != 12 else 1900, 900.0, power_cap if i == 13 else 0)
         for i in range(30)]
    r = _summary(tmp_path, s, 10.0095, 10.0205)  # samples 10..20
    assert r["samples"] == 11
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]
    assert r["basis"] == "the samples inside the timed region"


def test_short_region_takes_the_nearest_samples(tmp_path):
    slow = [bit for bit, name in bench.CLOCK_REASONS if name == "hw_slowdown"][0]
    # one read every 4 ms; a 2 ms region between two reads; the throttled
    # sample far from the region is not taken
    s = [(100.0 + 0.004 * i, 1500 if i == 0 else 2070, 800.0, slow if i == 0 else 0) for i in range(12)]
    r = _summary(tmp_path, s, 100.0205, 100.0225)
    assert r["samples"] == 0
    assert r["sm_mhz"] == 2070 and r["reasons"] == []
    assert r["basis"].startswith("0 samples inside the timed region; the 5 nearest")
    # a throttled sample right next to the region is reported
    s[5] = (s[5][0], 1600, 800.0, slow)
    r = _summary(tmp_path, s, 100.0205, 100.0225)
    assert r["reasons"] == ["hw_slowdown"]

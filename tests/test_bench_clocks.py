"""The bench's clock record on the CPU: nvidia-smi sample lines parsed and
summarised per timed window (no GPU, no nvidia-smi)."""
import bench

LINES = [
    # timestamp, index, sm, max sm, power, util, active, hw, hwt, swt, pcap
    "2026/12/02 10:00:00.000, 0, 2070, 2070, 900.5, 100, 0x0, Not Active, Not Active, Not Active, Not Active",
    "2026/12/02 10:00:00.050, 0, 2070, 2070, 1010.0, 100, 0x0, Not Active, Not Active, Not Active, Not Active",
    "2026/12/02 10:00:00.100, 0, 1905, 2070, 1395.0, 100, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/02 10:00:00.150, 0, 1890, 2070, 1398.0, 100, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/02 10:00:00.200, 0, 345, 2070, 120.0, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    "garbage line",
]


def rows_from(lines, tmp_path):
    s = bench.ClockSampler()
    f = tmp_path / "clocks.csv"
    f.write_text("\n".join(lines) + "\n")
    s.file = open(f, "a+")

    class Done:  # the sampler process, already ended
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = Done()
    return s.stop()


def test_windows_split_the_samples(tmp_path):
    rows = rows_from(LINES, tmp_path)
    assert len(rows) == 5
    t = [r["t"] for r in rows]
    first = bench.ClockSampler.summary(rows, (t[0], t[1]))
    assert first["sm_mhz"] == 2070 and first["reasons"] == [] and first["samples"] == 2
    assert abs(first["power_w_1s_mean"] - 955.25) < 1e-9
    second = bench.ClockSampler.summary(rows, (t[2], t[4]))
    # the idle sample (utilisation 0) is left out of the median and the reasons
    assert second["samples"] == 2 and second["sm_mhz"] == 1897.5
    assert second["reasons"] == ["sw_power_cap"]
    whole = bench.ClockSampler.summary(rows)
    assert whole["samples"] == 4 and whole["sm_max_mhz"] == 2070


def test_no_sampler_and_empty_window(tmp_path):
    none = bench.ClockSampler.summary(None, (0, 1))
    assert none["sm_mhz"] is None and none["reasons"] == ["nvidia-smi unavailable"]
    rows = rows_from(LINES[:2], tmp_path)
    # a window with no sample falls back to every sample taken
    far = bench.ClockSampler.summary(rows, (0.0, 1.0))
    assert far["samples"] == 2
    assert bench.ClockSampler.summary([], None)["reasons"] == ["no samples"]

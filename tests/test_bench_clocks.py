"""The benchmark's clock record (host logic, no GPU): which nvidia-smi samples it uses and
which throttle reasons it reports."""
import bench


def _sampler(tmp_path, lines, t0, t1):
    p = tmp_path / "clocks.csv"
    p.write_text("".join(lines))
    s = bench.ClockSampler(0)
    s.proc = object()  # as if nvidia-smi ran
    s.path = str(p)
    s.t0, s.t1 = t0, t1
    return s


def _line(sec, mhz, hw="Not Active", power_cap="Not Active"):
    # timestamp, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"2026/01/01 00:00:{sec:06.3f}, {mhz}, 2070, 500.0, 0x0, {hw}, Not Active, Not Active, {power_cap}\n"


def _ts(sec):
    import datetime
    return datetime.datetime.strptime(f"2026/01/01 00:00:{sec:06.3f}", "%Y/%m/%d %H:%M:%S.%f").timestamp()


def test_samples_inside_the_region_are_used(tmp_path):
    lines = [_line(1.0, 1500), _line(2.0, 2070), _line(2.1, 2070), _line(3.0, 1000)]
    s = _sampler(tmp_path, lines, _ts(1.5), _ts(2.5))
    out = s.summary()
    assert out["samples_in_region"] == 2 and out["samples_used"] == 2
    assert out["sm_mhz"] == 2070 and out["reasons"] == [] and "note" not in out


def test_a_short_region_uses_the_nearest_sample_on_each_side(tmp_path):
    lines = [_line(1.0, 1500), _line(2.0, 2060), _line(2.2, 2070), _line(3.0, 1000)]
    s = _sampler(tmp_path, lines, _ts(2.05), _ts(2.1))
    out = s.summary()
    assert out["samples_in_region"] == 0 and out["samples_used"] == 2
    assert out["sm_mhz"] == (2060 + 2070) / 2
    assert "shorter than the 100 ms sampling period" in out["note"]


def test_throttle_reasons_are_reported(tmp_path):
    lines = [_line(2.0, 1800, hw="Active"), _line(2.1, 1900, power_cap="Active")]
    s = _sampler(tmp_path, lines, _ts(1.9), _ts(2.2))
    out = s.summary()
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_weak_scaling_rate_counts_every_rank():
    assert bench.weak_scaling_rate(1000, 10, 4, 2.0) == 1000 * 10 * 4 / 2.0

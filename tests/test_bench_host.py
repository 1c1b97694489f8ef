"""Host logic of bench.py that needs no GPU: the clock record's reading of
nvidia-smi samples (only samples taken inside the timed region count, the
throttle reasons that reject a run are picked up) and its behaviour when
nvidia-smi is missing."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, mx=2070, hw="Not Active", therm="Not Active", sw_therm="Not Active", cap="Not Active"):
    return f"{sm}, {mx}, 900.5, 0x0000000000000000, {hw}, {therm}, {sw_therm}, {cap}"


def test_only_samples_inside_the_region_count():
    cs = bench.ClockSampler(0)
    cs.lines = [_line(1200, hw="Active"), _line(2070), _line(2040, cap="Active"), _line(2055)]
    cs.start = 1          # the first sample came in before the region began
    s = cs.summary()
    assert s["samples"] == 3 and s["samples_in_region"] == 3
    assert s["sm_mhz"] == 2055 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]          # the pre-region hw_slowdown is not counted


def test_rejecting_reasons_are_reported():
    cs = bench.ClockSampler(0)
    cs.lines = [_line(1900, therm="Active"), _line(1890, sw_therm="Active")]
    s = cs.summary()
    assert set(s["reasons"]) == {"hw_thermal_slowdown", "sw_thermal_slowdown"}
    assert any(r in s["reasons"] for r in bench.BAD_REASONS)


def test_short_region_uses_the_last_sample_before_it():
    cs = bench.ClockSampler(0)
    cs.lines = [_line(1500), _line(2070)]
    cs.start = 2          # no sample arrived during the region
    s = cs.summary()
    assert s["samples_in_region"] == 0 and s["samples"] == 1 and s["sm_mhz"] == 2070


def test_malformed_lines_are_skipped_and_missing_tool_gives_nulls(monkeypatch):
    cs = bench.ClockSampler(0)
    cs.lines = ["[N/A], [N/A]", "garbage", _line(2000)]
    assert cs.summary()["samples"] == 1

    def no_tool(*a, **k):
        raise FileNotFoundError("nvidia-smi")
    monkeypatch.setattr(bench.subprocess, "Popen", no_tool)
    with bench.ClockSampler(0) as cs2:
        pass
    s = cs2.summary()
    assert s["sm_mhz"] is None and s["samples"] == 0


def test_reference_arm_line(capsys, monkeypatch):
    """The reference arm (the fp64 oracle on the host cores) prints one JSON
    line with the contract's keys; under a launcher only rank 0 prints."""
    import json
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "0", "--workload", "tiny",
                "--cpu-budget", "0.01"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny",
                "--cpu-budget", "0.01"])
    assert capsys.readouterr().out.strip() == ""

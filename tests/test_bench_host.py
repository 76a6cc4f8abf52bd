"""Host logic of bench.py that needs no GPU (not marked gpu).

* ClockSampler.stop() turns nvidia-smi's CSV samples into the line's
  `clocks` object: the median SM clock, the maximum, and every throttle
  reason seen active (the timing rules reject a run with a thermal or
  hardware slowdown, so a dropped reason would hide a rejected number).
* ncu_traffic() hands out a committed DRAM-traffic figure only while the
  kernel's source is the one the counters were taken on: a figure from
  another source must read as null.
"""
import json
import os

import bench


def _fake_sampler(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(l + "\n" for l in lines))

    class _Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs = bench.ClockSampler(0)
    cs.path = str(path)
    cs.proc = _Proc()
    cs.f = open(os.devnull, "w")
    return cs


def _row(sm, mx=2032, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, active reasons mask, then
    # the four reasons, in the order of bench.CLOCK_FIELDS
    return f"0, {sm}, {mx}, 900.0, 0x0, {hw}, {hwt}, {swt}, {cap}"


def test_clock_fields_order_matches_the_parser():
    fields = bench.CLOCK_FIELDS.split(",")
    assert fields[1] == "clocks.sm" and fields[2] == "clocks.max.sm"
    assert fields[5:9] == ["clocks_event_reasons.hw_slowdown",
                           "clocks_event_reasons.hw_thermal_slowdown",
                           "clocks_event_reasons.sw_thermal_slowdown",
                           "clocks_event_reasons.sw_power_cap"]


def test_clock_median_and_no_reason(tmp_path):
    cs = _fake_sampler(tmp_path, [_row(2032), _row(1995), _row(2032), _row(2032), _row(1800)])
    c = cs.stop()
    assert c == {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": [], "samples": 5}
    assert not os.path.exists(cs.path)


def test_clock_reasons_are_collected(tmp_path):
    cs = _fake_sampler(tmp_path, [_row(1875, cap="Active"), _row(1500, hwt="Active"),
                                  _row(2032), "garbage line", _row("[N/A]")])
    c = cs.stop()
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert c["samples"] == 3 and c["sm_mhz"] == 1875.0


def test_clock_without_samples(tmp_path):
    c = _fake_sampler(tmp_path, []).stop()
    assert c["sm_mhz"] is None and c["samples"] == 0


def test_traffic_only_for_the_source_it_was_measured_on(tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_verify_accept_step_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("// kernel source, first version\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.source_hash("k.cu")
    entry = {"k.cu": {"wl": {"bytes_per_launch": 1.25e9, "source_sha": sha}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entry))
    assert bench.ncu_traffic("k.cu", "wl") == 1.25e9
    assert bench.ncu_traffic("k.cu", "other workload") is None
    (csrc / "k.cu").write_text("// kernel source, changed since the capture\n")
    assert bench.ncu_traffic("k.cu", "wl") is None


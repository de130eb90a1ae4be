"""bench.py's host logic on the CPU: the clock record of a timed region and
the check that disqualifies it, and the lookup of committed ncu traffic by
source hash."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s.summary()


# index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
def test_clock_summary_parses_nvidia_smi_lines():
    lines = ["0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 2055, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    s = _sampler(lines)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    assert bench.clocks_ok(s)            # a power cap alone is kept


def test_clock_summary_empty():
    assert _sampler([]) is None
    assert bench.clocks_ok(None)         # no nvidia-smi: nothing to judge


def test_throttle_disqualifies():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        s = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [r], "samples": 5}
        assert not bench.clocks_ok(s), r
    line = "0, 1500, 2070, 700.0, 0x8, Not Active, Active, Not Active, Not Active"
    assert not bench.clocks_ok(_sampler([line] * 4))


def test_clock_lock_without_reason_disqualifies():
    locked = {"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9}
    assert not bench.clocks_ok(locked)
    capped = dict(locked, reasons=["sw_power_cap"])
    assert bench.clocks_ok(capped)       # below max for a stated reason: kept
    near = dict(locked, sm_mhz=1950.0)
    assert bench.clocks_ok(near)


def test_recorded_traffic_keys_on_source_hash(tmp_path, monkeypatch):
    sha = bench.source_sha("stage1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(
        "# kernel workload sha bytes\n"
        f"stage1 fp8_decode {sha} 1234\n"
        "stage1 mla_fp8 000000000000 99\n")
    csrc = tmp_path / "paged_split_kv_03_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["stage1"]:
        src = os.path.join(ROOT, "paged_split_kv_03_gb300", "csrc", f)
        (csrc / f).write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("stage1", "fp8_decode") == 1234
    assert bench.recorded_traffic("stage1", "mla_fp8") is None       # other sources
    assert bench.recorded_traffic("stage1", "mixed") is None          # never captured
    (csrc / "pda_tc.cu").write_bytes(b"// changed\n" + (csrc / "pda_tc.cu").read_bytes())
    assert bench.recorded_traffic("stage1", "fp8_decode") is None     # kernel changed since


def test_parse_workload():
    assert bench.parse_workload(bench.HEADLINE)[:2] == (bench.HEADLINE, {})
    name, kw, desc = bench.parse_workload("longctx_fp8_pth:bs=16,R=8")
    assert (name, kw) == ("longctx_fp8_pth", {"bs": 16, "R": 8})
    name, kw, _ = bench.parse_workload("fp8_decode:layout=HND")
    assert kw == {"layout": "HND"}
    from paged_split_kv_03_gb300.synth import config_workload
    wl = config_workload("tiny", **kw)
    assert wl.layout == "HND"


def test_step_stats():
    st = bench.step_stats([0.1, 0.2, 0.3, 0.4, 10.0, 0.25, 0.15, 0.35])
    # sorted: .1 .15 .2 .25 .3 .35 .4 10 -> middle half .2 .25 .3 .35
    assert abs(st["us_median"] - 275.0) < 1e-9
    assert abs(st["us_iqm"] - 275.0) < 1e-9
    one = bench.step_stats([0.5])
    assert one == {"us_median": 500.0, "us_iqm": 500.0}
    three = bench.step_stats([0.3, 0.1, 0.2])
    assert abs(three["us_iqm"] - 200.0) < 1e-9 and abs(three["us_median"] - 200.0) < 1e-9

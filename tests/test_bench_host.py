"""Host logic of bench.py that feeds its JSON line (no GPU): the clock record parsed from
nvidia-smi's CSV samples, and the DRAM-traffic lookup from the profile summaries."""

import bench


def test_clock_summary_takes_the_median_and_collects_active_throttle_reasons():
    c = bench.ClockSampler(0)
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    c.lines = [
        "0, 1650, 2032, 900.1, 0x0004, Not Active, Not Active, Not Active, Active",
        "0, 1700, 2032, 950.0, 0x0000, Not Active, Not Active, Not Active, Not Active",
        "0, 1600, 2032, 1010.5, 0x0004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2032, 10, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 1650.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    c.lines = ["0, 1200, 2032, 500, 0x0, Active, Not Active, Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_reports_none():
    c = bench.ClockSampler(0)
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_record_matches_the_source_hash_and_scales_by_units(tmp_path, monkeypatch):
    src = tmp_path / "csrc"
    src.mkdir()
    (src / "a.cuh").write_text("kernel source one\n")
    (src / "b.cuh").write_text("kernel source two\n")
    import hashlib
    h = hashlib.sha1()
    h.update(b"kernel source one\0")
    h.update(b"kernel source two\0")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(
        "# summary\n"
        f"traffic-record: my_kernel sha1={h.hexdigest()} dram_bytes=1000 units=10\n"
        "traffic-record: other_kernel sha1=0 dram_bytes=5 units=1\n")
    monkeypatch.setattr(bench, "CSRC", str(src))
    monkeypatch.setattr(bench, "PROFILES", str(prof))
    assert bench.traffic_per_launch("my_kernel", ["a.cuh", "b.cuh"], 25) == 2500
    # another order of the hashed files finds no record: null traffic
    assert bench.traffic_per_launch("my_kernel", ["b.cuh", "a.cuh"], 25) is None
    # comments and layout do not count, code does
    (src / "a.cuh").write_text("// a note\nkernel   source /* inline */ one\n")
    assert bench.traffic_per_launch("my_kernel", ["a.cuh", "b.cuh"], 25) == 2500
    (src / "a.cuh").write_text("kernel source one, edited\n")
    assert bench.traffic_per_launch("my_kernel", ["a.cuh", "b.cuh"], 25) is None


def test_code_text_keeps_literals_and_drops_comments():
    src = 'asm("a // b"); /* c */ int x = 1; // d\nchar q = \'/\';'
    assert bench.code_text(src) == 'asm("a // b"); int x = 1; char q = \'/\';'


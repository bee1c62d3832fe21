"""Host-side logic of bench.py that decides what a benchmark line reports: the
clock summary (throttle reasons read from nvidia-smi's CSV), the replica
rates, and the rule that DRAM traffic from a committed profile is reported
only while the kernel source it was taken on is unchanged."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_clock_summary_median_and_reasons(bench):
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    s.lines = ["0, 1500, 2070, 700, 0x8, Active, Not Active, Active, Not Active"]
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples(bench):
    out = bench.ClockSampler(0).summary()
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_replica_rates(bench):
    gbs, tps = bench.replica_rates(step_bytes=500_000_000, steps=100, total_ms=10.0, world=4)
    assert gbs == pytest.approx(4 * 500e6 * 100 / 0.01 / 1e9)
    assert tps == pytest.approx(4 * 100 / 0.01)


def test_traffic_only_while_the_source_is_unchanged(bench, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "select_accumulate_stack30.json")) as f:
        d = json.load(f)
    monkeypatch.setattr(bench, "source_hash", lambda paths: d["source_hash"])
    assert bench.committed_traffic(0) == d["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "source_hash", lambda paths: "0" * 16)
    assert bench.committed_traffic(0) is None


def test_source_hash_sees_code_not_comments(bench, monkeypatch, tmp_path):
    """The traffic record is keyed on the kernel sources' code: a comment or a
    blank line does not change the hash, a changed statement does."""
    src = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src.write_text("int f(int x) {\n    return x + 1;   // one\n}\n")
    h0 = bench.source_hash(["k.cu"])
    src.write_text("// a new header\n/* a block\n   comment */\nint f(int x) {\n\n    return x + 1;   // two\n}\n")
    assert bench.source_hash(["k.cu"]) == h0
    src.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.source_hash(["k.cu"]) != h0



def test_batch_floors(bench):
    """The floors of the path each M takes: the HBM bytes at the copy peak; for
    the dp4a path the largest of the dp4a, logic, shared-memory and issue
    bounds at the given rates (rows in chunks of 8, the remainder staged as 2,
    4 or 8 rows); for the small-M tensor path the MMA bound; no compute floor
    without a sampled clock."""
    shapes = [(2560, 2560), (6912, 2560), (2560, 6912)]
    row_beats = 2560 * 40 + 6912 * 40 + 2560 * 108
    tiles = 20 * 40 + 54 * 40 + 20 * 108
    f = 2070e6 * 152
    rates = {"dp4a": {"lanes_per_clk": 64.0}, "lop3": {"lanes_per_clk": 64.0},
             "lds128": {"bytes_per_clk": 128.0}}
    one = bench.batch_floors(1, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert one["bound"] == "hbm" and one["hbm_floor_ms"] == pytest.approx(1e9 / 6785.2e9 * 1e3)
    m8 = bench.batch_floors(8, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert m8["path"] == "dp4a" and m8["chunks"] == [8]
    assert m8["alu_floors_ms"]["dp4a"] == pytest.approx(row_beats * 128 / 64 / f * 1e3, rel=1e-3)
    assert m8["alu_floors_ms"]["logic"] == pytest.approx(row_beats * 33 / 64 / f * 1e3, rel=1e-3)
    assert m8["alu_floors_ms"]["shared"] == pytest.approx(row_beats * 256 / 128 / f * 1e3, rel=1e-3)
    assert m8["alu_floor_ms"] == m8["alu_floors_ms"]["dp4a"]
    m2 = bench.batch_floors(2, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert m2["alu_floors_ms"]["logic"] == pytest.approx(row_beats * 29 / 64 / f * 1e3, rel=1e-3)
    assert m2["alu_floors_ms"]["issue"] == pytest.approx(row_beats * (32 + 29 + 4) / 128 / f * 1e3,
                                                         rel=1e-3)
    m12 = bench.batch_floors(12, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert m12["chunks"] == [8, 4]
    assert m12["alu_floors_ms"]["dp4a"] == pytest.approx(row_beats * 192 / 64 / f * 1e3, rel=1e-3)
    m3 = bench.batch_floors(3, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert m3["chunks"] == [4]
    m64 = bench.batch_floors(64, shapes, 10**9, 6785.2, 152, 2070.0, rates)
    assert m64["path"].startswith("tensor") and m64["bound"] in ("hbm", "mma")
    assert m64["mma_floor_ms"] == pytest.approx(tiles * 4 * 101.4 / f * 1e3)
    assert m64["floor_ms"] == max(m64["hbm_floor_ms"], m64["mma_floor_ms"])
    unsampled = bench.batch_floors(8, shapes, 10**9, 6785.2, 152, None, rates)
    assert "alu_floor_ms" not in unsampled and unsampled["floor_ms"] == unsampled["hbm_floor_ms"]


def test_issue_rates_from_records(bench):
    """Two SMs: SM 0 ran two CTAs over 1000 clocks in total, SM 5 one CTA over
    400 clocks; 64 threads x 32 x 10 instructions per CTA."""
    import numpy as np
    rec = np.array([[0, 100, 900], [0, 200, 1100], [5, 50, 450]], dtype=np.int64)
    r = bench.issue_rates(rec, threads=64, iters=10)
    per_cta = 64 * 32 * 10
    assert r["sms"] == 2
    assert r["min"] == round(2 * per_cta / 1000, 2)
    assert r["max"] == round(per_cta / 400, 2)

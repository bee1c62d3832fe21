"""The gates record (profiles/gates.md): every test it names exists, and every
bench record the driver wrote at the repository root meets the resource
gates.  CPU only: it reads files."""
import glob
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GATES = os.path.join(ROOT, "profiles", "gates.md")


def test_every_named_test_exists():
    text = open(GATES).read()
    names = re.findall(r"`(tests/[\w/.]+\.py)(?:::(\w+))?`|`::(\w+)`", text)
    current = None
    seen = 0
    for path, fn, cont in names:
        if path:
            current = path
            assert os.path.exists(os.path.join(ROOT, path)), path
        fn = fn or cont
        if fn:
            src = open(os.path.join(ROOT, current)).read()
            assert re.search(rf"^def {fn}\(", src, re.M), f"{current}::{fn}"
            seen += 1
    assert seen >= 15


def bench_records():
    out = []
    for p in sorted(glob.glob(os.path.join(ROOT, "BENCH_r*.json"))):
        d = json.load(open(p))
        line = d.get("parsed") if isinstance(d, dict) else None
        if isinstance(line, dict) and "roofline" in line:
            out.append((os.path.basename(p), line))
    return out


def test_bench_records_meet_the_resource_gates():
    for name, b in bench_records():
        assert b["roofline"]["frac"] >= 0.70, name                          # R1
        traffic, algo = b["roofline"].get("traffic"), b["roofline"].get("algorithmic_bytes_per_launch")
        if traffic and algo:
            assert 0.97 <= traffic / algo <= 1.01, name                     # R2
        assert b["e2e"]["value"] >= 0.90 * b["value"], name                # R3
        m2 = b.get("configs", {}).get("config3", {}).get("by_M", {}).get("2")
        if m2:
            assert m2["us_per_step"] <= 130.0 and m2["err_flag"] == 0, name  # R4
        c4 = b.get("configs", {}).get("config4", {}).get("by_M", {}).get("2048")
        if c4:
            assert c4["frac_of_sustained_peak"] >= 0.58, name               # R5
        co = b.get("configs", {}).get("config2_ordered")
        if isinstance(co, dict):
            assert co["us_per_token"] <= 700.0 and co["err_flag"] == 0, name  # R7
        clk = b.get("clocks", {})
        bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
        assert not bad & set(clk.get("reasons") or []), name                # R6
        if b.get("err_flag") is not None:
            assert b["err_flag"] == 0, name


def test_committed_traffic_meets_r2():
    d = json.load(open(os.path.join(ROOT, "profiles", "select_accumulate_stack30.json")))
    assert 0.97 <= d["dram_bytes_per_launch"] / d["algorithmic_bytes_per_launch"] <= 1.01

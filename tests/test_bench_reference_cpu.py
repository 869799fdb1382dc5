"""The bench's reference arm (the float64 oracle on the host cores) keeps
its JSON contract; it needs no GPU, so it runs here.  The GPU arm is timed
on the GB300 only."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line_with_its_baseline():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1", "--ref-batches", "1"],
                         capture_output=True, text=True, check=True, timeout=600, cwd=ROOT)
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["config"]["workload"] == "d4096_ragged360_loguniform"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_clock_summary_keeps_only_samples_inside_the_timed_region(tmp_path):
    """The bench's clock record is the median under load: samples before and
    after the timed region (idle clocks) are left out."""
    import datetime
    sys.path.insert(0, ROOT)
    import bench

    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    rows = []
    for k in range(20):  # 10 ms apart; the region holds samples 5..14
        t = base + datetime.timedelta(milliseconds=10 * k)
        load = 5 <= k <= 14
        rows.append(", ".join([t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], "0",
                               "1650" if load else "2070", "2070", "1380.5" if load else "210.0",
                               "Not Active", "Not Active", "Not Active",
                               "Active" if load else "Not Active"]))
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    c = bench.Clocks(str(path))
    c.t0 = (base + datetime.timedelta(milliseconds=45)).timestamp()
    c.t1 = (base + datetime.timedelta(milliseconds=145)).timestamp()
    s = c.summary()
    assert s["window"] == "timed region" and s["samples"] == 10
    assert s["sm_mhz"] == 1650 and s["sm_min_mhz"] == 1650 and s["sm_max_mhz"] == 2070
    assert s["power_w"] == 1380.5 and s["reasons"] == ["sw_power_cap"]
    # no sample inside a very short region: the whole run, said so
    c.t0 = c.t1 = (base + datetime.timedelta(milliseconds=47)).timestamp()
    s = c.summary()
    assert s["samples"] == 20 and s["window"].startswith("whole sampler run")

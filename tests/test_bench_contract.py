"""The reference arm of bench.py (the CPU oracle, timed as it stands) prints
the one JSON line the benchmark contract asks for, and the clock record of
a bench line is summarised as the contract reads it.  CPU only: neither
needs a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] and d["unit"] == "GB/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith("batch64_8b")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_clock_record_summary():
    """The clocks object of a bench line from nvidia-smi rows: the median SM
    clock, the highest maximum, and each throttle reason seen Active at least
    once; rows that do not parse are skipped, and no sample gives None."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    row = lambda sm, hw="Not Active", th="Not Active", swt="Not Active", cap="Not Active": \
        "0, %s, 2070, 950.12, 0x0000000000000000, %s, %s, %s, %s" % (sm, hw, th, swt, cap)
    text = "\n".join([row(2070), row(2055), row(1980, cap="Active"), "0, [N/A], 2070, 1, 0x0, a, b, c, d",
                      "garbage", row(2070)])
    c = bench.summarize_clocks(text)
    assert c == {"sm_mhz": 2062.5, "sm_max_mhz": 2070.0, "samples": 4, "reasons": ["sw_power_cap"]}
    c = bench.summarize_clocks(row(1500, hw="Active") + "\n" + row(1500, th="Active", swt="Active"))
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.summarize_clocks("") is None and bench.summarize_clocks("garbage\n") is None

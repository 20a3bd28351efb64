"""The benchmark's reference arm (the fp64 oracle timed on the host cores):
its JSON line carries the keys of the benchmark contract, and under a
multi-rank launch only rank 0 prints.  Runs on the CPU (c2, a few steps)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "c2",
                           "--steps", "2", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["ms_per_step"] > 0 and abs(d["ms_per_step"] - 1e3 / d["value"]) < 1e-6 * d["ms_per_step"] + 1e-9
    assert "c2" in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_clock_record_from_nvidia_smi_rows():
    """The clocks entry that decides whether a timed run is kept: the median
    SM clock, the maximum, and every throttle reason active in any sample."""
    import bench
    idle = "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
    capped = "0, 1965, 2070, 1398.7, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
    thermal = "0, 1500, 2070, 1200.0, 0x0000000000000020, Not Active, Active, Not Active, Not Active\n"
    bad = ["0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n", "garbage\n", "\n"]
    r = bench.summarise_clock_rows([idle, idle, capped] + bad)
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    r = bench.summarise_clock_rows([idle, thermal, thermal, capped])
    assert r["sm_mhz"] == 1965.0 and r["samples"] == 4
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.summarise_clock_rows(bad) is None

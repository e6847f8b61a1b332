"""Host logic of bench.py that decides whether a timed run stands: the summary
of the nvidia-smi clock samples taken during the timed region (median SM
clock under load, throttle reasons seen, power), from a synthetic CSV in
nvidia-smi's `--format=csv,noheader,nounits` layout. No GPU involved."""
import os
import tempfile

import bench


class _Done:
    """Stands for the finished nvidia-smi process."""


def _summary(lines):
    fd, path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    cs = bench.ClockSampler("0")
    cs.proc, cs.path = _Done(), path
    out = cs.summary()
    assert not os.path.exists(path)  # the sample file is removed
    return out


def test_median_under_load_and_reasons():
    lines = [
        # index, sm, max sm, power, active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
        "0, 2070, 2070, 0.00, 0x0, Not Active, Not Active, Not Active, Not Active",    # idle: left out
        "0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2010, 2070, 1200.25, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, x, 2070, 5, 0x0, Not Active, Not Active, Not Active, Not Active",         # unparsable
    ]
    s = _summary(lines)
    assert s["sm_mhz"] == 2010.0            # median of the three loaded samples
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]  # kept and noted, not a rejection reason
    assert s["samples"] == 4
    assert s["power_w_max"] == 1200.25


def test_thermal_and_hardware_slowdown_are_reported():
    lines = [
        "0, 1500, 2070, 800, 0x48, Active, Not Active, Active, Not Active",
        "0, 1600, 2070, 850, 0x0, Not Active, Active, Not Active, Not Active",
    ]
    s = _summary(lines)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1550.0


def test_missing_power_counts_as_loaded_and_empty_file_gives_none():
    s = _summary(["0, 2070, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["power_w_max"] is None
    assert _summary(["not a sample"]) is None
    cs = bench.ClockSampler("0")           # nvidia-smi could not be started
    assert cs.summary() is None


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores (the
    reference arm) and prints one JSON line with the arm's keys; it needs no
    GPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1", "--ref-budget-s", "1"],
                         capture_output=True, text=True, check=True, timeout=600).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["metric"] == bench.METRIC and d["config"]["workload"] == bench.WORKLOAD

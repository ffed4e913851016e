"""The bench's reference arm on CPU: `bench.py --impl reference` times the
oracle on the host cores and prints one JSON line with the same metric, unit
and workload as the GPU arm, plus its own cpu_baseline and e2e objects."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "prefill_t32768"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == (os.cpu_count() or 1) and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_clock_sampler_summary_keeps_the_timed_windows():
    # fake nvidia-smi rows (host time, fields): only samples inside a timed
    # window (with 50 ms of slack) count towards the median and the reasons
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.p = object()
    row = lambda mhz, hw="Not Active", cap="Not Active": ["0", str(mhz), "2070", "900", "0x0", hw, "Not Active",
                                                          "Not Active", cap]
    cs.rows = [(0.0, row(1400, hw="Active")), (1.0, row(2070)), (1.2, row(2040, cap="Active")), (3.0, row(1000))]
    cs.windows = [(0.98, 1.21)]
    s = cs.summary()
    assert s["sm_mhz"] == 2055.0 and s["samples"] == 2 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert cs.summary([(2.9, 3.1)])["sm_mhz"] == 1000.0


def test_recorded_traffic_matches_workload_token_count_and_sources():
    # the roofline's `traffic` is the committed ncu capture of that kernel and
    # workload, dropped when the token count differs or the GEMM sources changed
    sys.path.insert(0, ROOT)
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "roofline_traffic.json")))
    key = "decode_t32/fc1"
    assert key in rec and rec[key]["T"] == 32
    got = bench.measured_traffic("decode_t32", 32, "fc1")
    if rec[key]["gemm_source_hash"] == bench.gemm_source_hash():
        assert got == rec[key]["dram_bytes_per_launch"]
    else:
        assert got is None
    assert bench.measured_traffic("decode_t32", 31, "fc1") is None
    assert bench.measured_traffic("decode_t32_T31", 31, "fc1") is None
    assert bench.measured_traffic("no_such_workload", 32, "fc1") is None

"""The benchmark's reference arm (the fp64 oracle on the host cores) prints the
contract's JSON line; it needs no GPU, so it runs here on a small workload."""
import json
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "layer_h512", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "layer_h512"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _traffic_records():
    prof = os.path.join(ROOT, "profiles")
    return sorted(os.path.join(prof, f) for f in os.listdir(prof)
                  if f.startswith("traffic_") and f.endswith(".json"))


def test_traffic_records_are_whole_and_consistent():
    """Each committed DRAM-traffic record names its kernel, workload, the ncu
    command (clocks left alone, committed files only), the source hash it was
    taken on, and bytes that add up: read + write = per launch, and at least
    the kernel's algorithmic bytes (the stream is read once; the excess is the
    look-ahead of the next kernel's bytes)."""
    recs = _traffic_records()
    assert recs
    for p in recs:
        d = json.load(open(p))
        for key in ("kernel", "workload", "dram_bytes_per_launch", "dram_bytes_read",
                    "dram_bytes_write", "algorithmic_bytes_per_launch", "kernel_source_sha",
                    "command"):
            assert key in d, (p, key)
        name = os.path.basename(p)[len("traffic_"):-len(".json")]
        assert name.endswith(d["workload"].split()[0]), (p, d["workload"])
        tot = d["dram_bytes_read"] + d["dram_bytes_write"]
        assert abs(d["dram_bytes_per_launch"] - tot) <= 1e5 + 1e-6 * tot, p
        assert d["dram_bytes_per_launch"] >= d["algorithmic_bytes_per_launch"], p
        cmd = d["command"]
        assert "--clock-control none" in cmd and "python bench.py" in cmd, p
        assert "/root" not in cmd and "_work" not in cmd, p
        assert len(d["kernel_source_sha"]) == 16, p


def test_bench_reports_traffic_only_for_matching_sources(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    p = _traffic_records()[0]
    d = json.load(open(p))
    kernel, workload = os.path.basename(p)[len("traffic_"):-len(".json")].rsplit("_stack", 1)
    workload = "stack" + workload
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: d["kernel_source_sha"])
    assert bench.profiled_traffic(workload, kernel) == d["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0" * 16)
    assert bench.profiled_traffic(workload, kernel) is None


def test_cpu_baseline_sample_is_sized_by_time_and_wraps():
    """The oracle sample beside the GPU line runs whole tokens at the timed
    positions until its time budget is spent, rewinding the cache at each
    wrap (the oracle itself insists on strictly sequential positions)."""
    sys.path.insert(0, ROOT)
    import bench
    from transformer_layer_decode_gb300 import synth
    w = synth.WORKLOADS["layer_h512"]
    host = bench.host_workload(w)
    n, t = bench.time_oracle_tokens(w, host, budget_s=0.2, positions=3)
    assert n > 3 and t >= 0.2            # wrapped at least once, sized by the budget
    n, _ = bench.time_oracle_tokens(w, host, budget_s=10.0, positions=4, max_tokens=9)
    assert n == 9                        # the token cap holds


def test_profile_summaries_name_safe_commands():
    """Every ncu command a committed profile summary gives leaves the clocks
    alone and runs committed files only (no scratch or machine paths)."""
    prof = os.path.join(ROOT, "profiles")
    seen = 0
    for f in sorted(os.listdir(prof)):
        text = open(os.path.join(prof, f)).read()
        for line in text.splitlines():
            if line.lstrip().startswith("#"):
                continue  # a heading
            if re.search(r"(^|\s|&&)ncu\s+--", line) and ("--metrics" in line or "--set" in line):
                seen += 1
                assert "--clock-control none" in line, (f, line)
        assert "_work/" not in text and "/root/" not in text, f
    assert seen > 0

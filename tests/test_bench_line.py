"""The JSON line of `bench.py --impl reference` (the oracle on the host cores; no GPU): one line
with the contract's keys, the reference arm's extras and a positive throughput."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_line_has_the_contract_keys():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3", "--ref-seconds", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["config"]["workload"] and d["config"]["nbs"] == [1, 2, 4, 8, 16]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] == 1 and cb["sample"]
    assert cb["host_cores"] >= 1 and cb["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_host_info_names_an_arm_cpu_from_its_part_number(monkeypatch):
    """Arm hosts list implementer and part numbers instead of a model name in /proc/cpuinfo."""
    import builtins
    import io

    import bench

    text = ("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\n"
            "CPU variant\t: 0x0\nCPU part\t: 0xd4f\nCPU revision\t: 0\n")
    real_open = builtins.open

    def fake_open(path, *a, **k):
        return io.StringIO(text) if path == "/proc/cpuinfo" else real_open(path, *a, **k)

    monkeypatch.setattr(builtins, "open", fake_open)
    info = bench.host_info()
    assert info["cpu_model"] == "Arm Neoverse-V2 (CPU implementer 0x41, part 0xd4f)"
    assert info["host_cores"] >= 1

"""bench.py's host-side pieces on the CPU: the clock record taken during the
timed region, the staleness rule of the committed DRAM-traffic figures, the
kernel the line names for a workload and the contract's argument checks."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_samples_median_and_reasons():
    rows = [
        "0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 2070, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 1980, 2070, 1400.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "garbage line\n",
    ]
    c = bench.parse_clock_samples(rows)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = rows[:1] + ["0, 1500, 2070, 1400.0, 0x48, Active, Not Active, Active, Not Active\n"]
    c = bench.parse_clock_samples(hot)
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and c["sm_mhz"] == 1785.0
    assert bench.parse_clock_samples(["0, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n"]) == {
        "sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 1}
    assert bench.parse_clock_samples([])["reasons"] == ["no samples"]


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "decode_attention_product_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "decode_pq.cu").write_bytes(b"kernel v1")
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"page1/step": {"dram_bytes": 123, "decode_pq_sha256": sha}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("page1", "step") == 123.0
    assert bench.measured_traffic("long", "step") is None          # never captured
    (src / "decode_pq.cu").write_bytes(b"kernel v2")                # source changed since
    assert bench.measured_traffic("page1", "step") is None


def test_committed_traffic_entries_name_their_capture():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for key in ("page1/step", "ragged/step", "long/step", "qwen_gqa/step"):
        e = t[key]
        assert e["dram_bytes"] == e["dram_read"] + e["dram_write"] > 0
        assert len(e["decode_pq_sha256"]) == 64 and "--clock-control none" in e["capture"]


def test_kernel_named_for_each_workload(monkeypatch):
    monkeypatch.delenv("AQPQ_DECODE_KERNEL", raising=False)
    assert bench.step_kernel_name(1, 4).startswith("pq_decode_kernel")
    assert bench.step_kernel_name(8, 4).startswith("pq_headsplit_kernel")
    assert bench.step_kernel_name(4, 8).startswith("pq_attend_kernel")
    monkeypatch.setenv("AQPQ_DECODE_KERNEL", "1")
    assert bench.step_kernel_name(8, 4).startswith("pq_decode_kernel")


def test_too_few_warmup_steps_rejected():
    r = subprocess.run([sys.executable, "bench.py", "--warmup", "2", "--steps", "1"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_clock_sampler_reads_what_nvidia_smi_printed(tmp_path, monkeypatch):
    """The sampler's own path end to end, with a stand-in nvidia-smi on PATH
    that prints two samples and then waits to be stopped."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 2070, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, 2055, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.start()
    c = s.stop()
    assert c == {"sm_mhz": 2062.5, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}
    assert not os.path.exists(s.path)

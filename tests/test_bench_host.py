"""Host-side logic of bench.py, on CPU: the reference arm's JSON line, the
max-over-ranks reduction with two gloo ranks, rank>0 silence of the
reference arm, and the clock-sample summary."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--ref-budget-s", "0.5"], capture_output=True,
                         text=True, timeout=600, env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "elements/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert rec["metric"] == bench.METRIC and rec["higher_is_better"] is True


def test_reference_arm_other_ranks_silent():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         env={**os.environ, "RANK": "1", "WORLD_SIZE": "2"})
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
rank = int(os.environ["RANK"])
bench.dist_init(2, "gloo")
got = bench.reduce_max(10.0 + 5 * rank, 2)
bench.barrier(2)
print("MAX", got)
"""


def test_reduce_max_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = {**os.environ, "RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank),
               "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)}
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
        assert "MAX 15.0" in o


def test_clock_summary(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "c.csv")
    with open(s.path, "w") as f:
        f.write("0, 1965, 2070, 400.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1980, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1990, 2070, 1250.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    out = s.summary()
    assert out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["sm_mhz"] == pytest.approx(1985.0)
    assert out["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_matches_sources_and_size(tmp_path, monkeypatch):
    """The committed DRAM traffic is reported only for the kernel sources and
    the launch size it was taken on."""
    import json

    import bench

    rec = {"source_hash": bench.kernel_source_hash(),
           "workloads": {"uniform": {"units_per_launch": 1 << 29, "traffic_bytes_per_launch": 4_000_000_000}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("uniform", 1 << 29) == 4_000_000_000
    assert bench.recorded_traffic("uniform", 1 << 26) is None  # a scaled run
    assert bench.recorded_traffic("skewed", 1 << 29) is None  # no record
    rec["source_hash"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("uniform", 1 << 29) is None  # kernels changed since

"""Host-side helpers of bench.py, on the CPU: the DRAM traffic records keyed
to source hashes, and the placement of the process on its GPU's local CPUs."""
import builtins
import hashlib
import io
import json
import os

import bench


def _write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(text)


def test_recorded_traffic_follows_its_sources(tmp_path, monkeypatch):
    root = str(tmp_path)
    _write(os.path.join(root, "src", "a.cu"), "kernel a")
    _write(os.path.join(root, "src", "b.cuh"), "header b")
    sha = lambda t: hashlib.sha256(t.encode()).hexdigest()
    rec = {"k": {"sources_sha256": {"src/a.cu": sha("kernel a"), "src/b.cuh": sha("header b")},
                 "dram_bytes_per_launch": 1234}}
    _write(os.path.join(root, "profiles", "dram_traffic.json"), json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.recorded_traffic("k", ["src/a.cu", "src/b.cuh"]) == 1234
    # a record keyed to other sources, or a missing key, gives nothing
    assert bench.recorded_traffic("k", ["src/a.cu"]) is None
    assert bench.recorded_traffic("other", ["src/a.cu", "src/b.cuh"]) is None
    # any change to a source (a comment counts) makes the record stale
    _write(os.path.join(root, "src", "b.cuh"), "header b // edited")
    assert bench.recorded_traffic("k", ["src/a.cu", "src/b.cuh"]) is None


def test_recorded_traffic_without_a_record_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k", []) is None


def test_gpu_local_cpus_from_the_pci_device(monkeypatch):
    calls = []
    monkeypatch.setattr(bench.subprocess, "check_output",
                        lambda cmd, **kw: calls.append(cmd) or "00000009:01:00.0\n")
    real_open = builtins.open

    def fake_open(path, *a, **kw):
        if str(path) == "/sys/bus/pci/devices/0009:01:00.0/local_cpulist":
            return io.StringIO("0-3,8,10-11\n")
        return real_open(path, *a, **kw)

    monkeypatch.setattr(builtins, "open", fake_open)
    monkeypatch.setattr(bench.os, "sched_getaffinity", lambda pid: {0, 1, 2, 3, 4, 5, 8, 9, 10})
    placed = []
    monkeypatch.setattr(bench.os, "sched_setaffinity", lambda pid, cpus: placed.append(set(cpus)))
    assert bench.bind_gpu_local_cpus("GPU-x") == [0, 1, 2, 3, 8, 10]  # local and allowed
    assert placed == [{0, 1, 2, 3, 8, 10}]
    assert calls and calls[0][-2:] == ["-i", "GPU-x"]


def test_gpu_local_cpus_without_the_topology(monkeypatch):
    def missing(cmd, **kw):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "check_output", missing)
    placed = []
    monkeypatch.setattr(bench.os, "sched_setaffinity", lambda pid, cpus: placed.append(cpus))
    assert bench.bind_gpu_local_cpus(None) is None
    assert placed == []  # nothing changed

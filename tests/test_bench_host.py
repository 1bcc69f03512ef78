"""Host logic of bench.py that shapes its JSON line, on the CPU: the clock
record (median SM clock over the samples under load, throttle reasons), the DRAM
traffic lookup (an entry is used only for the kernel sources, workload, chunk and
variant it was captured for) and the source hash it keys on."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler(lines):
    c = bench.ClockSampler()
    c.proc = _DoneProc()
    c.lines = lines
    return c


def test_clock_record_uses_the_samples_under_load():
    na = "Not Active"
    rows = [f"2070, 2070, 150.0, 0x0, {na}, {na}, {na}, {na}",      # idle before the region
            f"1700, 2070, 950.0, 0x4, {na}, {na}, {na}, Active",
            f"1690, 2070, 1000.0, 0x4, {na}, {na}, {na}, Active",
            f"1710, 2070, 980.0, 0x4, {na}, {na}, {na}, Active",
            f"2070, 2070, 300.0, 0x0, {na}, {na}, Active, {na}",     # idle after it
            "garbled line"]
    rec = _sampler([r + "\n" for r in rows]).stop()
    assert rec["sm_mhz"] == 1700.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["samples"] == 5 and rec["samples_under_load"] == 3
    assert rec["power_w_max"] == 1000.0
    # a reason seen only while idle is not reported for the timed region
    assert rec["reasons"] == ["sw_power_cap"]


def test_clock_record_flags_a_thermal_slowdown_under_load():
    na = "Not Active"
    rows = [f"1500, 2070, 900.0, 0x20, {na}, Active, {na}, {na}",
            f"1550, 2070, 920.0, 0x20, {na}, Active, {na}, Active"]
    rec = _sampler([r + "\n" for r in rows]).stop()
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == 1525.0


def test_clock_record_without_samples():
    assert _sampler([]).stop()["sm_mhz"] is None
    assert bench.ClockSampler().stop()["reasons"] == ["nvidia-smi unavailable"]


def _traffic_file(tmp_path, entries):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kernels": entries}))


def test_traffic_entries_are_keyed_on_sources_workload_chunk_and_variant(tmp_path, monkeypatch):
    src = ["lce_gemm.cu", "lce_internal.h", "lce_ptx.cuh"]
    sha = bench.kernel_source_hash(src)
    _traffic_file(tmp_path, {
        "phase": {"sources": src, "sha256_16": sha, "dram_bytes_per_launch_bench": 5.7e9,
                  "workload": "llama3-8b", "chunk": 1024},
        "stale": {"sources": src, "sha256_16": "0" * 16, "dram_bytes_per_launch_bench": 1.0,
                  "workload": "llama3-8b", "chunk": 1024},
        "fp16": {"sources": src, "sha256_16": sha, "dram_bytes_per_launch_bench": 2.0,
                 "workload": "llama3-8b", "chunk": 1024, "variant": "fp16"},
    })
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the hash reads the package sources, which stay where they are
    monkeypatch.setattr(bench, "kernel_source_hash",
                        lambda files: sha if files == src else "x")
    assert bench.load_traffic("llama3-8b", 1024, "") == {"phase": 5.7e9}
    assert bench.load_traffic("llama3-8b", 1024, "fp16") == {"fp16": 2.0}
    assert bench.load_traffic("qwen2.5-7b", 1024, "") == {}
    assert bench.load_traffic("llama3-8b", 2048, "") == {}


def test_traffic_lookup_without_the_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("llama3-8b", 1024, "") == {}


def test_kernel_source_hash_follows_the_file_contents():
    h = bench.kernel_source_hash(["lce_gemm.cu", "lce_internal.h", "lce_ptx.cuh"])
    assert len(h) == 16 and int(h, 16) >= 0
    assert h != bench.kernel_source_hash(["lce_internal.h", "lce_gemm.cu", "lce_ptx.cuh"])
    assert h == bench.kernel_source_hash(["lce_gemm.cu", "lce_internal.h", "lce_ptx.cuh"])


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)["kernels"]
    csrc = os.path.join(ROOT, "linear_cross_entropy_chunked_gb300", "csrc")
    assert entries
    for name, e in entries.items():
        assert e["sources"] and all(os.path.exists(os.path.join(csrc, s)) for s in e["sources"]), name
        assert len(e["sha256_16"]) == 16 and e["dram_bytes_per_launch_bench"] > 0, name

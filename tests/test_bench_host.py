"""Host logic of bench.py that needs no GPU: the ncu traffic records under profiles/ are
attached to a bench line only for the workload and kernel path they were captured on, and
only while the kernel's sources are the ones they were captured from."""
import re

import bench


def _record(kernel):
    text = open(f"{bench.ROOT}/profiles/traffic_{kernel}.md").read()
    return (re.search(r"workload:\s*(\S+)", text).group(1), re.search(r"path:\s*(\S+)", text).group(1),
            float(re.search(r"dram_bytes_per_launch_scaled:\s*([0-9.eE+]+)", text).group(1)),
            re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1))


def test_records_name_their_workload_and_path():
    for kernel in ("draft", "verify"):
        workload, path, nbytes, _ = _record(kernel)
        assert workload in ("qwen", "tiny", "highc", "dsv4", "ragged")
        assert nbytes > 0
        assert path in ("tensor-core", "verify")


def test_traffic_only_for_the_captured_workload_and_path(monkeypatch):
    for kernel in ("draft", "verify"):
        workload, path, nbytes, sha = _record(kernel)
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k, sha=sha: sha)
        assert bench.profiled_traffic(kernel, workload, path) == nbytes
        assert bench.profiled_traffic(kernel, "highc" if workload != "highc" else "qwen", path) is None
        assert bench.profiled_traffic(kernel, workload, "cuda-core-rnn") is None


def test_traffic_dropped_once_the_sources_change(monkeypatch):
    workload, path, _, sha = _record("draft")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 64)
    assert bench.profiled_traffic("draft", workload, path) is None
    assert bench.profiled_traffic("schedule", workload, path) is None   # no record at all

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
        assert path in ("tensor-core", "recompute", "stored")


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


def test_algorithmic_work_of_a_hand_worked_step():
    # B = 2 requests, V = 10, r = 4, bf16 (2 bytes); K_r = (2, 3); request 0 drafts 2 and
    # accepts 1 at T = 1 (rejection: its draft row is read for the residual), request 1 drafts 1
    # and accepts it at T = 0 (bonus row only)
    import numpy as np

    from speculative_decoding_draft_gb300 import workloads as wl
    cfg = wl.small_config("qwen", B=2, V=10, rank=4, dtype="bf16")
    K_r, ell, n_acc, T = np.array([2, 3]), np.array([2, 1]), np.array([1, 1]), np.array([1.0, 0.0])
    alg = bench.algorithmic(cfg, K_r, ell, n_acc, T)
    V, r, e = 10, cfg.rank, 2
    assert alg["draft_bytes"] == 5 * V * e + r * V * e + 5 * r * e       # U rows, W2 once, W1 rows
    assert alg["draft_flops"] == 2.0 * 5 * r * V
    assert alg["verify_bytes"] == (2 + 1 + 2) * V * e                     # rows to the decision (+ residual)
    assert alg["verify_bytes_dense"] == (5 + 3) * V * e                   # every row 2 l + 1
    assert (alg["positions"], alg["draft_positions"], alg["verify_positions"]) == (10, 5, 5)
    rnn = bench.algorithmic(cfg, K_r, ell, n_acc, T, head="rnn")
    assert rnn["draft_flops"] - alg["draft_flops"] == 2.0 * 5 * 3 * r * 2 * r   # the cell per position


def test_reference_arm_line_on_the_host(capsys, monkeypatch):
    # the oracle on the host cores; on a machine without a GPU it runs a reduced copy of the
    # workload and says so in the line
    import json

    import torch
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    if not torch.cuda.is_available():
        assert "reduced copy without a GPU" in line["config"]["workload"]

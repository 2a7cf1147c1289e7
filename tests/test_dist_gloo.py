"""The multi-process path of bench.py on CPU: two gloo ranks, no GPU.

Under torchrun every rank is one replica that drafts, schedules and verifies its own batch
of requests; the only collectives are the barrier around the timed region and the maximum
of the elapsed times.  Checked here: the plumbing (init, barrier, max over ranks, the
whole-job aggregate), that replicas get distinct batches (rank 0 keeps the configuration's
own), and that the reference arm leaves the other ranks without work.
"""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    try:
        import torch.distributed as dist

        import bench
        from speculative_decoding_draft_gb300 import workloads as wl
        r, w, _ = bench.dist_env()
        bench.dist_init(w, "gloo")
        bench.barrier(w)
        elapsed = 0.5 + r                       # rank 1 is the slower one
        slowest = bench.max_over_ranks(elapsed, w)
        value = bench.aggregate(960.0, slowest, w)
        cfg = wl.replica(wl.CONFIGS["qwen"], r)
        anchors = wl.request_params(wl.replica(wl.small_config("qwen", B=8, V=4096), r))["anchor"].tolist()
        bench.barrier(w)
        dist.destroy_process_group()
        q.put((r, slowest, value, cfg.data_seed, cfg.philox_seed, anchors, None))
    except Exception as exc:  # reported to the parent
        q.put((rank, None, None, None, None, None, repr(exc)))


def test_two_gloo_ranks_barrier_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        r, slowest, value, dseed, pseed, anchors, err = q.get(timeout=240)
        assert err is None, err
        out[r] = (slowest, value, dseed, pseed, anchors)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert out[r][0] == 1.5                      # the slowest rank's time on every rank
        assert out[r][1] == pytest.approx(960.0 * 2 / 1.5)
    from speculative_decoding_draft_gb300 import workloads as wl
    base = wl.CONFIGS["qwen"]
    assert (out[0][2], out[0][3]) == (base.data_seed, base.philox_seed)   # rank 0: the configuration
    assert out[1][2] != out[0][2] and out[1][3] != out[0][3]               # rank 1: its own batch
    assert out[0][4] != out[1][4]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""

"""Failure detection on the GPU without a fault: a bounded wait that runs out.

With DSPARK_FLAG_TEST_BARRIER_TIMEOUT the tensor-core draft's grid barrier before position 2
waits for one arrival more than the grid gives.  Nothing ever sets it, so the wait gives up
after its budget (about 2 s); every CTA drains its issued copies and MMAs, frees its tensor
memory and leaves, and the device status word reports DSPARK_ERR_DEVICE_TIMEOUT.  The context
stays usable: after the status is read and cleared, the same call without the flag gives the
same tokens as before.
"""
import ctypes
import time

import pytest
import torch

import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def test_barrier_wait_runs_out_and_the_context_stays_usable():
    cfg = wl.small_config(name="qwen", B=8, K_max=3, V=1032)
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    ref = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], cfg.philox_seed)
    assert ds.check(ref["status"]) == "DSPARK_OK"

    B, K, V, rank = cfg.B, cfg.K_max, cfg.V, cfg.rank
    dims = ds.Dims(B, K, V, rank, ds.BF16, ds.FLAG_TEST_BARRIER_TIMEOUT)
    ws = torch.empty(ds.lib().dspark_draft_workspace_bytes(dims), dtype=torch.uint8, device=DEV)
    tok = torch.full((B, K), -7, dtype=torch.int32, device=DEV)
    status = ds.new_status(DEV)
    t0 = time.perf_counter()
    code = ds.lib().dspark_draft_markov_sample(_p(g["U"]), _p(g["E"]), _p(g["W"]), _p(g["anchor"]), _p(g["K_r"]),
                                               _p(g["temperature"]), ctypes.c_uint64(cfg.philox_seed), dims, _p(tok),
                                               _p(None), _p(None), _p(None), _p(ws), ctypes.c_size_t(ws.numel()),
                                               _p(status),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert ds.STATUS_NAMES[code] == "DSPARK_OK"          # host-side validation passed
    assert ds.check(status) == "DSPARK_ERR_DEVICE_TIMEOUT"
    assert 0.5 < time.perf_counter() - t0 < 60.0        # the wait ran to its budget, then gave up

    again = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"],
                                   cfg.philox_seed, status=status)
    assert ds.check(again["status"]) == "DSPARK_OK"
    assert torch.equal(again["draft_tok"], ref["draft_tok"])
    live = torch.arange(K, device=DEV)[None, :] < g["K_r"][:, None]
    assert torch.equal(again["draft_lse"][live], ref["draft_lse"][live])

"""The workspace-free scheduler entry point agrees with the workspace entry point.

dspark_schedule_survival_noalloc serves callers that cannot allocate device
memory where they schedule (a serving loop that must not call cudaMalloc
between steps, or a plugin whose host owns every allocation and gives it no
workspace).  It runs on a static scratch array of the library instead of a
caller workspace.  This file is collected last so that a failure here comes
after every other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
MAX_CANDIDATES = 32768


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(conf, K_r, sps):
    B, K = conf.shape
    out = dict(ell=torch.full((B,), -7, dtype=torch.int32, device=DEV),
               tgt_off=torch.full((B + 1,), -7, dtype=torch.int32, device=DEV),
               theta_best=torch.zeros(1, dtype=torch.float64, device=DEV),
               b_star=torch.zeros(1, dtype=torch.int64, device=DEV),
               survival=torch.zeros(B, K, dtype=torch.float32, device=DEV))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    code = ds.lib().dspark_schedule_survival_noalloc(
        _p(conf), _p(K_r), _p(sps), sps.numel(), B, K, _p(out["ell"]), _p(out["tgt_off"]), _p(out["theta_best"]),
        _p(out["b_star"]), _p(out["survival"]), _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert ds.STATUS_NAMES[code] == "DSPARK_OK"
    assert ds.check(status) == "DSPARK_OK"
    return out


def _inputs(name, variant):
    cfg = wl.CONFIGS[name]
    conf = wl.confidences(cfg, "cpu").to(DEV)
    K_r = wl.request_params(cfg, "cpu")["K_r"].to(DEV)
    sps = wl.sps_table(cfg, variant).to(DEV)
    return conf, K_r, sps


def _same(a, b):
    for k in ("ell", "tgt_off", "theta_best", "b_star", "survival"):
        assert torch.equal(a[k], b[k]), k      # the schedule is bit-exact


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [_inputs("ragged", "step"), _inputs("dsv4", "literal")]
    refs = [ds.schedule_survival(*c) for c in cases]
    for ref in refs:
        assert ds.check(ref["status"]) == "DSPARK_OK"
    # two calls in a row on the same shape, then a different shape: the shared scratch keeps the
    # previous call's contents, which must not matter
    _same(_noalloc(*cases[0]), refs[0])
    _same(_noalloc(*cases[0]), refs[0])
    _same(_noalloc(*cases[1]), refs[1])


def test_noalloc_rejects_oversize_calls():
    B, K = MAX_CANDIDATES // 8 + 1, 8
    conf = torch.full((B, K), 0.5, device=DEV)
    K_r = torch.full((B,), K, dtype=torch.int32, device=DEV)
    sps = torch.ones(B * (K + 1) + 1, dtype=torch.float64, device=DEV)
    z = torch.zeros(B + 1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    code = ds.lib().dspark_schedule_survival_noalloc(_p(conf), _p(K_r), _p(sps), sps.numel(), B, K, _p(z), _p(z),
                                                     None, None, None, _p(status), None)
    assert ds.STATUS_NAMES[code] == "DSPARK_ERR_WORKSPACE"

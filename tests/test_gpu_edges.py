"""Edge cases on the GPU against the CPU oracle: the largest block (K_max = 16) on both
draft paths and in verification, verification with nothing to verify (every length 0: bonus
tokens only), and schedules without a single candidate."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

from parity_helpers import compare_draft, compare_verify, host, oracle_draft

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("simt", [False, True])
def test_draft_largest_block(simt):
    cfg = wl.small_config(name="ragged", B=24, K_max=16, V=2056)
    inp = wl.draft_inputs(cfg, "cpu")
    g = {k: v.to(DEV) for k, v in inp.items()}
    out = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], cfg.philox_seed,
                                 force_simt=simt)
    assert ds.check(out["status"]) == "DSPARK_OK"
    orc = oracle_draft(inp, cfg.philox_seed)
    assert compare_draft(out, orc, inp["K_r"].numpy(), cfg.dtype) >= 0.8 * int(inp["K_r"].sum())


def _verify_case(cfg, ell, seed):
    inp = wl.draft_inputs(cfg, "cpu")
    od = oracle_draft(inp, cfg.philox_seed)
    tgt_dense = wl.target_dense(cfg, inp["U"], inp["K_r"])
    flat, off = wl.flatten_targets(tgt_dense, torch.from_numpy(ell))
    D = torch.from_numpy(od["draft_logits"])
    if cfg.dtype == "bf16":
        D = D.view(torch.bfloat16)
    g = ds.verify_ragged(D.to(DEV), flat.to(DEV), off.to(DEV), torch.from_numpy(ell).to(DEV),
                         torch.from_numpy(od["draft_tok"]).to(DEV), inp["temperature"].to(DEV), seed)
    assert ds.check(g["status"]) == "DSPARK_OK"
    o = oracle.verify_ragged(host(D), host(flat), off.numpy(), ell, od["draft_tok"], inp["temperature"].numpy(), seed)
    return g, o


def test_verify_largest_block():
    cfg = wl.small_config(name="ragged", B=20, K_max=16, V=2056)
    K_r = wl.request_params(cfg)["K_r"].numpy()
    ell = K_r.astype(np.int32).copy()                 # verify every drafted position
    g, o = _verify_case(cfg, ell, 31)
    assert compare_verify(g, o) >= 0.8 * cfg.B


def test_verify_nothing_to_verify():
    cfg = wl.small_config(name="ragged", B=12, K_max=7, V=2056)
    ell = np.zeros(cfg.B, np.int32)                    # every request: one bonus token from its only row
    g, o = _verify_case(cfg, ell, 32)
    n = g["n_acc"].cpu().numpy()
    out = g["out_tok"].cpu().numpy()
    assert (n == 0).all()
    assert (out[:, 1:] == -1).all() and (out[:, 0] >= 0).all()
    assert compare_verify(g, o) >= 0.8 * cfg.B


def test_schedules_without_candidates():
    B, K = 40, 7
    conf = torch.zeros(B, K, device=DEV)
    conf[:, 0] = 0.0
    K_r = torch.full((B,), K, dtype=torch.int32, device=DEV)
    sps = torch.ones(B * (K + 1) + 1, dtype=torch.float64, device=DEV)
    s = ds.schedule_survival(conf, K_r, sps)
    c = ds.schedule_capacity(conf, K_r, sps)
    t = ds.schedule_topk(conf, K_r, torch.tensor([5], dtype=torch.int32, device=DEV))
    h = ds.schedule_threshold(conf, K_r, 0.0)
    for out in (s, c, t, h):
        assert ds.check(out["status"]) == "DSPARK_OK"
        assert int(out["ell"].sum()) == 0
        assert out["tgt_off"].cpu().tolist() == list(range(B + 1))
    assert c["capacity"].item() == 0
    o = oracle.schedule_survival(conf.cpu().numpy(), K_r.cpu().numpy(), sps.cpu().numpy())
    assert s["theta_best"].item() == o["theta_best"] and s["b_star"].item() == B

"""Verification with the rejecting draft rows recomputed (dspark_verify_markov) on the GPU.

The draft runs without storing its logits; the recompute verification must give exactly
what the stored-row verification gives on the same draft with its logits stored: the same
accept rule on log q(x_j) = z(x_j) / T - lse, and at a rejection the residual drawn from the
recomputed row, which the tensor-core kernel forms as the draft formed it ("DSpark" S2.1,
S3.1; "Speculative decoding, from zero to DSpark" S2, S6).  Outcomes are compared bit-exactly.
"""
import numpy as np
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


def _both(cfg, g, sps_variant="literal", packed=True):
    pk = ds.pack_projection(g["W"])
    d = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], cfg.philox_seed)
    n = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], cfg.philox_seed,
                               want_logits=False)
    conf = wl.confidences(cfg, "cpu")
    s = ds.schedule_survival(conf.to(DEV), g["K_r"], wl.sps_table(cfg, sps_variant).to(DEV))
    assert ds.check(d["status"]) == "DSPARK_OK" and ds.check(n["status"]) == "DSPARK_OK"
    assert ds.check(s["status"]) == "DSPARK_OK"
    assert torch.equal(d["draft_tok"], n["draft_tok"])
    tgt = wl.target_dense(cfg, g["U"], g["K_r"])
    flat, _ = wl.flatten_targets(tgt, s["ell"])
    del tgt
    seed = cfg.philox_seed + 7919
    a = ds.verify_ragged(d["draft_logits"], flat, s["tgt_off"], s["ell"], d["draft_tok"], g["temperature"], seed,
                         draft_lse=d["draft_lse"])
    b = ds.verify_markov(g["U"], g["E"], pk if packed else g["W"], g["anchor"], n["draft_lse"], n["draft_tok_logit"],
                         flat, s["tgt_off"], s["ell"], n["draft_tok"], g["temperature"], seed)
    assert ds.check(a["status"]) == "DSPARK_OK" and ds.check(b["status"]) == "DSPARK_OK"
    return a, b, s


CASES = {
    "ragged-greedy-mix": dict(name="ragged", B=150, K_max=5, V=4104),
    "qwen": dict(name="qwen", B=40, K_max=7, V=2056),
    "qwen-multitile": dict(name="qwen", B=300, K_max=3, V=64040),
    "rank64": dict(name="qwen", B=9, K_max=3, V=520, rank=64),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("packed", [True, False])
def test_verify_markov_equals_stored_rows(case, packed):
    cfg = wl.small_config(**CASES[case])
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    a, b, s = _both(cfg, g, packed=packed)
    assert torch.equal(a["n_acc"], b["n_acc"])
    assert torch.equal(a["out_tok"], b["out_tok"])
    # the comparison covers rejections with a residual draw
    ell = s["ell"].cpu().numpy()
    T = g["temperature"].cpu().numpy()
    assert ((a["n_acc"].cpu().numpy() < ell) & (T > 0)).sum() > 0


@pytest.mark.parametrize("name", ["qwen", "ragged"])
def test_verify_markov_full_size(name):
    cfg = wl.CONFIGS[name]
    g = wl.draft_inputs(cfg, DEV)
    a, b, s = _both(cfg, g, sps_variant="literal")
    assert torch.equal(a["n_acc"], b["n_acc"])
    assert torch.equal(a["out_tok"], b["out_tok"])
    del g, a, b, s
    torch.cuda.empty_cache()


def test_verify_markov_no_rejection_and_no_verification():
    # every length 0 (nothing to verify: bonus draws only) and greedy requests only (no residual pass work)
    cfg = wl.small_config("qwen", B=6, K_max=3, V=1032)
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    pk = ds.pack_projection(g["W"])
    n = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 5, want_logits=False)
    d = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 5)
    for ell_v, T in [(0, 1.0), (3, 0.0)]:
        ell = torch.full((cfg.B,), ell_v, dtype=torch.int32, device=DEV)
        off = torch.arange(cfg.B + 1, dtype=torch.int32, device=DEV) * (ell_v + 1)
        tgt = torch.randn(cfg.B * (ell_v + 1), cfg.V, device=DEV).to(torch.bfloat16)
        temp = torch.full((cfg.B,), T, device=DEV)
        b = ds.verify_markov(g["U"], g["E"], pk, g["anchor"], n["draft_lse"], n["draft_tok_logit"], tgt, off, ell,
                             n["draft_tok"], temp, 9)
        a = ds.verify_ragged(d["draft_logits"], tgt, off, ell, d["draft_tok"], temp, 9, draft_lse=d["draft_lse"])
        assert ds.check(b["status"]) == "DSPARK_OK" and ds.check(a["status"]) == "DSPARK_OK"
        assert torch.equal(a["out_tok"], b["out_tok"]) and torch.equal(a["n_acc"], b["n_acc"])

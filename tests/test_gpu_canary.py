"""Out-of-bounds writes: every output buffer of every entry point sits between guard regions.

Each output tensor is the middle of a larger allocation whose 4 KB before and after are
filled with a canary byte pattern; after the call the guards must be untouched.  The
shapes cover odd V, V not a multiple of 16 (the draft's 32-byte logit stores fall back to
16-byte ones), K_max = 16, a single request and ragged lengths, on both draft paths.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 4096          # bytes on each side (a multiple of 256: the inner view keeps its alignment)
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    """Allocations with canary guards; check() asserts every guard is intact."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        inner = raw[GUARD:GUARD + n].view(dtype).view(*shape)
        self.bufs.append((raw, n))
        return inner

    def check(self, what):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.bufs):
            head = raw[:GUARD]
            tail = raw[GUARD + n:]
            assert bool((head == CANARY).all()), f"{what}: output {i} written before its start"
            assert bool((tail == CANARY).all()), f"{what}: output {i} written past its end"


CASES = {
    "bf16-tc-ragged": dict(name="ragged", B=150, K_max=5, V=4104),
    "bf16-tc-V%16": dict(name="qwen", B=33, K_max=3, V=1032),
    "bf16-tc-Kmax16": dict(name="ragged", B=20, K_max=16, V=2056),
    "bf16-tc-single": dict(name="qwen", B=1, K_max=1, V=1032),
    "bf16-simt-odd": dict(name="qwen", B=7, K_max=4, V=1003),
    "fp32-oddV": dict(name="tiny", B=5, K_max=4, V=1003, rank=7),
}


def _draft_outputs(gd, cfg, U, conf_head=False, logits=True):
    B, K = cfg.B, cfg.K_max
    out = dict(draft_tok=gd((B, K), torch.int32), draft_lse=gd((B, K), torch.float32),
               draft_tok_logit=gd((B, K), torch.float32))
    if logits:
        out["draft_logits"] = gd(tuple(U.shape), U.dtype)
    if conf_head:
        out["conf"] = gd((B, K), torch.float32)
    return out


@pytest.mark.parametrize("case", list(CASES))
def test_guards_draft_schedule_verify(case):
    cfg = wl.small_config(**CASES[case])
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    B, K, V = cfg.B, cfg.K_max, cfg.V
    gd = Guarded()
    d = _draft_outputs(gd, cfg, g["U"])
    r = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 3, out=d)
    assert ds.check(r["status"]) == "DSPARK_OK"
    gd.check("draft")
    # confidence head fused into the draft
    h = wl.confidence_head(cfg, "cpu")
    dc = _draft_outputs(gd, cfg, g["U"], conf_head=True)
    r = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 3,
                               conf_h=h["conf_h"].to(DEV), conf_w=h["conf_w"].to(DEV), out=dc)
    assert ds.check(r["status"]) == "DSPARK_OK"
    gd.check("draft with the confidence head")
    # schedulers
    conf = wl.confidences(cfg, "cpu").to(DEV)
    sps = torch.ones(B * (K + 1) + 2, dtype=torch.float64, device=DEV)
    so = dict(ell=gd((B,), torch.int32), tgt_off=gd((B + 1,), torch.int32), theta_best=gd((1,), torch.float64),
              b_star=gd((1,), torch.int64), survival=gd((B, K), torch.float32))
    s = ds.schedule_survival(conf, g["K_r"], sps, out=so)
    assert ds.check(s["status"]) == "DSPARK_OK"
    cap = gd((1,), torch.int32)
    c = ds.schedule_capacity(conf, g["K_r"], sps, out=dict(capacity=cap, theta_best=gd((1,), torch.float64),
                                                          ell=gd((B,), torch.int32), tgt_off=gd((B + 1,), torch.int32)))
    assert ds.check(c["status"]) == "DSPARK_OK"
    t = ds.schedule_topk(conf, g["K_r"], cap, out=dict(ell=gd((B,), torch.int32), tgt_off=gd((B + 1,), torch.int32),
                                                      b_star=gd((1,), torch.int64), survival=gd((B, K), torch.float32)))
    assert ds.check(t["status"]) == "DSPARK_OK"
    th = ds.schedule_threshold(conf, g["K_r"], 0.5, out=dict(ell=gd((B,), torch.int32),
                                                             tgt_off=gd((B + 1,), torch.int32),
                                                             b_star=gd((1,), torch.int64),
                                                             survival=gd((B, K), torch.float32)))
    assert ds.check(th["status"]) == "DSPARK_OK"
    gd.check("schedulers")
    # verification over the schedule (every candidate admitted by the flat SPS table)
    ell = s["ell"]
    tgt = wl.target_dense(cfg, g["U"], g["K_r"])
    flat, _ = wl.flatten_targets(tgt, ell)
    for with_lse in (True, False):
        vo = dict(n_acc=gd((B,), torch.int32), out_tok=gd((B, K + 1), torch.int32))
        v = ds.verify_ragged(d["draft_logits"], flat, s["tgt_off"], ell, d["draft_tok"], g["temperature"], 5,
                             draft_lse=d["draft_lse"] if with_lse else None, out=vo)
        assert ds.check(v["status"]) == "DSPARK_OK"
    gd.check("verify_ragged")
    tc = cfg.dtype == "bf16" and cfg.rank % 64 == 0 and V % 8 == 0
    if tc:
        pk = ds.pack_projection(g["W"])
        n = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 3,
                                   out=_draft_outputs(gd, cfg, g["U"], logits=False))
        assert ds.check(n["status"]) == "DSPARK_OK"
        vo = dict(n_acc=gd((B,), torch.int32), out_tok=gd((B, K + 1), torch.int32))
        v = ds.verify_markov(g["U"], g["E"], pk, g["anchor"], n["draft_lse"], n["draft_tok_logit"], flat,
                             s["tgt_off"], ell, n["draft_tok"], g["temperature"], 5, out=vo)
        assert ds.check(v["status"]) == "DSPARK_OK"
        gd.check("draft without logits, verify_markov")


def test_guards_rnn_head():
    cfg = wl.small_config(name="ragged", B=40, K_max=5, V=2056)
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    h = {k: v.to(DEV) for k, v in wl.rnn_head(cfg, "cpu").items()}
    gd = Guarded()
    out = dict(draft_tok=gd((cfg.B, cfg.K_max), torch.int32), draft_lse=gd((cfg.B, cfg.K_max), torch.float32),
               draft_tok_logit=gd((cfg.B, cfg.K_max), torch.float32), draft_logits=gd(tuple(g["U"].shape), g["U"].dtype))
    r = ds.draft_rnn_sample(g["U"], g["E"], g["W"], h["rnn_W"], h["rnn_x"], g["anchor"], g["K_r"], g["temperature"],
                            3, out=out)
    assert ds.check(r["status"]) == "DSPARK_OK"
    gd.check("RNN-head draft")

"""The draft with the confidence head's Markov term fused in, against the CPU oracle.

The head's output at position k depends on the token drafted at k - 1, so it is compared
at every position whose previous token the oracle does not flag as a near tie; beyond K_r
it is zero.  The draft's own outputs must not change when the head is fused in.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

from parity_helpers import TOKEN_FLAGS, compare_draft, host, oracle_draft

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CONF_RTOL = 1e-5     # fp32 probabilities: relative tolerance stated for the method


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _compare_conf(conf, orc, inp, head, rows=None):
    """conf from the GPU vs the oracle's head applied to the oracle's own tokens.

    inp / head hold the compared requests only (GPU rows `rows`, default all)."""
    K_r = inp["K_r"].cpu().numpy()
    o = oracle.draft_confidence(host(inp["E"]), inp["anchor"].cpu().numpy(), orc["draft_tok"], K_r,
                                head["conf_h"].cpu().numpy(), head["conf_w"].cpu().numpy())
    c = conf.cpu().numpy()
    rows = range(c.shape[0]) if rows is None else rows
    n = 0
    for i, b in enumerate(rows):
        for k in range(c.shape[1]):
            if k >= K_r[i]:
                assert c[b, k] == 0.0
                continue
            if k > 0 and int(orc["flags"][i, k - 1]) & TOKEN_FLAGS:
                break          # the previous token may differ by a rounding-sized decision
            assert abs(c[b, k] - o[i, k]) <= CONF_RTOL * abs(o[i, k]), (b, k, c[b, k], o[i, k])
            n += 1
    return n


CASES = {
    "tiny-fp32": (dict(name="tiny"), False),
    "bf16-tc-ragged": (dict(name="ragged", B=150, K_max=3, V=4104), False),
    "bf16-tc-qwen": (dict(name="qwen", B=40, K_max=4, V=2056), False),
    "bf16-tc-rank64": (dict(name="qwen", B=9, K_max=3, V=520, rank=64), False),
    "bf16-simt-ragged": (dict(name="ragged", B=150, K_max=3, V=1048), True),
    "fp32-simt-oddV": (dict(name="tiny", B=5, K_max=4, V=1003, rank=7), False),
}


@pytest.mark.parametrize("case", list(CASES))
def test_fused_confidence_parity(case):
    kw, simt = CASES[case]
    cfg = wl.small_config(**kw)
    inp = wl.draft_inputs(cfg, "cpu")
    head = wl.confidence_head(cfg, "cpu")
    g = {k: v.to(DEV) for k, v in inp.items()}
    hd = {k: v.to(DEV) for k, v in head.items()}
    plain = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"],
                                   cfg.philox_seed, force_simt=simt)
    fused = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"],
                                   cfg.philox_seed, force_simt=simt, **hd)
    assert ds.check(plain["status"]) == "DSPARK_OK" and ds.check(fused["status"]) == "DSPARK_OK"
    # fusing the head changes none of the draft's outputs (entries past K_r are not written)
    live = torch.arange(cfg.K_max, device=DEV)[None, :] < g["K_r"][:, None]
    assert torch.equal(plain["draft_tok"], fused["draft_tok"])
    assert torch.equal(plain["draft_logits"][live], fused["draft_logits"][live])
    assert torch.equal(plain["draft_lse"][live], fused["draft_lse"][live])
    orc = oracle_draft(inp, cfg.philox_seed)
    compare_draft(fused, orc, inp["K_r"].numpy(), cfg.dtype, check_logits=False)
    n = _compare_conf(fused["conf"], orc, inp, head)
    assert n >= 0.9 * int(inp["K_r"].sum())


def test_fused_confidence_full_size_qwen():
    cfg = wl.CONFIGS["qwen"]
    g = wl.draft_inputs(cfg, DEV)
    head = wl.confidence_head(cfg, DEV)
    out = ds.draft_markov_sample(g["U"], g["E"], ds.pack_projection(g["W"]), g["anchor"], g["K_r"],
                                 g["temperature"], cfg.philox_seed, spare_sm=True, **head)
    assert ds.check(out["status"]) == "DSPARK_OK"
    rows = np.array([0, 17, 40, cfg.B - 1])
    idx = torch.from_numpy(rows).to(DEV)
    sub = {k: (v[idx] if k not in ("E", "W") else v) for k, v in g.items()}
    orc = oracle_draft(sub, cfg.philox_seed, req_id=rows.astype(np.int64))
    compare_draft(out, orc, sub["K_r"].cpu().numpy(), cfg.dtype, rows=rows)
    hsub = dict(conf_h=head["conf_h"][idx], conf_w=head["conf_w"])
    n = _compare_conf(out["conf"], orc, sub, hsub, rows=rows)
    assert n > 0
    # the scheduler consumes the fused confidences directly
    sps = wl.sps_table(cfg, "step").to(DEV)
    s = ds.schedule_survival(out["conf"], g["K_r"], sps)
    assert ds.check(s["status"]) == "DSPARK_OK"
    del g, out
    torch.cuda.empty_cache()

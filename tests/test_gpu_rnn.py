"""The RNN-head draft on the GPU against the CPU oracle, through the C ABI.

Tokens bit-exact outside the oracle's near-tie flags, normalisers within 1e-5 relative,
stored logits as for the Markov head except the fp32 absolute tolerance: the head's feature
is computed in fp32 (sigmoid, tanh and the recurrence), about 1e-6 per element, and enters
the bias through sum_i f_i W2[i, v], so the bias may move by up to ~1e-6 * sum_i |W2[i, v]|
(2e-5 for the fp32 case's rank 16, W2 ~ N(0, 0.1)).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

from parity_helpers import comparable, compare_draft, host

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _oracle_rnn(inp, head, seed, rows=None, req_id=None):
    sel = slice(None) if rows is None else rows
    return oracle.draft_rnn_sample(host(inp["U"][sel]), host(inp["E"]), host(inp["W"]), host(head["rnn_W"]),
                                   head["rnn_x"][sel].cpu().numpy(), inp["anchor"][sel].cpu().numpy(),
                                   inp["K_r"][sel].cpu().numpy(), inp["temperature"][sel].cpu().numpy(), seed,
                                   req_id=req_id, want_spread=inp["U"].dtype == torch.bfloat16)


CASES = {
    "tiny-fp32": dict(name="tiny"),
    "bf16-ragged-greedy-mix": dict(name="ragged", B=40, K_max=5, V=2056),
    "bf16-qwen": dict(name="qwen", B=16, K_max=7, V=4104),
    "fp32-oddV": dict(name="tiny", B=5, K_max=4, V=1003, rank=7),
}


@pytest.mark.parametrize("case", list(CASES))
def test_rnn_draft_parity(case):
    cfg = wl.small_config(**CASES[case])
    inp = wl.draft_inputs(cfg, "cpu")
    head = wl.rnn_head(cfg, "cpu")
    g = {k: v.to(DEV) for k, v in inp.items()}
    h = {k: v.to(DEV) for k, v in head.items()}
    out = ds.draft_rnn_sample(g["U"], g["E"], g["W"], h["rnn_W"], h["rnn_x"], g["anchor"], g["K_r"],
                              g["temperature"], cfg.philox_seed)
    assert ds.check(out["status"]) == "DSPARK_OK"
    orc = _oracle_rnn(inp, head, cfg.philox_seed)
    n = compare_draft(out, orc, inp["K_r"].numpy(), cfg.dtype, f32_atol=2e-5)
    assert n == comparable(orc["flags"], inp["K_r"].numpy())


def test_rnn_draft_full_size_qwen_sampled():
    cfg = wl.CONFIGS["qwen"]
    g = wl.draft_inputs(cfg, DEV)
    h = wl.rnn_head(cfg, DEV)
    out = ds.draft_rnn_sample(g["U"], g["E"], g["W"], h["rnn_W"], h["rnn_x"], g["anchor"], g["K_r"],
                              g["temperature"], cfg.philox_seed)
    assert ds.check(out["status"]) == "DSPARK_OK"
    rows = np.array([0, 17, 31, 48, cfg.B - 1])
    idx = torch.from_numpy(rows).to(DEV)
    sub = {k: (v[idx] if k not in ("E", "W") else v) for k, v in g.items()}
    hsub = dict(rnn_W=h["rnn_W"], rnn_x=h["rnn_x"][idx])
    orc = _oracle_rnn(sub, hsub, cfg.philox_seed, req_id=rows.astype(np.int64))
    n = compare_draft(out, orc, sub["K_r"].cpu().numpy(), cfg.dtype, rows=rows)
    assert n == comparable(orc["flags"], sub["K_r"].cpu().numpy())
    del g, out
    torch.cuda.empty_cache()


def test_rnn_closed_output_gate_matches_independent_drafting():
    # the oracle's pinned limit, on the GPU: no feature, so the draft of a zero projection
    cfg = wl.small_config(name="qwen", B=8, K_max=3, V=1032)
    inp = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    r = cfg.rank
    Wc = torch.zeros(3 * r, 2 * r, dtype=inp["U"].dtype, device=DEV)
    x = torch.zeros(cfg.B, cfg.K_max, 3 * r, device=DEV)
    x[..., 2 * r:] = -800.0
    a = ds.draft_rnn_sample(inp["U"], inp["E"], inp["W"], Wc, x, inp["anchor"], inp["K_r"], inp["temperature"], 3)
    b = ds.draft_markov_sample(inp["U"], inp["E"], torch.zeros_like(inp["W"]), inp["anchor"], inp["K_r"],
                               inp["temperature"], 3, force_simt=True)
    assert ds.check(a["status"]) == "DSPARK_OK" and ds.check(b["status"]) == "DSPARK_OK"
    assert torch.equal(a["draft_tok"], b["draft_tok"])
    assert torch.equal(a["draft_logits"], b["draft_logits"])

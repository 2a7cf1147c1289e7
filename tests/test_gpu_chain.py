"""The benchmark's step chained through the C ABI, against the oracle's chain.

The GPU step is the one the benchmark times: the draft (W2 packed once) writes tokens,
normalisers and the drawn tokens' logits; the scheduler computes the lengths and offsets;
verification consumes the GPU's own draft outputs and the target rows laid out by the GPU's
offsets, recomputing the rejecting draft rows (the same step with stored logits and the
stored-row verification is checked as well).  The
oracle runs the same chain on its own: its draft of the compared requests, its schedule of the
whole batch, its verification of those requests on its own draft.  Schedules are compared
bit-exactly in full; drafts as in the draft parity tests; verification outcomes (accepted
counts and emitted tokens) bit-exactly for every compared request whose verified draft
positions carry no token flag, outside the verification oracle's own near-tie flags (which
also cover the draft logits an fp32 evaluation may round the other way, "DSpark" S2.1;
"Speculative decoding, from zero to DSpark" S2).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

from parity_helpers import (comparable, compare_draft, compare_verify, draft_unflagged_upto, host, oracle_draft,
                            sample_rows)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
VERIFY_SEED_OFFSET = 7919          # the benchmark's verification seed is the draft's plus this


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gpu_step(cfg, g, sps_variant, markov=False):
    """markov: the benchmark's step -- the draft stores no logits and verification recomputes the
    rejecting rows (dspark_verify_markov); otherwise the draft stores its logits and
    dspark_verify_ragged reads them."""
    W = ds.pack_projection(g["W"]) if cfg.dtype == "bf16" and cfg.rank % 64 == 0 and cfg.rank <= 256 \
        and cfg.V % 8 == 0 else g["W"]
    d = ds.draft_markov_sample(g["U"], g["E"], W, g["anchor"], g["K_r"], g["temperature"], cfg.philox_seed,
                               want_logits=not markov)
    conf = wl.confidences(cfg, "cpu")
    sps = wl.sps_table(cfg, sps_variant)
    s = ds.schedule_survival(conf.to(DEV), g["K_r"], sps.to(DEV), status=d["status"])
    tgt = wl.target_dense(cfg, g["U"], g["K_r"])
    flat, off = wl.flatten_targets(tgt, s["ell"])
    del tgt
    if markov:
        v = ds.verify_markov(g["U"], g["E"], W, g["anchor"], d["draft_lse"], d["draft_tok_logit"], flat,
                             s["tgt_off"], s["ell"], d["draft_tok"], g["temperature"],
                             cfg.philox_seed + VERIFY_SEED_OFFSET, status=d["status"])
    else:
        v = ds.verify_ragged(d["draft_logits"], flat, s["tgt_off"], s["ell"], d["draft_tok"], g["temperature"],
                             cfg.philox_seed + VERIFY_SEED_OFFSET, draft_lse=d["draft_lse"], status=d["status"])
    assert ds.check(d["status"]) == "DSPARK_OK"
    assert torch.equal(off.to(DEV), s["tgt_off"])
    return d, s, v, flat, conf, sps


def _oracle_chain(cfg, g, rows, flat, conf, sps):
    """The oracle's chain for the requests `rows` (all of them when None)."""
    K_r = g["K_r"].cpu().numpy()
    o_s = oracle.schedule_survival(conf.numpy(), K_r, sps.numpy())
    sel = torch.from_numpy(rows).to(g["U"].device)
    sub = {k: (v[sel] if k not in ("E", "W") else v) for k, v in g.items()}
    od = oracle_draft(sub, cfg.philox_seed, req_id=rows.astype(np.int64))
    ell = o_s["ell"][rows]
    off = o_s["tgt_off"]
    parts = [host(flat[int(off[r]):int(off[r + 1])]) for r in rows]
    sub_flat = np.concatenate(parts)
    sub_off = np.zeros(len(rows) + 1, np.int32)
    sub_off[1:] = np.cumsum(ell + 1)
    T = sub["temperature"].cpu().numpy()
    ov = oracle.verify_ragged(od["draft_logits"], sub_flat, sub_off, ell, od["draft_tok"], T,
                              cfg.philox_seed + VERIFY_SEED_OFFSET, req_id=rows.astype(np.int64),
                              draft_spread=od["spread"])
    return o_s, od, ov, sub


def _check(cfg, g, rows, d, s, v, flat, conf, sps):
    o_s, od, ov, sub = _oracle_chain(cfg, g, rows, flat, conf, sps)
    np.testing.assert_array_equal(s["ell"].cpu().numpy(), o_s["ell"])
    np.testing.assert_array_equal(s["tgt_off"].cpu().numpy(), o_s["tgt_off"])
    assert s["theta_best"].item() == o_s["theta_best"]
    K_r = sub["K_r"].cpu().numpy()
    n = compare_draft(d, od, K_r, cfg.dtype, rows=rows)
    assert n == comparable(od["flags"], K_r)
    ok = draft_unflagged_upto(od["flags"], K_r, o_s["ell"][rows])
    keep = np.nonzero(ok)[0]
    assert len(keep) >= 0.75 * len(rows), (len(keep), len(rows))
    ov_keep = {k: val[keep] for k, val in ov.items()}
    compared = compare_verify(v, ov_keep, rows=rows[keep])
    assert compared >= 0.6 * len(rows), (compared, len(rows))
    return compared


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("ragged", dict(B=150, K_max=5, V=4104)),
                                     ("qwen", dict(B=40, K_max=7, V=2056))])
@pytest.mark.parametrize("sps_variant", ["literal", "step"])
def test_step_chain_small(name, kw, sps_variant):
    cfg = wl.small_config(name, **kw)
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    d, s, v, flat, conf, sps = _gpu_step(cfg, g, sps_variant)
    _check(cfg, g, np.arange(cfg.B), d, s, v, flat, conf, sps)


@pytest.mark.parametrize("name,kw", [("ragged", dict(B=150, K_max=5, V=4104)), ("qwen", dict(B=40, K_max=7, V=2056))])
@pytest.mark.parametrize("sps_variant", ["literal", "step"])
def test_step_chain_small_recompute(name, kw, sps_variant):
    cfg = wl.small_config(name, **kw)
    g = {k: v.to(DEV) for k, v in wl.draft_inputs(cfg, "cpu").items()}
    d, s, v, flat, conf, sps = _gpu_step(cfg, g, sps_variant, markov=True)
    _check(cfg, g, np.arange(cfg.B), d, s, v, flat, conf, sps)


@pytest.mark.parametrize("name", ["qwen", "ragged"])
@pytest.mark.parametrize("markov", [True, False])
def test_step_chain_full_size(name, markov):
    cfg = wl.CONFIGS[name]
    g = wl.draft_inputs(cfg, DEV)
    d, s, v, flat, conf, sps = _gpu_step(cfg, g, "literal", markov=markov)
    _check(cfg, g, sample_rows(cfg, 16), d, s, v, flat, conf, sps)
    del g, d, s, v, flat
    torch.cuda.empty_cache()

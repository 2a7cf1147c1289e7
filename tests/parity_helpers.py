"""Shared comparison helpers for the GPU-vs-oracle parity tests.

The oracle flags decisions that fp32 rounding could flip (near ties); a draft
position after a flagged one depends on the flagged token, so comparisons stop
at the first flagged position of a request.
"""
import numpy as np
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

LSE_RTOL = 1e-5   # fp32 probabilities / normalisers: relative tolerance stated for the method
# oracle draft flags that mean the token itself may differ: block/greedy margin, bf16
# rounding ambiguity, in-block boundary (bit 2 only concerns the log-sum-exp)
TOKEN_FLAGS = 1 | 2 | 8
LOGIT_ATOL = 1e-6   # absolute floor for stored logits: fp32 accumulation error of U + W1[x] . W2


def host(t):
    return wl.bf16_bits(t)


def oracle_draft(inp, seed, req_id=None, rows=None):
    sel = slice(None) if rows is None else rows
    U = host(inp["U"][sel])
    return oracle.draft_markov_sample(U, host(inp["E"]), host(inp["W"]), inp["anchor"][sel].cpu().numpy(),
                                      inp["K_r"][sel].cpu().numpy(), inp["temperature"][sel].cpu().numpy(), seed,
                                      req_id=req_id)


def compare_draft(gpu, orc, K_r, dtype, rows=None, check_logits=True, f32_atol=2e-6):
    """Compare stored logits, log-sum-exp and tokens; returns the number of compared tokens.

    Logits and the normaliser of position k depend only on earlier tokens, so they are
    compared at a flagged position too; the token is not, and the walk of that request
    stops there."""
    tok = gpu["draft_tok"].cpu().numpy()
    lse = None if gpu["draft_lse"] is None else gpu["draft_lse"].cpu().numpy()
    D = None
    if check_logits and gpu["draft_logits"] is not None:
        D = gpu["draft_logits"].float().cpu().numpy() if dtype == "bf16" else gpu["draft_logits"].cpu().numpy()
    oD = None
    if check_logits and orc["draft_logits"] is not None:
        oD = orc["draft_logits"]
        if dtype == "bf16":
            oD = (oD.astype(np.uint32) << 16).view(np.float32)
    rows = range(tok.shape[0]) if rows is None else rows
    n_cmp = 0
    mism_logits = 0
    total_logits = 0
    for i, b in enumerate(rows):
        for k in range(tok.shape[1]):
            if k >= K_r[i]:
                assert tok[b, k] == -1, (b, k)
                continue
            f = int(orc["flags"][i, k])
            if D is not None:
                d, o = D[b, k], oD[i, k]
                if dtype == "bf16":
                    bad = d != o
                    # only rounding-boundary cases may differ, by one bf16 step; where U and the
                    # bias cancel to a value near zero the fp32 sum's own error (~1e-9 here)
                    # exceeds that step, hence the absolute floor
                    if bad.any():
                        step = np.abs(o[bad]) * 2.0 ** -7 * 1.01 + LOGIT_ATOL
                        assert (np.abs(d[bad] - o[bad]) <= step).all(), (b, k)
                    mism_logits += int(bad.sum())
                else:
                    np.testing.assert_allclose(d, o, rtol=2e-6, atol=f32_atol)
                total_logits += d.size
            if lse is not None and not (f & 4):
                assert abs(lse[b, k] - orc["lse"][i, k]) <= LSE_RTOL * max(1.0, abs(orc["lse"][i, k])), \
                    (b, k, lse[b, k], orc["lse"][i, k])
            if f & TOKEN_FLAGS:
                break      # a rounding-sized change may move this token; later positions depend on it
            assert tok[b, k] == orc["draft_tok"][i, k], (b, k, tok[b, k], orc["draft_tok"][i, k], orc["margin"][i, k])
            n_cmp += 1
            if f:
                break
    if total_logits:
        assert mism_logits <= max(4, total_logits * 1e-4), (mism_logits, total_logits)
    return n_cmp


def compare_verify(gpu, orc, rows=None):
    n = gpu["n_acc"].cpu().numpy()
    out = gpu["out_tok"].cpu().numpy()
    rows = range(n.shape[0]) if rows is None else rows
    compared = 0
    for i, b in enumerate(rows):
        fp = int(orc["flag_pos"][i])
        if orc["flags"][i]:
            # decisions before the flagged position still agree
            m = min(fp - 1, int(orc["n_acc"][i]))
            assert (out[b, :m] == orc["out_tok"][i, :m]).all(), (b, out[b], orc["out_tok"][i])
            continue
        assert n[b] == orc["n_acc"][i], (b, n[b], orc["n_acc"][i])
        assert (out[b] == orc["out_tok"][i]).all(), (b, out[b], orc["out_tok"][i])
        compared += 1
    return compared

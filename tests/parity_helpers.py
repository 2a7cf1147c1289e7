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


def host(t):
    return wl.bf16_bits(t)


def oracle_draft(inp, seed, req_id=None, rows=None):
    sel = slice(None) if rows is None else rows
    U = host(inp["U"][sel])
    return oracle.draft_markov_sample(U, host(inp["E"]), host(inp["W"]), inp["anchor"][sel].cpu().numpy(),
                                      inp["K_r"][sel].cpu().numpy(), inp["temperature"][sel].cpu().numpy(), seed,
                                      req_id=req_id, want_spread=U.dtype == np.uint16)


def sample_rows(cfg, n):
    """n sampled requests of a full-size configuration: the first and the last, the rest drawn
    at random; where the configuration mixes temperatures, at least a quarter greedy ones."""
    rng = np.random.default_rng(1 + cfg.index)
    rows = set([0, cfg.B - 1])
    T = wl.request_params(cfg, "cpu")["temperature"].numpy()
    greedy = np.nonzero(T == 0.0)[0]
    if len(greedy):
        rows.update(rng.choice(greedy, size=n // 4, replace=False).tolist())
    while len(rows) < n:
        rows.add(int(rng.integers(cfg.B)))
    return np.array(sorted(rows))


def draft_unflagged_upto(flags, K_r, ell):
    """Requests whose oracle draft has no token flag at a verified position (k <= ell): the
    GPU draft tokens that verification reads then equal the oracle's."""
    ok = np.ones(len(ell), bool)
    for i in range(len(ell)):
        for k in range(min(int(ell[i]), int(K_r[i]))):
            if int(flags[i, k]) & TOKEN_FLAGS:
                ok[i] = False
                break
    return ok


def comparable(flags, K_r):
    """Positions compare_draft compares: each request up to its first flagged position, whose
    token is compared unless the flag says the token itself may differ."""
    n = 0
    for b, kr in enumerate(K_r):
        for k in range(int(kr)):
            f = int(flags[b, k])
            if f & TOKEN_FLAGS:
                break
            n += 1
            if f:
                break
    return n


def compare_draft(gpu, orc, K_r, dtype, rows=None, check_logits=True, f32_atol=2e-6, stats=None):
    """Compare stored logits, log-sum-exp and tokens; returns the number of compared tokens.

    Logits and the normaliser of position k depend only on earlier tokens, so they are
    compared at a flagged position too; the token is not, and the walk of that request
    stops there.  bf16 logits are bit-exact except at elements the oracle marks ambiguous
    (orc["spread"] > 0: another fp32 evaluation of U + bias may store another value), and
    there they lie within that spread of the oracle's."""
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
    spread = orc.get("spread")
    if D is not None and dtype == "bf16":
        assert spread is not None, "bf16 logit parity needs the oracle's per-element spread (want_spread=True)"
    rows = range(tok.shape[0]) if rows is None else rows
    n_cmp = 0
    counts = dict(logits=0, mismatch=0, flagged=0)
    for i, b in enumerate(rows):
        for k in range(tok.shape[1]):
            if k >= K_r[i]:
                assert tok[b, k] == -1, (b, k)
                continue
            f = int(orc["flags"][i, k])
            if D is not None:
                d, o = D[b, k], oD[i, k]
                if dtype == "bf16":
                    # |GPU - oracle| within the oracle's spread: bit-exact where the spread is 0
                    sp = spread[i, k].astype(np.float64)
                    diff = np.abs(d.astype(np.float64) - o.astype(np.float64))
                    bad = diff > sp
                    assert not bad.any(), (b, k, np.nonzero(bad)[0][:8], d[bad][:4], o[bad][:4], sp[bad][:4])
                    counts["mismatch"] += int((d != o).sum())
                    counts["flagged"] += int((sp > 0).sum())
                else:
                    np.testing.assert_allclose(d, o, rtol=2e-6, atol=f32_atol)
                counts["logits"] += d.size
            if lse is not None and not (f & 4):
                assert abs(lse[b, k] - orc["lse"][i, k]) <= LSE_RTOL * max(1.0, abs(orc["lse"][i, k])), \
                    (b, k, lse[b, k], orc["lse"][i, k])
            if f & TOKEN_FLAGS:
                break      # a rounding-sized change may move this token; later positions depend on it
            assert tok[b, k] == orc["draft_tok"][i, k], (b, k, tok[b, k], orc["draft_tok"][i, k], orc["margin"][i, k])
            n_cmp += 1
            if f:
                break
    if stats is not None:
        stats.update(counts)
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

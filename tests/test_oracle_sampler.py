"""Pins for the oracle's two-level categorical sampler.

The pages ask for a draw from a softmax (draft, bonus) or from the normalised
residual max(0, p - q) ("DSpark", S2.1 and S3.1; "Speculative decoding, from
zero to DSpark", S2 and S6) and fix no mechanism.  The oracle draws a block of
32 indices by Gumbel-max on the block masses and then an index inside the block
by inverse CDF.  These checks pin the law of that draw (Monte-Carlo frequencies
against w / sum(w) on ragged block counts, including laws that a wrong block
mass or a wrong in-block rule would produce), its limits, and the end-to-end
laws of the draft and verification steps over several blocks.
"""
import numpy as np
from scipy import stats

import oracle


def _chi2_p(counts, probs):
    counts = np.asarray(counts, np.float64)
    exp = np.asarray(probs, np.float64) * counts.sum()
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    e = e * c.sum() / e.sum()
    return stats.chisquare(c, e).pvalue


def _softmax(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def _draws(lw, n_draws, seed=7, position=1, tag=(oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)):
    return np.array([oracle.block_race(lw, seed, position, r, *tag)["pick"] for r in range(n_draws)])


def test_law_over_ragged_blocks():
    # 70 indices = blocks of 32, 32 and 6
    rng = np.random.default_rng(1)
    lw = rng.normal(0, 1.5, 70)
    lw[40] = 3.5                       # one heavy element inside the middle block
    w = np.exp(lw)
    p = w / w.sum()
    picks = _draws(lw, 60000)
    counts = np.bincount(picks, minlength=70)
    assert _chi2_p(counts, p) > 1e-4
    # a block chosen uniformly (masses ignored), then inverse CDF inside it
    blocks = [slice(0, 32), slice(32, 64), slice(64, 70)]
    wrong_uniform = np.concatenate([w[b] / w[b].sum() / 3 for b in blocks])
    assert _chi2_p(counts, wrong_uniform) < 1e-6
    # a block chosen by its largest weight instead of its mass
    mx = np.array([w[b].max() for b in blocks])
    wrong_max = np.concatenate([w[b] / w[b].sum() * mx[i] / mx.sum() for i, b in enumerate(blocks)])
    assert _chi2_p(counts, wrong_max) < 1e-6
    # uniform inside the block instead of proportional
    L = np.array([w[b].sum() for b in blocks])
    wrong_inblock = np.concatenate([np.full(b.stop - b.start, L[i] / L.sum() / (b.stop - b.start))
                                    for i, b in enumerate(blocks)])
    assert _chi2_p(counts, wrong_inblock) < 1e-6


def test_law_over_many_blocks():
    rng = np.random.default_rng(2)
    lw = rng.normal(0, 2.5, 1000)       # 32 blocks, the last one 8 wide
    p = _softmax(lw)
    picks = _draws(lw, 30000, seed=11, position=3, tag=(oracle.TAG_RESID, oracle.TAG_RESID_PICK))
    assert _chi2_p(np.bincount(picks, minlength=1000), p) > 1e-4


def test_zero_weights_are_never_drawn():
    rng = np.random.default_rng(3)
    lw = rng.normal(0, 1.0, 100)
    lw[::3] = -np.inf
    lw[64:96] = -np.inf                 # one whole block without mass
    picks = _draws(lw, 5000, seed=5)
    assert np.isfinite(lw[picks]).all()
    p = np.where(np.isfinite(lw), np.exp(np.where(np.isfinite(lw), lw, 0)), 0.0)
    assert _chi2_p(np.bincount(picks, minlength=100), p / p.sum()) > 1e-4


def test_single_element_and_empty_limits():
    lw = np.full(77, -np.inf)
    lw[50] = -3.0
    for r in range(50):
        out = oracle.block_race(lw, 9, 2, r, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)
        assert out["pick"] == 50 and out["block"] == 1
        assert out["margin"] == np.inf and not out["near_block"]
    out = oracle.block_race(np.full(40, -np.inf), 9, 2, 0, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)
    assert out["pick"] == -1


def test_shift_invariance():
    # adding a constant to every log-weight leaves the distribution and, away from
    # flagged near ties, every individual draw unchanged
    rng = np.random.default_rng(4)
    lw = rng.normal(0, 1.0, 90)
    same = 0
    for r in range(1500):
        a = oracle.block_race(lw, 3, 1, r, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)
        b = oracle.block_race(lw + 37.25, 3, 1, r, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)
        if a["near_err"] or b["near_err"]:
            continue
        assert a["pick"] == b["pick"]
        same += 1
    assert same > 1400


def test_uncertainty_flags_close_decisions():
    # two blocks with equal masses: the block scores differ only by the noise, so the
    # margin is small on some streams; a large uncertainty on one weight flags them all
    lw = np.zeros(64)
    le = np.full(64, -np.inf)
    le[3] = np.log(0.5)                 # +-0.5 on one unit weight of block 0 (mass 32)
    n_err = n_pure = 0
    for r in range(400):
        out = oracle.block_race(lw, 1, 1, r, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK)
        out_e = oracle.block_race(lw, 1, 1, r, oracle.TAG_DRAFT, oracle.TAG_DRAFT_PICK, log_err=le)
        assert out["pick"] == out_e["pick"]
        n_pure += out["near_err"]
        n_err += out_e["near_err"]
        # |log(32.5 / 32)| = 0.0155 bounds the score change; close margins must be flagged
        if abs(out["margin"]) < 0.015:
            assert out_e["near_err"]
    assert n_err > n_pure


def test_draft_marginal_over_blocks():
    # zero projection: every position is an independent softmax(U_k / T) draw over 100 ids
    V, N = 100, 40000
    rng = np.random.default_rng(6)
    U1 = rng.normal(0, 1.5, V).astype(np.float32)
    U = np.ascontiguousarray(np.broadcast_to(U1, (N, 1, V)))
    E = np.zeros((V, 2), np.float32)
    W = np.zeros((2, V), np.float32)
    for T in (1.0, 0.5):
        tok = oracle.draft_markov_sample(U, E, W, np.zeros(N), np.ones(N), np.full(N, T), seed=13,
                                         want_logits=False)["draft_tok"][:, 0]
        assert _chi2_p(np.bincount(tok, minlength=V), _softmax(U1.astype(np.float64) / T)) > 1e-4, T


def test_verify_output_law_over_blocks():
    # one draft position over 70 ids: the emitted first token follows the target p whatever
    # the draft q, and the acceptance rate is sum min(p, q)
    V, N = 70, 40000
    rng = np.random.default_rng(8)
    q_logits = rng.normal(0, 1.5, V).astype(np.float32)
    p_logits = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    E = np.zeros((V, 2), np.float32)
    W = np.zeros((2, V), np.float32)
    U = np.ascontiguousarray(np.broadcast_to(q_logits, (N, 1, V)))
    d = oracle.draft_markov_sample(U, E, W, np.zeros(N), np.ones(N), np.ones(N), seed=21)
    rows = np.ascontiguousarray(np.tile(p_logits, (N, 1)))
    off = np.arange(N + 1, dtype=np.int32) * 2
    v = oracle.verify_ragged(d["draft_logits"], rows, off, np.ones(N), d["draft_tok"], np.ones(N), seed=22)
    p = _softmax(p_logits[0])
    q = _softmax(q_logits)
    assert _chi2_p(np.bincount(v["out_tok"][:, 0], minlength=V), p) > 1e-4
    acc = np.mean(v["n_acc"] == 1)
    a = np.minimum(p, q).sum()
    assert abs(acc - a) < 5 * np.sqrt(a * (1 - a) / N)
    # corrections alone follow norm(max(0, p - q))
    rej = v["n_acc"] == 0
    r = np.maximum(p - q, 0)
    assert _chi2_p(np.bincount(v["out_tok"][rej, 0], minlength=V), r / r.sum()) > 1e-4

"""Pins for the oracle's ragged rejection-sampling verification.

Rule ("DSpark", S2.1; "Speculative decoding, from zero to DSpark", S2 and
Appendix A1): accept x_j with probability min(1, p_j(x_j) / q_j(x_j)), left to
right; at the first rejection sample norm(max(0, p_j - q_j)); if everything is
accepted sample a bonus token from the next target row.  Checked against the
printed two-token numbers, the closed form acceptance = sum_v min(p, q), and
Monte-Carlo output laws against the target rows on enumerated tiny cases with
Markov-biased (prefix-dependent) draft distributions.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


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


def _tile(x, n):
    return np.ascontiguousarray(np.broadcast_to(x, (n,) + x.shape))


def _draft_then_verify(U, E, W, anchor, tgt_rows, ell, N, T=1.0, seed=5):
    """N independent requests sharing one draft block and one set of target rows."""
    K = U.shape[0]
    d = oracle.draft_markov_sample(_tile(U, N), E, W, np.full(N, anchor), np.full(N, K), np.full(N, T), seed=seed)
    rows = np.ascontiguousarray(np.tile(tgt_rows[: ell + 1], (N, 1)))
    off = np.arange(N + 1, dtype=np.int32) * (ell + 1)
    v = oracle.verify_ragged(d["draft_logits"], rows, off, np.full(N, ell), d["draft_tok"], np.full(N, T),
                             seed=seed + 1)
    return d, v


def test_two_token_worked_numbers():
    g = json.load(open(os.path.join(GOLDEN, "resample_example.json")))
    p = np.array(g["p_target"])
    q = np.array(g["p_draft"])
    N = 200000
    U = np.log(q).astype(np.float32)[None, :]                 # one draft position
    E = np.zeros((2, 1), np.float32)
    W = np.zeros((1, 2), np.float32)
    p2 = np.array([0.2, 0.8])
    tgt = np.log(np.stack([p, p2])).astype(np.float32)        # target at position 1, bonus row
    d, v = _draft_then_verify(U, E, W, 0, tgt, ell=1, N=N)
    y1 = v["out_tok"][:, 0]
    acc = v["n_acc"] == 1
    sd = np.sqrt(0.25 / N)
    assert np.mean(y1 == 0) == pytest.approx(g["lossless_P_A"], abs=5 * sd)
    assert abs(np.mean(y1 == 0) - g["full_target_resample_P_A"]) > 20 * sd
    assert np.mean(acc) == pytest.approx(g["acceptance"], abs=5 * sd)
    assert np.mean(acc) == pytest.approx(np.minimum(p, q).sum(), abs=5 * sd)
    # every rejection resamples from norm(max(0, p - q)) = (1, 0)
    assert (y1[~acc] == 0).all()
    # the rejected token is always B (q(A) <= p(A) so A is always kept)
    assert (d["draft_tok"][~acc, 0] == 1).all()
    # after an accepted position the bonus is drawn from the next target row
    y2 = v["out_tok"][acc, 1]
    assert _chi2_p(np.bincount(y2, minlength=2), p2) > 1e-4
    assert (v["out_tok"][~acc, 1] == -1).all()


def test_output_law_equals_target_with_markov_drafts():
    V, K, rank, N = 4, 3, 2, 240000
    rng = np.random.default_rng(21)
    U = rng.normal(0, 1.0, (K, V)).astype(np.float32)
    E = rng.normal(0, 1.2, (V, rank)).astype(np.float32)
    W = rng.normal(0, 1.2, (rank, V)).astype(np.float32)
    tgt = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
    for T in (1.0, 0.6):
        d, v = _draft_then_verify(U, E, W, 1, tgt, ell=K, N=N, T=T, seed=91)
        out, n = v["out_tok"], v["n_acc"]
        P = [_softmax(tgt[k].astype(np.float64) / T) for k in range(K + 1)]
        for k in range(K + 1):
            reach = n >= k
            assert _chi2_p(np.bincount(out[reach, k], minlength=V), P[k]) > 1e-4, (T, k)
        # conditioned on each accepted first token the second output is still p_2
        for y in range(V):
            sel = (n >= 1) & (out[:, 0] == y)
            if sel.sum() > 2000:
                assert _chi2_p(np.bincount(out[sel, 1], minlength=V), P[1]) > 1e-4, (T, y)
        # acceptance at position 1 = sum_v min(p_1, q_1) (total-variation closed form)
        q1 = _softmax(d["draft_logits"][0, 0].astype(np.float64) / T)
        a1 = np.minimum(P[0], q1).sum()
        assert np.mean(n >= 1) == pytest.approx(a1, abs=5 * np.sqrt(a1 * (1 - a1) / N))
        assert 0.0 < a1 < 1.0


def test_greedy_verification():
    # T = 0: accept iff the draft token is the target argmax; correction/bonus = argmax
    V = 6
    D = np.zeros((2, 3, V), np.float32)
    tgt = np.zeros((2 + 4, V), np.float32)
    # request 0: ell = 1; target argmax 4; draft token 4 -> accepted; bonus row argmax 2
    tgt[0, 4] = 3.0
    tgt[1, 2] = 1.0
    # request 1: ell = 3; target argmaxes (1, 5, 0) / bonus 3; drafts (1, 2, 0) -> reject at 2, correction 5
    tgt[2, 1] = 1.0
    tgt[3, 5] = 1.0
    tgt[4, 0] = 1.0
    tgt[5, 3] = 1.0
    off = np.array([0, 2, 6], np.int32)
    tok = np.array([[4, 0, 0], [1, 2, 0]], np.int32)
    v = oracle.verify_ragged(D, tgt, off, [1, 3], tok, [0.0, 0.0], seed=0)
    assert v["n_acc"].tolist() == [1, 1]
    assert v["out_tok"].tolist() == [[4, 2, -1, -1], [1, 5, -1, -1]]


def test_zero_length_is_a_plain_target_sample():
    V, N = 5, 100000
    rng = np.random.default_rng(4)
    tgt_row = rng.normal(0, 1, (1, V)).astype(np.float32)
    D = np.zeros((N, 2, V), np.float32)
    rows = np.ascontiguousarray(np.tile(tgt_row, (N, 1)))
    off = np.arange(N + 1, dtype=np.int32)
    v = oracle.verify_ragged(D, rows, off, np.zeros(N), np.zeros((N, 2)), np.ones(N), seed=3)
    assert (v["n_acc"] == 0).all() and (v["out_tok"][:, 1:] == -1).all()
    assert _chi2_p(np.bincount(v["out_tok"][:, 0], minlength=V), _softmax(tgt_row[0])) > 1e-4


def test_retrospective_scheduler_bias_and_early_stop():
    # Appendix A: a scheduler that looks at c_2 (which depends on the sampled x_1) before
    # admitting x_1 outputs (0.85, 0.15); Algorithm 1's early stop never admits x_1 here and
    # the output stays (0.7, 0.3).
    g = json.load(open(os.path.join(GOLDEN, "appendix_a.json")))
    ex = g["two_token_example"]
    p = np.array(ex["p_target"])
    q = np.array(ex["p_draft"])
    sps = np.array([0.0, 1.0, 0.5, 0.45])
    N = 100000
    U = np.log(np.stack([q, q])).astype(np.float32)
    E = np.zeros((2, 1), np.float32)
    W = np.zeros((1, 2), np.float32)
    d = oracle.draft_markov_sample(np.ascontiguousarray(np.broadcast_to(U, (N, 2, 2))), E, W, np.zeros(N),
                                   np.full(N, 2), np.ones(N), seed=8)
    x1 = d["draft_tok"][:, 0]
    c2 = np.where(x1 == 0, 0.9, 0.0)                         # A -> confident continuation
    tgt = np.log(np.stack([p, p, p])).astype(np.float32)

    def run(ells):
        rows, off = [], [0]
        for l in ells:
            rows.append(tgt[: l + 1])
            off.append(off[-1] + l + 1)
        v = oracle.verify_ragged(d["draft_logits"], np.concatenate(rows), np.array(off, np.int32),
                                 np.array(ells), d["draft_tok"], np.ones(N), seed=9)
        return np.mean(v["out_tok"][:, 0] == 0)

    # Algorithm 1 per request (one request at a time, R = 1)
    ell_alg = []
    for r in range(N if N <= 200 else 200):
        conf = np.array([[0.8, c2[r]]], np.float32)
        ell_alg.append(int(oracle.schedule_survival(conf, [2], sps)["ell"][0]))
    assert set(ell_alg) == {0}
    sd = np.sqrt(0.25 / N)
    assert run([0] * N) == pytest.approx(ex["lossless_output"][0], abs=5 * sd)
    # the retrospective argmax picks ell = 2 after A and ell = 0 after B
    ell_retro = np.where(x1 == 0, 2, 0)
    assert run(ell_retro.tolist()) == pytest.approx(ex["retrospective_output"][0], abs=5 * sd)


def test_errors():
    D = np.zeros((2, 2, 4), np.float32)
    tgt = np.zeros((4, 4), np.float32)
    tok = np.zeros((2, 2), np.int32)
    oracle.verify_ragged(D, tgt, [0, 2, 4], [1, 1], tok, [1.0, 1.0], seed=0)
    cases = [
        (dict(tgt_off=[0, 2, 5]), "ERR_OFFSETS"),
        (dict(tgt_off=[1, 2, 4]), "ERR_OFFSETS"),
        (dict(ell=[3, 1], tgt_off=[0, 4, 6]), "ERR_LENGTHS"),
        (dict(draft_tok=np.array([[4, 0], [0, 0]], np.int32)), "ERR_TOKEN_RANGE"),
        (dict(temperature=[1.0, -0.5]), "ERR_TEMPERATURE"),
    ]
    for over, name in cases:
        args = dict(draft_logits=D, tgt_logits=tgt, tgt_off=[0, 2, 4], ell=[1, 1], draft_tok=tok,
                    temperature=[1.0, 1.0], seed=0)
        args.update(over)
        with pytest.raises(oracle.OracleError) as e:
            oracle.verify_ragged(**args)
        assert e.value.name == name


def _bits(x):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _vals(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _step(b, direction):
    # the bf16 neighbour of each value in the given direction (+1 / -1), exact in bit space
    v = _vals(b).astype(np.float64)
    up = (direction > 0) == (v >= 0)
    nb = np.where(up, b.astype(np.int32) + 1, b.astype(np.int32) - 1)
    nb = np.where(b == 0, np.where(direction > 0, 1, 0x8001), nb)
    return nb.astype(np.uint16)


def test_draft_ambiguity_marks_cover_one_step_changes():
    # Soundness of the draft_spread input: moving marked draft logits by one bf16 step (either
    # way, any subset) never changes the outcome of a request the marked run leaves unflagged
    # when the spread covers that step, the marks themselves never change the outcome, and
    # with dense marks some requests are flagged (the check is not vacuous).
    rng = np.random.default_rng(11)
    B, K, V = 96, 3, 256
    D = _bits(rng.normal(0, 2.0, (B, K, V)))
    tgt_dense = _vals(D).astype(np.float64)
    tgt = np.concatenate([tgt_dense + rng.normal(0, 0.7, (B, K, V)),
                          rng.normal(0, 2.0, (B, 1, V))], axis=1)
    flat = _bits(tgt.reshape(B * (K + 1), V))
    ell = np.full(B, K, np.int32)
    off = np.arange(B + 1, dtype=np.int32) * (K + 1)
    T = np.ones(B, np.float32)
    tok = np.zeros((B, K), np.int32)
    for b in range(B):                         # plausible drafts: argmax-ish tokens of their rows
        for k in range(K):
            tok[b, k] = int(rng.choice(np.argsort(_vals(D[b, k]))[-8:]))
    amb = (rng.uniform(size=D.shape) < 0.2).astype(np.uint8)
    # spread: the larger of the two bf16 steps around each marked value
    v = np.abs(_vals(D).astype(np.float64))
    spread = (amb * np.maximum(v * 2.0 ** -7, 2.0 ** -133)).astype(np.float32)
    base = oracle.verify_ragged(D, flat, off, ell, tok, T, seed=3)
    marked = oracle.verify_ragged(D, flat, off, ell, tok, T, seed=3, draft_spread=spread)
    np.testing.assert_array_equal(base["n_acc"], marked["n_acc"])
    np.testing.assert_array_equal(base["out_tok"], marked["out_tok"])
    clean = marked["flags"] == 0
    assert 0 < clean.sum() < B
    assert (marked["flags"] & ~base["flags"]).any()      # the marks add flags
    for trial in range(6):
        sel = (amb == 1) & (rng.uniform(size=D.shape) < 0.7)
        direction = np.where(rng.uniform(size=D.shape) < 0.5, 1, -1)
        Dp = np.where(sel, _step(D, direction), D).astype(np.uint16)
        pert = oracle.verify_ragged(Dp, flat, off, ell, tok, T, seed=3)
        np.testing.assert_array_equal(pert["n_acc"][clean], marked["n_acc"][clean])
        np.testing.assert_array_equal(pert["out_tok"][clean], marked["out_tok"][clean])

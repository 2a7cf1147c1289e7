"""Pins for the oracle's Markov-head draft sampler.

p_k(v | x_0, x_<k) = softmax(U_k(v) + W1[x_{k-1}] . W2 (v)), sampled left to
right from the anchor x_0 ("DSpark", S3.1; "Speculative decoding, from zero to
DSpark", S6).  The checks below do not restate the oracle's code: they use
hand-computed worked examples, the exact joint law by enumeration against
Monte-Carlo frequencies, and closed-form invariants.
"""
import itertools
import math

import numpy as np
import torch
import pytest
from scipy import stats

import oracle


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


def test_hand_worked_example_greedy():
    # V = 4, rank 2, fp32, greedy.  Worked by hand:
    #  x0 = 2 -> E[2] = (3, 0) -> bias = 3*W[0] = (3, 0, -3, 6);  z1 = U1 + bias = (3.5, -1, -1, 6) -> x1 = 3
    #  x1 = 3 -> E[3] = (1, 1) -> bias = W[0]+W[1] = (1, 1, 0, 1); z2 = (1, 1, 0, 1) -> tie, smallest -> x2 = 0
    #  x2 = 0 -> E[0] = (1, 2) -> bias = W[0]+2W[1] = (1, 2, 1, 0); z3 = U3 + bias = (1, 0, 1.25, 0) -> x3 = 2
    U = np.array([[[0.5, -1, 2, 0], [0, 0, 0, 0], [0, -2, 0.25, 0]]], np.float32)
    E = np.array([[1, 2], [0, 1], [3, 0], [1, 1]], np.float32)
    W = np.array([[1, 0, -1, 2], [0, 1, 1, -1]], np.float32)
    out = oracle.draft_markov_sample(U, E, W, anchor=[2], K_r=[3], temperature=[0.0], seed=0)
    assert out["draft_tok"].tolist() == [[3, 0, 2]]
    np.testing.assert_array_equal(out["draft_logits"][0],
                                  np.array([[3.5, -1, -1, 6], [1, 1, 0, 1], [1, 0, 1.25, 0]], np.float32))
    assert out["lse"][0].tolist() == [6.0, 1.0, 1.25]       # greedy: the row maximum
    assert out["flags"][0, 1] & 1                            # exact tie at position 2 is a near tie


def test_one_hot_transition_chain():
    # rank 2, one-hot embeddings: token 3 -> row 0 boosts v = 5; token 5 -> row 1 boosts v = 2;
    # every other token has a zero embedding.  Base logits prefer v = 1 everywhere.
    V = 6
    E = np.zeros((V, 2), np.float32)
    E[3, 0] = 1.0
    E[5, 1] = 1.0
    W = np.zeros((2, V), np.float32)
    W[0, 5] = 5.0
    W[1, 2] = 5.0
    U = np.zeros((2, 4, V), np.float32)
    U[:, :, 1] = 1.0
    out = oracle.draft_markov_sample(U, E, W, anchor=[3, 2], K_r=[4, 4], temperature=[0.0, 0.0], seed=1)
    assert out["draft_tok"][0].tolist() == [5, 2, 1, 1]     # anchor 3 -> 5 -> 2 -> (no bias) 1 -> 1
    assert out["draft_tok"][1].tolist() == [1, 1, 1, 1]     # anchor 2 has no transition
    assert out["flags"].max() == 0


def test_ragged_lengths_and_padding():
    V, K = 16, 5
    rng = np.random.default_rng(3)
    U = rng.normal(0, 2, (3, K, V)).astype(np.float32)
    E = rng.normal(0, 1, (V, 4)).astype(np.float32)
    W = rng.normal(0, 1, (4, V)).astype(np.float32)
    out = oracle.draft_markov_sample(U, E, W, anchor=[0, 1, 2], K_r=[1, 5, 3], temperature=[1.0, 1.0, 0.0], seed=9)
    tok = out["draft_tok"]
    assert (tok[0, 1:] == -1).all() and (tok[2, 3:] == -1).all() and (tok[1] >= 0).all()
    assert (tok[0, :1] >= 0).all() and (tok[2, :3] >= 0).all()


def test_exact_joint_law_by_enumeration():
    # Exact law of (x1, x2, x3) from the factorisation, against Monte-Carlo frequencies of
    # the oracle's Gumbel-max sampler over independent request streams.
    V, K, rank, N = 5, 3, 2, 120000
    rng = np.random.default_rng(11)
    U = rng.normal(0, 1.0, (K, V)).astype(np.float32)
    E = rng.normal(0, 1.0, (V, rank)).astype(np.float32)
    W = rng.normal(0, 1.0, (rank, V)).astype(np.float32)
    anchor = 4
    for T in (1.0, 0.7):
        law = {}
        for seq in itertools.product(range(V), repeat=K):
            prev, p = anchor, 1.0
            for k in range(K):
                z = U[k].astype(np.float64) + E[prev].astype(np.float64) @ W.astype(np.float64)
                p *= _softmax(z / T)[seq[k]]
                prev = seq[k]
            law[seq] = p
        out = oracle.draft_markov_sample(_tile(U, N), E, W, anchor=np.full(N, anchor), K_r=np.full(N, K),
                                         temperature=np.full(N, T), seed=2024, want_logits=False)
        tok = out["draft_tok"]
        code = (tok[:, 0] * V + tok[:, 1]) * V + tok[:, 2]
        counts = np.bincount(code, minlength=V ** K)
        probs = np.array([law[s] for s in itertools.product(range(V), repeat=K)])
        assert _chi2_p(counts, probs) > 1e-4, T
        # a transposed factor or a wrong conditioning index gives a visibly different law
        wrong = {}
        for seq in itertools.product(range(V), repeat=K):
            p = 1.0
            for k in range(K):
                z = U[k].astype(np.float64) + E[seq[k]].astype(np.float64) @ W.astype(np.float64)
                p *= _softmax(z / T)[seq[k]]
            wrong[seq] = p
        wprobs = np.array([wrong[s] for s in itertools.product(range(V), repeat=K)])
        wprobs /= wprobs.sum()
        assert _chi2_p(counts, wprobs) < 1e-6


def test_zero_bias_is_independent_parallel_drafting():
    # W2 = 0 removes the transition: tokens no longer depend on the anchor or on earlier
    # tokens, and each position is an independent draw from softmax(U_k / T).
    V, K, N = 7, 3, 60000
    rng = np.random.default_rng(5)
    U = rng.normal(0, 1.0, (K, V)).astype(np.float32)
    E = rng.normal(0, 1.0, (V, 3)).astype(np.float32)
    W = np.zeros((3, V), np.float32)
    a = oracle.draft_markov_sample(_tile(U, N), E, W, np.zeros(N), np.full(N, K), np.ones(N), seed=77,
                                   want_logits=False)["draft_tok"]
    b = oracle.draft_markov_sample(_tile(U, N), E, W, np.full(N, 6), np.full(N, K), np.ones(N), seed=77,
                                   want_logits=False)["draft_tok"]
    np.testing.assert_array_equal(a, b)
    for k in range(K):
        assert _chi2_p(np.bincount(a[:, k], minlength=V), _softmax(U[k])) > 1e-4
    # independence of positions 1 and 2
    ct = np.zeros((V, V))
    np.add.at(ct, (a[:, 0], a[:, 1]), 1)
    assert stats.chi2_contingency(ct + 0.0)[1] > 1e-4
    # with a non-zero projection the anchor matters
    W2 = rng.normal(0, 1.0, (3, V)).astype(np.float32)
    c = oracle.draft_markov_sample(_tile(U, 200), E, W2, np.zeros(200), np.full(200, K), np.ones(200), seed=77,
                                   want_logits=False)["draft_tok"]
    d = oracle.draft_markov_sample(_tile(U, 200), E, W2, np.full(200, 6), np.full(200, K), np.ones(200), seed=77,
                                   want_logits=False)["draft_tok"]
    assert not np.array_equal(c, d)


def test_log_sum_exp_normalises():
    V, K = 300, 4
    rng = np.random.default_rng(8)
    U = rng.normal(0, 3, (3, K, V)).astype(np.float32)
    E = rng.normal(0, 0.5, (V, 8)).astype(np.float32)
    W = rng.normal(0, 0.5, (8, V)).astype(np.float32)
    T = np.array([0.5, 1.0, 2.0], np.float32)
    out = oracle.draft_markov_sample(U, E, W, [1, 2, 3], [K] * 3, T, seed=4)
    D = out["draft_logits"].astype(np.float64)
    for b in range(3):
        for k in range(K):
            s = np.exp(D[b, k] / T[b] - out["lse"][b, k]).sum()
            assert s == pytest.approx(1.0, abs=1e-12)


def test_bf16_storage_rounding():
    # bf16 biased logits are the exact value rounded to nearest, ties to even.
    # Spacing of bf16 near 1.0 is 2^-7.
    def bits(x):
        return (np.array(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)

    def val(b):
        return (b.astype(np.uint32) << 16).view(np.float32)

    cases = [  # (U, W value with E = 1, expected stored logit)
        (1.0, 3 * 2.0 ** -9, 1.0078125),     # 1 + 0.75 q  -> up
        (1.0, 2.0 ** -9, 1.0),               # 1 + 0.25 q  -> down
        (1.0, 2.0 ** -8, 1.0),               # 1 + 0.5 q   -> tie, even (128)
        (1.0078125, 2.0 ** -8, 1.015625),    # 129.5 q     -> tie, even (130)
    ]
    for u, w, want in cases:
        U = bits([[[u, -8.0]]])
        E = bits([[1.0], [1.0]])
        W = bits([[w, 0.0]])
        out = oracle.draft_markov_sample(U, E, W, [0], [1], [0.0], seed=0)
        assert float(val(out["draft_logits"])[0, 0, 0]) == want
        assert oracle.round_bf16(u + w) == want


def test_bf16_rounding_ambiguity_is_flagged():
    # greedy row whose top value sits on a rounding midpoint and whose runner-up equals the
    # other rounding: an fp32 evaluation could pick either token -> flagged.
    def bits(x):
        return (np.array(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    U = bits([[[1.0, 1.0078125, -3.0]]])
    E = bits([[1.0], [1.0], [1.0]])
    W = bits([[2.0 ** -8, 0.0, 0.0]])            # element 0: 1 + q/2 (midpoint), element 1: 1 + q
    out = oracle.draft_markov_sample(U, E, W, [0], [1], [0.0], seed=0)
    assert out["flags"][0, 0] & 2


def test_argument_errors():
    U = np.zeros((2, 3, 8), np.float32)
    E = np.zeros((8, 2), np.float32)
    W = np.zeros((2, 8), np.float32)
    ok = dict(anchor=[0, 1], K_r=[3, 2], temperature=[1.0, 0.0], seed=0)
    oracle.draft_markov_sample(U, E, W, **ok)
    for key, bad, name in [("K_r", [0, 2], "ERR_LENGTHS"), ("K_r", [4, 2], "ERR_LENGTHS"),
                           ("anchor", [8, 0], "ERR_TOKEN_RANGE"), ("anchor", [-1, 0], "ERR_TOKEN_RANGE"),
                           ("temperature", [-1.0, 1.0], "ERR_TEMPERATURE"),
                           ("temperature", [1e-4, 1.0], "ERR_TEMPERATURE"),
                           ("temperature", [float("nan"), 1.0], "ERR_TEMPERATURE")]:
        args = dict(ok)
        args[key] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.draft_markov_sample(U, E, W, **args)
        assert e.value.name == name


def _bf16_bits_from_f32(x):
    # round-to-nearest-even fp32 -> bf16 by torch (a library routine, not the oracle's rounding)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _f32_of_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def test_ambiguity_covers_fp32_evaluations():
    # Every bf16 logit an fp32 evaluation of U + W1[x] . W2 stores, whatever the summation order,
    # lies within the oracle's spread of the oracle's value (so equals it where the spread is 0);
    # forced cancellations (U = -bias) get spreads of several bf16 steps.
    rng = np.random.default_rng(5)
    V, rank, K = 8192, 256, 2
    bits = lambda a: _bf16_bits_from_f32(a.astype(np.float32))
    E = bits(rng.normal(0, 0.02, (V, rank)))
    W = bits(rng.normal(0, 0.02, (rank, V)))
    U = bits(rng.normal(0, 3.0, (1, K, V)))
    anchor = 17
    Ef, Wf = _f32_of_bits(E).astype(np.float64), _f32_of_bits(W).astype(np.float64)
    cancel = rng.choice(V, 64, replace=False)
    U[0, 0, cancel] = bits(-(Ef[anchor] @ Wf)[cancel])          # U + bias cancels to near zero
    out = oracle.draft_markov_sample(U, E, W, [anchor], [K], [0.0], seed=0, want_spread=True)
    spread = out["spread"].astype(np.float64)
    stored = _f32_of_bits(out["draft_logits"]).astype(np.float64)
    steps = np.abs(stored) * 2.0 ** -8       # at least one bf16 step is below this
    assert (spread[0, 0, cancel] > 2 * steps[0, 0, cancel]).mean() > 0.9
    prev = [anchor, int(out["draft_tok"][0, 0])]
    Uf = _f32_of_bits(U)
    W32 = _f32_of_bits(W)
    mism = 0
    for k in range(K):
        e = _f32_of_bits(E[prev[k]])
        terms = e[:, None] * W32                                # exact in fp32 (bf16 x bf16)
        orders = [np.arange(rank), np.arange(rank)[::-1], rng.permutation(rank)]
        sums = []
        for order in orders:                                    # sequential fp32 accumulation
            acc = np.zeros(V, np.float32)
            for i in order:
                acc = (acc + terms[i]).astype(np.float32)
            sums.append(acc)
        # chunks of 16 summed pairwise, then the chunk sums in order (a tensor-core-like order)
        chunk = terms.reshape(rank // 16, 16, V).sum(axis=1, dtype=np.float32)
        acc = np.zeros(V, np.float32)
        for c in chunk:
            acc = (acc + c).astype(np.float32)
        sums.append(acc)
        for s in sums:
            z = (Uf[0, k] + s).astype(np.float32)
            got = _f32_of_bits(_bf16_bits_from_f32(z)).astype(np.float64)
            diff = np.abs(got - stored[0, k])
            assert (diff <= spread[0, k]).all(), np.nonzero(diff > spread[0, k])[0][:8]
            mism += int((diff > 0).sum())
    assert mism > 0                                   # the check is not vacuous
    assert (spread > 0).mean() < 0.02                 # and the marks stay rare

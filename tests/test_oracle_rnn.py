"""Pins for the oracle's RNN-head draft ("DSpark" S3.1, RNN head).

Checked against limits that reduce it to pinned functions (a closed output gate gives
independent parallel drafting; saturated gates with an identity candidate block give the
Markov head on tanh(W1)), the closed form of the state under constant pre-activations,
s_k = c (1 - g^k) from s_0 = 0, and the memory the Markov head lacks.
"""
import math

import numpy as np
import pytest

import oracle


def _case(seed, B=3, K=4, V=300, rank=8, T=1.0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2.0, (B, K, V)).astype(np.float32)
    E = rng.normal(0, 0.3, (V, rank)).astype(np.float32)
    W = rng.normal(0, 0.3, (rank, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    K_r = np.full(B, K, np.int32)
    temp = np.full(B, T, np.float32)
    return U, E, W, anchor, K_r, temp


def test_closed_output_gate_is_independent_drafting():
    U, E, W, anchor, K_r, temp = _case(0)
    B, K, V = U.shape
    r = E.shape[1]
    rng = np.random.default_rng(1)
    Wc = rng.normal(0, 0.5, (3 * r, 2 * r)).astype(np.float32)
    cx = rng.normal(0, 1.0, (B, K, 3 * r)).astype(np.float32)
    cx[..., 2 * r:] = -800.0                      # sigmoid(-800) = 0 exactly: no feature
    rnn = oracle.draft_rnn_sample(U, E, W, Wc, cx, anchor, K_r, temp, seed=5, want_feat=True)
    assert np.all(rnn["feat"] == 0.0)
    ind = oracle.draft_markov_sample(U, E, np.zeros_like(W), anchor, K_r, temp, seed=5)
    np.testing.assert_array_equal(rnn["draft_tok"], ind["draft_tok"])
    np.testing.assert_array_equal(rnn["draft_logits"], ind["draft_logits"])
    np.testing.assert_array_equal(rnn["lse"], ind["lse"])


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_saturated_gates_reduce_to_the_markov_head_on_tanh_w1(T):
    U, E, W, anchor, K_r, temp = _case(2, T=T)
    B, K, V = U.shape
    r = E.shape[1]
    Wc = np.zeros((3 * r, 2 * r), np.float32)
    Wc[r:2 * r, r:2 * r] = np.eye(r, dtype=np.float32)   # candidate = the previous token's embedding
    cx = np.zeros((B, K, 3 * r), np.float32)
    cx[..., :r] = -800.0                                  # gate 0: the state is replaced each step
    cx[..., 2 * r:] = 800.0                               # output 1
    rnn = oracle.draft_rnn_sample(U, E, W, Wc, cx, anchor, K_r, temp, seed=9, want_feat=True)
    Et = np.tanh(E.astype(np.float64)).astype(np.float32)
    mk = oracle.draft_markov_sample(U, Et, W, anchor, K_r, temp, seed=9)
    toks = rnn["draft_tok"]
    for b in range(B):
        prev = anchor[b]
        for k in range(K):
            np.testing.assert_allclose(rnn["feat"][b, k], np.tanh(E[prev].astype(np.float64)), rtol=1e-15,
                                       atol=1e-300)
            if rnn["flags"][b, k] or mk["flags"][b, k]:
                break                  # a near tie: the fp32 rounding of tanh(W1) may flip it
            assert toks[b, k] == mk["draft_tok"][b, k]
            np.testing.assert_allclose(rnn["draft_logits"][b, k], mk["draft_logits"][b, k], rtol=0, atol=1e-6)
            prev = toks[b, k]


def test_constant_preactivations_closed_form():
    U, E, W, anchor, K_r, temp = _case(3, K=7)
    B, K, V = U.shape
    r = E.shape[1]
    rng = np.random.default_rng(4)
    pre = rng.normal(0, 1.5, 3 * r).astype(np.float32)
    cx = np.broadcast_to(pre, (B, K, 3 * r)).copy()
    Wc = np.zeros((3 * r, 2 * r), np.float32)            # no dependence on the state or the tokens
    rnn = oracle.draft_rnn_sample(U, E, W, Wc, cx, anchor, K_r, temp, seed=1, want_feat=True)
    p = pre.astype(np.float64)
    g = 1.0 / (1.0 + np.exp(-p[:r]))
    c = np.tanh(p[r:2 * r])
    o = 1.0 / (1.0 + np.exp(-p[2 * r:]))
    for k in range(1, K + 1):
        want = o * c * (1.0 - g ** k)                      # s_k = c (1 - g^k) from s_0 = 0
        for b in range(B):
            np.testing.assert_allclose(rnn["feat"][b, k - 1], want, rtol=1e-12, atol=1e-15)


def test_the_state_remembers_tokens_before_the_previous_one():
    # greedy drafts forced by spikes in U: x_1 differs between the two runs, x_2 and x_3 do not
    B, K, V, r = 1, 3, 64, 4
    rng = np.random.default_rng(6)
    E = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    W = rng.normal(0, 0.01, (r, V)).astype(np.float32)
    Wc = rng.normal(0, 0.7, (3 * r, 2 * r)).astype(np.float32)
    cx = rng.normal(0, 0.5, (B, K, 3 * r)).astype(np.float32)
    base = np.zeros((B, K, V), np.float32)
    base[0, 1, 20] = 50.0
    base[0, 2, 30] = 50.0
    U1, U2 = base.copy(), base.copy()
    U1[0, 0, 5] = 50.0
    U2[0, 0, 6] = 50.0
    args = ([7], [K], np.zeros(1, np.float32))
    a = oracle.draft_rnn_sample(U1, E, W, Wc, cx, *args, seed=0, want_feat=True)
    b = oracle.draft_rnn_sample(U2, E, W, Wc, cx, *args, seed=0, want_feat=True)
    assert a["draft_tok"].tolist() == [[5, 20, 30]] and b["draft_tok"].tolist() == [[6, 20, 30]]
    np.testing.assert_array_equal(a["feat"][0, 0], b["feat"][0, 0])      # position 1: same anchor
    assert np.abs(a["feat"][0, 2] - b["feat"][0, 2]).max() > 1e-3         # position 3 recalls x_1
    # without the state feedback and with a gate that forgets, position 3 sees only x_2
    Wc0 = Wc.copy()
    Wc0[:, :r] = 0.0
    cx0 = cx.copy()
    cx0[..., :r] = -800.0
    a0 = oracle.draft_rnn_sample(U1, E, W, Wc0, cx0, *args, seed=0, want_feat=True)
    b0 = oracle.draft_rnn_sample(U2, E, W, Wc0, cx0, *args, seed=0, want_feat=True)
    np.testing.assert_array_equal(a0["feat"][0, 2], b0["feat"][0, 2])


def test_bf16_storage_matches_its_float_values():
    U, E, W, anchor, K_r, temp = _case(7)
    B, K, V = U.shape
    r = E.shape[1]
    rng = np.random.default_rng(8)
    Wc = rng.normal(0, 0.5, (3 * r, 2 * r)).astype(np.float32)
    cx = rng.normal(0, 1.0, (B, K, 3 * r)).astype(np.float32)

    def bits(x):
        return (x.view(np.uint32) >> 16).astype(np.uint16)

    def back(h):
        return (h.astype(np.uint32) << 16).view(np.float32)
    Ub, Eb, Wb, Cb = bits(U), bits(E), bits(W), bits(Wc)
    hb = oracle.draft_rnn_sample(Ub, Eb, Wb, Cb, cx, anchor, K_r, temp, seed=3, want_feat=True)
    hf = oracle.draft_rnn_sample(back(Ub), back(Eb), back(Wb), back(Cb), cx, anchor, K_r, temp, seed=3,
                                 want_feat=True)
    np.testing.assert_array_equal(hb["feat"], hf["feat"])    # the cell reads the same values
    assert hb["draft_tok"][:, 0].tolist() == hf["draft_tok"][:, 0].tolist() or hb["flags"][:, 0].any()


def test_errors():
    U, E, W, anchor, K_r, temp = _case(9)
    B, K, V = U.shape
    r = E.shape[1]
    with pytest.raises(ValueError):
        oracle.draft_rnn_sample(U, E, W, np.zeros((3 * r, r), np.float32), np.zeros((B, K, 3 * r), np.float32),
                                anchor, K_r, temp, seed=0)
    with pytest.raises(oracle.OracleError) as e:
        oracle.draft_rnn_sample(U, E, W, np.zeros((3 * r, 2 * r), np.float32), np.zeros((B, K, 3 * r), np.float32),
                                np.full(B, V, np.int32), K_r, temp, seed=0)
    assert e.value.name == "ERR_TOKEN_RANGE"

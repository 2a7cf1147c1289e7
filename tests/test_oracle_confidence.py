"""Pins for the oracle's confidence head with its Markov term ("DSpark" S3.2.1; tutorial S8).

c_k = sigmoid(w_h . h_k + b + w_e . W1[x_{k-1}]) with x_0 the anchor: checked on one-hot
embedding rows (the dot picks one weight), with the Markov weight off (no token dependence),
at the sigmoid's fixed point and reflection, and for its dependence on x_{k-1} alone.
"""
import math

import numpy as np
import pytest

import oracle


def _sigmoid(s):
    return 1.0 / (1.0 + math.exp(-s))


def test_one_hot_rows_select_one_weight():
    V, rank = 6, 4
    E = np.zeros((V, rank), np.float32)
    for v in range(V):
        E[v, v % rank] = 1.0                      # token v embeds as unit vector e_{v mod 4}
    w = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    anchor = np.array([3, 0], np.int32)
    tok = np.array([[1, 2, 5], [4, 4, 0]], np.int32)
    h = np.array([[0.0, 0.25, -0.5], [1.0, 0.0, 0.0]], np.float32)
    c = oracle.draft_confidence(E, anchor, tok, [3, 3], h, w)
    # previous tokens: r0: 3, 1, 2 -> weights 0, -1, 2 ; r1: 0, 4, 4 -> 0.5, 0.5, 0.5
    want = [[_sigmoid(0.0 + 0.0), _sigmoid(0.25 - 1.0), _sigmoid(-0.5 + 2.0)],
            [_sigmoid(1.0 + 0.5), _sigmoid(0.5), _sigmoid(0.5)]]
    np.testing.assert_allclose(c, np.array(want, np.float32), rtol=0, atol=0)   # fp64 then one rounding
    assert c[0, 0] == 0.5


def test_zero_markov_weight_ignores_the_tokens():
    rng = np.random.default_rng(0)
    V, rank, B, K = 50, 16, 5, 4
    E = rng.normal(0, 1, (V, rank)).astype(np.float32)
    h = rng.normal(0, 2, (B, K)).astype(np.float32)
    K_r = np.array([4, 1, 2, 4, 3], np.int32)
    zero = np.zeros(rank, np.float32)
    c1 = oracle.draft_confidence(E, rng.integers(0, V, B), rng.integers(0, V, (B, K)), K_r, h, zero)
    c2 = oracle.draft_confidence(E, rng.integers(0, V, B), rng.integers(0, V, (B, K)), K_r, h, zero)
    np.testing.assert_array_equal(c1, c2)
    for r in range(B):
        for k in range(K):
            want = np.float32(_sigmoid(float(h[r, k]))) if k < K_r[r] else np.float32(0.0)
            assert c1[r, k] == want


def test_reflection_and_range():
    rng = np.random.default_rng(1)
    V, rank, B, K = 40, 8, 6, 5
    E = rng.normal(0, 1, (V, rank)).astype(np.float32)
    w = rng.normal(0, 1, rank).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    h = rng.normal(0, 3, (B, K)).astype(np.float32)
    K_r = np.full(B, K, np.int32)
    c = oracle.draft_confidence(E, anchor, tok, K_r, h, w).astype(np.float64)
    cneg = oracle.draft_confidence(-E, anchor, tok, K_r, -h, w).astype(np.float64)   # s -> -s
    np.testing.assert_allclose(c + cneg, 1.0, atol=1e-7)
    assert np.all((c > 0) & (c < 1))


def test_depends_on_the_previous_token_only():
    rng = np.random.default_rng(2)
    V, rank, K = 30, 8, 5
    E = rng.normal(0, 1, (V, rank)).astype(np.float32)
    w = rng.normal(0, 1, rank).astype(np.float32)
    h = rng.normal(0, 1, (1, K)).astype(np.float32)
    tok = rng.integers(0, V, (1, K)).astype(np.int32)
    base = oracle.draft_confidence(E, [7], tok, [K], h, w)
    for j in range(K):                       # change x_{j+1}: only c_{j+2} may move
        t2 = tok.copy()
        t2[0, j] = (t2[0, j] + 1) % V
        c2 = oracle.draft_confidence(E, [7], t2, [K], h, w)
        moved = np.nonzero(c2[0] != base[0])[0].tolist()
        assert set(moved) <= {j + 1}
    c3 = oracle.draft_confidence(E, [8], tok, [K], h, w)       # the anchor feeds position 1
    assert c3[0, 0] != base[0, 0] and (c3[0, 1:] == base[0, 1:]).all()


def test_bf16_embedding_table_matches_its_float_values():
    rng = np.random.default_rng(3)
    V, rank = 20, 8
    E = rng.normal(0, 1, (V, rank)).astype(np.float32)
    bits = (E.view(np.uint32) >> 16).astype(np.uint16)         # truncation: exactly representable values
    Ef = (bits.astype(np.uint32) << 16).view(np.float32)
    w = rng.normal(0, 1, rank).astype(np.float32)
    h = rng.normal(0, 1, (2, 3)).astype(np.float32)
    tok = rng.integers(0, V, (2, 3)).astype(np.int32)
    a = oracle.draft_confidence(bits, [1, 2], tok, [3, 3], h, w)
    b = oracle.draft_confidence(Ef, [1, 2], tok, [3, 3], h, w)
    np.testing.assert_array_equal(a, b)


def test_errors():
    E = np.zeros((4, 2), np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.draft_confidence(E, [4], np.zeros((1, 2), np.int32), [2], np.zeros((1, 2), np.float32),
                                np.zeros(2, np.float32))
    assert e.value.name == "ERR_TOKEN_RANGE"

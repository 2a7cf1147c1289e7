"""Pins for the oracle's scheduler variants.

- Capacity of the asynchronous scheduler ("DSpark" S5.2; tutorial S9): the early-stopping
  break is removed and the objective's global maximum along the greedy path is taken.
- Dynamic top-K admission (same sections): the current candidates, ranked by their current
  survival, fill the capacity fixed two steps earlier.
- Static threshold ("DSpark" S3.2.2, the prior methods it contrasts with; S4.3.3, Fig. 5).

Checked against hand-worked numbers, exhaustive search over every admissible length tuple,
Appendix A's retrospective lengths and output law, and an exact enumeration of the output law
of rejection-sampling verification under each scheduler (non-anticipation).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _theta(a, ell, sps):
    """Objective of S3.2.2 for a length tuple: (R + sum_r sum_{j<=ell_r} a_rj) * SPS(R + sum ell)."""
    R = len(ell)
    tau = R + sum(float(a[r][j]) for r in range(R) for j in range(ell[r]))
    return tau * sps[R + sum(ell)]


def _random_case(rng, trial):
    R = int(rng.integers(1, 4))
    K = int(rng.integers(1, 4))
    K_r = rng.integers(1, K + 1, R)
    conf = rng.uniform(0.05, 1.0, (R, K)).astype(np.float32)
    if trial % 4 == 0:
        conf[0, -1] = 0.0                      # a zero survival is not a candidate
    n = R * (K + 1) + 2
    kind = trial % 3
    if kind == 0:     # smoothly falling step rate
        sps = np.array([0.0] + [1.0 / (1 + b / rng.uniform(1, 6)) for b in range(1, n)])
    elif kind == 1:   # jagged
        sps = np.concatenate([[0.0], rng.uniform(0.2, 1.0, n - 1)])
    else:             # plateaus with cliffs (graph-bucket sawtooth)
        step = int(rng.integers(1, 4))
        sps = np.array([0.0] + [1.0 / (1 + ((b + step - 1) // step) * step / rng.uniform(2, 8))
                                for b in range(1, n)])
    return R, K, K_r, conf, sps


def _admissible(a, K_r):
    """Every length tuple within the candidate pool {(r, j) : a_rj > 0} (a prefix per request)."""
    n_pos = [int((a[r, :K_r[r]] > 0).sum()) for r in range(len(K_r))]
    return list(itertools.product(*[range(n + 1) for n in n_pos]))


# ---------------------------------------------------------------------------
# capacity: global maximum of Theta without the early stop
# ---------------------------------------------------------------------------
def test_capacity_crosses_an_sps_cliff_hand_worked():
    # One request, four confident drafts; SPS drops from 1.0 to 0.6 after two verify tokens.
    # a = 0.9, 0.81, 0.729, 0.6561; Theta_0..4 = 1.0, 1.9, 1.626, 2.0634, 2.45706.
    conf = np.full((1, 4), 0.9, np.float32)
    sps = np.array([0.0, 1.0, 1.0, 0.6, 0.6, 0.6])
    cap = oracle.schedule_capacity(conf, [4], sps)
    assert cap["capacity"] == 4
    assert cap["theta_best"] == pytest.approx(2.45706, rel=1e-6)
    assert cap["ell"].tolist() == [4]
    assert cap["tgt_off"].tolist() == [0, 5]
    # Algorithm 1 stops at the dip after one token
    a1 = oracle.schedule_survival(conf, [4], sps)
    assert a1["ell"].tolist() == [1]
    assert a1["theta_best"] == pytest.approx(1.9, rel=1e-6)


def test_capacity_reproduces_appendix_a_retrospective_lengths():
    g = json.load(open(os.path.join(GOLDEN, "appendix_a.json")))
    sps = np.zeros(4)
    for k, v in g["sps"].items():
        sps[int(k)] = v
    for case in g["cases"]:
        conf = np.array([[g["a1"], case["c2"]]], np.float32)
        cap = oracle.schedule_capacity(conf, [2], sps)
        assert cap["ell"].tolist() == [case["retrospective_ell"]]
        assert cap["theta_best"] == pytest.approx(max(g["theta0"], case["theta2"]), rel=1e-6)


def test_capacity_is_the_global_maximum_exhaustive():
    rng = np.random.default_rng(10)
    crossed = 0
    for trial in range(300):
        R, K, K_r, conf, sps = _random_case(rng, trial)
        cap = oracle.schedule_capacity(conf, K_r, sps)
        a = cap["survival"].astype(np.float64)
        tuples = _admissible(a, K_r)
        thetas = {t: _theta(a, t, sps) for t in tuples}
        gmax = max(thetas.values())
        ell = cap["ell"].tolist()
        assert all(0 <= ell[r] <= K_r[r] for r in range(R))
        assert sum(ell) == cap["capacity"]
        assert cap["theta_best"] == pytest.approx(gmax, rel=1e-9)
        assert _theta(a, ell, sps) == pytest.approx(gmax, rel=1e-9)
        # the first maximum: no admissible tuple with fewer verified tokens reaches it
        for t, th in thetas.items():
            if sum(t) < cap["capacity"]:
                assert th < gmax * (1 - 1e-9)
        alg1 = oracle.schedule_survival(conf, K_r, sps)
        assert alg1["n_admitted"] <= cap["capacity"]
        crossed += alg1["n_admitted"] < cap["capacity"]
    assert crossed > 20       # the jagged curves do trap the early stop


def test_capacity_errors():
    conf = np.full((2, 3), 0.5, np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_capacity(conf, [3, 3], np.ones(8))          # needs R + N + 1 = 9 entries
    assert e.value.name == "ERR_SPS_TOO_SHORT"
    bad = conf.copy()
    bad[0, 1] = np.nan
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_capacity(bad, [3, 3], np.ones(9))
    assert e.value.name == "ERR_CONFIDENCE"


# ---------------------------------------------------------------------------
# top-K admission
# ---------------------------------------------------------------------------
def test_topk_hand_worked():
    # survivals: r0 = 0.9, 0.72, 0.36; r1 = 0.6, 0.54, 0.486
    # ranking: (r0,1) .9, (r0,2) .72, (r1,1) .6, (r1,2) .54, (r1,3) .486, (r0,3) .36
    conf = np.array([[0.9, 0.8, 0.5], [0.6, 0.9, 0.9]], np.float32)
    want = {0: [0, 0], 1: [1, 0], 2: [2, 0], 3: [2, 1], 4: [2, 2], 5: [2, 3], 6: [3, 3], 9: [3, 3]}
    for k, ell in want.items():
        out = oracle.schedule_topk(conf, [3, 3], k)
        assert out["ell"].tolist() == ell
        assert out["n_admitted"] == min(k, 6)
        assert out["tgt_off"].tolist() == [0, ell[0] + 1, ell[0] + ell[1] + 2]


def test_topk_maximises_expected_accepts_for_its_size_exhaustive():
    # S3.2.2: for a fixed verify batch the greedy top set maximises tau
    rng = np.random.default_rng(11)
    for trial in range(200):
        R, K, K_r, conf, _ = _random_case(rng, trial)
        a = oracle.schedule_topk(conf, K_r, 0)["survival"].astype(np.float64)
        tuples = _admissible(a, K_r)
        N = int(sum((a[r, :K_r[r]] > 0).sum() for r in range(R)))
        for k in range(0, N + 2):
            out = oracle.schedule_topk(conf, K_r, k)
            ell = out["ell"].tolist()
            size = min(k, N)
            assert sum(ell) == size == out["n_admitted"]
            assert all(ell[r] <= K_r[r] for r in range(R))
            assert all(a[r, j] > 0 for r in range(R) for j in range(ell[r]))
            best = max(sum(a[r, j] for r in range(R) for j in range(t[r])) for t in tuples if sum(t) == size)
            got = sum(a[r, j] for r in range(R) for j in range(ell[r]))
            assert got == pytest.approx(best, rel=1e-12, abs=1e-15)


def test_topk_at_the_early_stop_size_is_algorithm_1():
    rng = np.random.default_rng(12)
    for trial in range(100):
        R, K, K_r, conf, sps = _random_case(rng, trial)
        alg1 = oracle.schedule_survival(conf, K_r, sps)
        out = oracle.schedule_topk(conf, K_r, alg1["n_admitted"])
        assert out["ell"].tolist() == alg1["ell"].tolist()


# ---------------------------------------------------------------------------
# non-anticipation: exact output law of verification under each scheduler
# ---------------------------------------------------------------------------
def _emission_law(x, p, q, ell):
    """Exact law of the first two emitted tokens of one request (rejection sampling, S2.1).

    x: draft tokens; p[j], q[j]: target / draft rows at position j+1 given x[:j]; ell: length.
    Returns (P(Y1 = v) [V], P(Y1 = y, Y2 = v) [V, V]); Y2 exists only when x_1 is accepted.
    """
    V = len(p[0])
    y1, y12 = np.zeros(V), np.zeros((V, V))
    if ell == 0:
        return p[0].copy(), y12
    acc1 = min(1.0, p[0][x[0]] / q[0][x[0]])
    res = np.maximum(0.0, p[0] - q[0])
    if res.sum() > 0:
        y1 += (1 - acc1) * res / res.sum()
    y1[x[0]] += acc1
    if ell == 1:
        y12[x[0]] += acc1 * p[1]                          # bonus row after the accepted token
    else:
        acc2 = min(1.0, p[1][x[1]] / q[1][x[1]])
        res2 = np.maximum(0.0, p[1] - q[1])
        if res2.sum() > 0:
            y12[x[0]] += acc1 * (1 - acc2) * res2 / res2.sum()
        y12[x[0], x[1]] += acc1 * acc2
    return y1, y12


def _markov_system(seed, V):
    """Two requests, two positions; rows and the position-2 confidence depend on x_1."""
    rng = np.random.default_rng(seed)

    def row():
        w = rng.uniform(0.05, 1.0, V)
        return w / w.sum()
    reqs = []
    for _ in range(2):
        reqs.append(dict(p1=row(), q1=row(), p2=[row() for _ in range(V)], q2=[row() for _ in range(V)],
                         c1=float(rng.uniform(0.3, 0.95)), c2=[float(rng.uniform(0.0, 1.0)) for _ in range(V)]))
    return reqs


def _law_under(schedule, reqs, V):
    """Accumulate each request's emitted-token law over every draft draw."""
    laws = [(np.zeros(V), np.zeros((V, V))) for _ in reqs]
    for xs in itertools.product(range(V), repeat=4):
        x = [xs[0:2], xs[2:4]]
        prob = 1.0
        conf = np.zeros((2, 2), np.float32)
        for r, q in enumerate(reqs):
            prob *= q["q1"][x[r][0]] * q["q2"][x[r][0]][x[r][1]]
            conf[r] = [q["c1"], q["c2"][x[r][0]]]
        ell = schedule(conf)
        for r, q in enumerate(reqs):
            y1, y12 = _emission_law(x[r], [q["p1"], q["p2"][x[r][0]]], [q["q1"], q["q2"][x[r][0]]], ell[r])
            laws[r][0][:] += prob * y1
            laws[r][1][:] += prob * y12
    return laws


def test_topk_with_a_fixed_capacity_recovers_the_target_law():
    V = 3
    for seed in range(3):
        reqs = _markov_system(seed, V)
        for capacity in range(0, 5):
            laws = _law_under(lambda c: oracle.schedule_topk(c, [2, 2], capacity)["ell"], reqs, V)
            for r, q in enumerate(reqs):
                y1, y12 = laws[r]
                np.testing.assert_allclose(y1, q["p1"], atol=1e-12)
                for y in range(V):
                    m = y12[y].sum()
                    if m > 1e-12:
                        np.testing.assert_allclose(y12[y] / m, q["p2"][y], atol=1e-12)


def test_retrospective_search_on_live_confidences_leaks_appendix_a():
    # The capacity search applied to the CURRENT step's confidences is Appendix A's
    # retrospective scheduler: the output law moves from (0.7, 0.3) to (0.85, 0.15).
    g = json.load(open(os.path.join(GOLDEN, "appendix_a.json")))
    ex = g["two_token_example"]
    sps = np.zeros(4)
    for k, v in g["sps"].items():
        sps[int(k)] = v
    p1, q1 = np.array(ex["p_target"]), np.array(ex["p_draft"])
    c2 = {0: 0.9, 1: 0.0}                                   # A -> confident, B -> hopeless
    out = {"retro": np.zeros(2), "alg1": np.zeros(2), "topk": np.zeros(2)}
    for x1 in (0, 1):
        conf = np.array([[g["a1"], c2[x1]]], np.float32)
        ells = {"retro": oracle.schedule_capacity(conf, [2], sps)["ell"][0],
                "alg1": oracle.schedule_survival(conf, [2], sps)["ell"][0],
                "topk": oracle.schedule_topk(conf, [2], 1)["ell"][0]}
        for name, ell in ells.items():
            y1, _ = _emission_law([x1, 0], [p1, p1], [q1, q1], int(ell))
            out[name] += q1[x1] * y1
    np.testing.assert_allclose(out["retro"], ex["retrospective_output"], atol=1e-12)
    np.testing.assert_allclose(out["alg1"], ex["lossless_output"], atol=1e-12)
    np.testing.assert_allclose(out["topk"], ex["lossless_output"], atol=1e-12)


# ---------------------------------------------------------------------------
# static threshold
# ---------------------------------------------------------------------------
def test_threshold_hand_worked():
    conf = np.array([[0.9, 0.8, 0.5], [0.6, 0.9, 0.9]], np.float32)
    # confidences >= 0.7: r0 passes 0.9, 0.8 then stops at 0.5; r1 stops at once
    assert oracle.schedule_threshold(conf, [3, 3], 0.7)["ell"].tolist() == [2, 0]
    # equality passes
    assert oracle.schedule_threshold(conf, [3, 3], np.float32(0.6))["ell"].tolist() == [2, 3]
    # survivals 0.9, 0.72, 0.36 / 0.6, 0.54, 0.486 against 0.5
    out = oracle.schedule_threshold(conf, [3, 3], 0.5, oracle.THRESHOLD_SURVIVAL)
    assert out["ell"].tolist() == [2, 2]
    assert out["tgt_off"].tolist() == [0, 3, 6]
    # K_r caps the prefix
    assert oracle.schedule_threshold(conf, [1, 2], 0.0)["ell"].tolist() == [1, 2]


def test_threshold_limits_match_algorithm_1_empty_system():
    rng = np.random.default_rng(13)
    conf = rng.uniform(0.0, 1.0, (30, 6)).astype(np.float32)
    conf[4, 2] = 0.0                      # zero survival from position 3 on
    K_r = rng.integers(1, 7, 30)
    K_r[4] = 6
    sps = np.array([0.0] + [1.0] * 300)  # non-decreasing SPS: Algorithm 1 admits every candidate
    alg1 = oracle.schedule_survival(conf, K_r, sps)
    for mode in (oracle.THRESHOLD_CONFIDENCE, oracle.THRESHOLD_SURVIVAL):
        for theta in (0.0, -1.0):
            out = oracle.schedule_threshold(conf, K_r, theta, mode)
            assert out["ell"].tolist() == alg1["ell"].tolist()
            assert out["tgt_off"].tolist() == alg1["tgt_off"].tolist()
        assert oracle.schedule_threshold(conf, K_r, 1.0001, mode)["ell"].tolist() == [0] * 30
    assert alg1["ell"][4] == 2


def test_threshold_lengths_fall_as_the_threshold_rises():
    rng = np.random.default_rng(14)
    conf = rng.uniform(0.2, 1.0, (50, 7)).astype(np.float32)
    K_r = rng.integers(1, 8, 50)
    for mode in (oracle.THRESHOLD_CONFIDENCE, oracle.THRESHOLD_SURVIVAL):
        prev = None
        for theta in np.linspace(0.0, 1.0, 21):
            ell = oracle.schedule_threshold(conf, K_r, theta, mode)["ell"]
            if prev is not None:
                assert np.all(ell <= prev)
            prev = ell
    # on the same threshold the survival cut is never longer than the confidence cut
    for theta in (0.3, 0.5, 0.8):
        c = oracle.schedule_threshold(conf, K_r, theta, oracle.THRESHOLD_CONFIDENCE)["ell"]
        s = oracle.schedule_threshold(conf, K_r, theta, oracle.THRESHOLD_SURVIVAL)["ell"]
        assert np.all(s <= c)


def test_threshold_errors():
    conf = np.full((2, 3), 0.5, np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_threshold(conf, [3, 3], np.nan)
    assert e.value.name == "ERR_CONFIDENCE"
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_threshold(conf, [3, 4], 0.5)
    assert e.value.name == "ERR_LENGTHS"

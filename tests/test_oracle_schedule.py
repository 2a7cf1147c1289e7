"""Pins for the oracle's hardware-aware prefix scheduler ("DSpark", S3.2.2, Algorithm 1).

Checked against the pages' printed worked numbers (Appendix A; the two-request
example of the paperglide digest), exhaustive search over every admissible
length tuple on tiny inputs, the empty-system limit, the marginal-threshold
form of the comparison, and the survival-product invariants.
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


def test_appendix_a_counterexample_numbers():
    g = json.load(open(os.path.join(GOLDEN, "appendix_a.json")))
    sps = np.zeros(4)
    for k, v in g["sps"].items():
        sps[int(k)] = v
    for case in g["cases"]:
        c1 = g["a1"]
        conf = np.array([[c1, case["c2"]]], np.float32)
        out = oracle.schedule_survival(conf, [2], sps)
        assert out["ell"].tolist() == [case["algorithm1_ell"]]
        assert out["theta_best"] == pytest.approx(g["theta0"], abs=1e-12)
        assert out["B_star"] == 1
        a = out["survival"][0]
        assert a[0] == pytest.approx(g["a1"], rel=1e-7)
        assert a[1] == pytest.approx(case["a2"], rel=1e-6)
        # the printed objective values along the path
        assert _theta([a], [1], sps) == pytest.approx(g["theta1"], rel=1e-6)
        assert _theta([a], [2], sps) == pytest.approx(case["theta2"], rel=1e-6)
        # a retrospective search (argmax over every prefix length) picks the printed length
        best = max(range(3), key=lambda L: (_theta([a], [L], sps), -L))
        assert best == case["retrospective_ell"]


def test_two_request_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "two_request_example.json")))
    conf = np.array(g["conf"], np.float32)
    sps = np.array([0, 1, 1, 1, 1, 1, 0.9, 0.9, 0.9], np.float64)
    out = oracle.schedule_survival(conf, [3, 3], sps)
    np.testing.assert_allclose(out["survival"], np.array(g["survival"]), rtol=1e-6)
    B = conf.shape[0]
    pairs = [[int(i) % B + 1, int(i) // B + 1] for i in out["order"]]
    assert pairs == g["sorted_pairs_1based"]
    assert out["ell"].tolist() == g["ell"]
    assert out["B_star"] == g["B"]
    assert out["tau_star"] == pytest.approx(2 + g["printed_tau"], abs=1e-6)   # fp32 confidences
    assert out["tgt_off"].tolist() == [0, 3, 5]


def test_exhaustive_search_tiny():
    rng = np.random.default_rng(0)
    n_unimodal = 0
    for trial in range(300):
        R = int(rng.integers(1, 4))
        K = int(rng.integers(1, 4))
        K_r = rng.integers(1, K + 1, R)
        conf = rng.uniform(0.05, 1.0, (R, K)).astype(np.float32)
        kind = trial % 3
        if kind == 0:     # smoothly falling step rate
            sps = np.array([0.0] + [1.0 / (1 + b / rng.uniform(1, 6)) for b in range(1, R * (K + 1) + 2)])
        elif kind == 1:   # jagged
            sps = np.concatenate([[0.0], rng.uniform(0.2, 1.0, R * (K + 1) + 1)])
        else:             # flat then falling
            knee = rng.integers(R, R * (K + 1) + 1)
            sps = np.array([0.0] + [1.0 if b <= knee else knee / b for b in range(1, R * (K + 1) + 2)])
        out = oracle.schedule_survival(conf, K_r, sps)
        a = out["survival"].astype(np.float64)
        # every admissible tuple
        tuples = list(itertools.product(*[range(int(k) + 1) for k in K_r]))
        thetas = [_theta(a, t, sps) for t in tuples]
        gmax = max(thetas)
        # the greedy path by survival probability: prefixes of the global sort
        order = sorted([(a[r, j], j, r) for r in range(R) for j in range(int(K_r[r]))],
                       key=lambda t: (-t[0], t[1], t[2]))
        path, cur = [], [0] * R
        path.append(_theta(a, cur, sps))
        for _, j, r in order:
            cur[r] += 1
            path.append(_theta(a, cur, sps))
        # S3.2.2: for fixed B the greedy top-(B-R) set maximises tau, so the best point on the
        # greedy path is the global optimum
        assert max(path) == pytest.approx(gmax, rel=1e-9)
        # the oracle's schedule is admissible and its reported objective is its own value
        ell = out["ell"].tolist()
        assert all(0 <= ell[r] <= K_r[r] for r in range(R))
        assert out["theta_best"] == pytest.approx(_theta(a, ell, sps), rel=1e-9)
        assert out["theta_best"] >= R * sps[R] - 1e-12
        # early stop: the returned point is the last strict rise before the first decline
        stop = next((i for i in range(1, len(path)) if not path[i] > path[i - 1] * (1 + 1e-12)), len(path))
        assert out["B_star"] == R + stop - 1 or abs(path[stop] - path[stop - 1]) < 1e-9 * path[stop - 1]
        # unimodal along the path -> the early stop finds the global maximum
        diffs = np.diff(path)
        signs = np.sign(diffs[np.abs(diffs) > 1e-12])
        unimodal = not np.any((signs[:-1] < 0) & (signs[1:] > 0)) if len(signs) > 1 else True
        if unimodal:
            n_unimodal += 1
            assert out["theta_best"] == pytest.approx(gmax, rel=1e-9)
    assert n_unimodal > 50


def test_empty_system_limit_admits_everything():
    # non-decreasing SPS: every admitted token only adds to tau, so all candidates are verified
    rng = np.random.default_rng(1)
    conf = rng.uniform(0.1, 1.0, (6, 5)).astype(np.float32)
    K_r = np.array([5, 1, 3, 5, 2, 4])
    sps = np.array([0.0] + [min(b, 12) / 12 for b in range(1, 40)])
    out = oracle.schedule_survival(conf, K_r, sps)
    assert out["ell"].tolist() == K_r.tolist()
    assert out["tgt_off"].tolist() == np.concatenate([[0], np.cumsum(K_r + 1)]).tolist()


def test_marginal_threshold_form():
    # continue iff a > tau * (SPS(B) / SPS(B+1) - 1)  (algebra of the Theta comparison)
    rng = np.random.default_rng(2)
    for _ in range(50):
        R, K = 5, 4
        conf = rng.uniform(0.3, 1.0, (R, K)).astype(np.float32)
        sps = np.array([0.0] + [1.0 / (1 + b / 6.0) for b in range(1, R * (K + 1) + 2)])
        out = oracle.schedule_survival(conf, [K] * R, sps)
        a = out["survival"]
        order = out["order"]
        tau, Bt = float(R), R
        for i, idx in enumerate(order):
            j, r = divmod(int(idx), R)
            aij = float(a[r, j])
            go = aij > tau * (sps[Bt] / sps[Bt + 1] - 1.0)
            if i < out["n_admitted"]:
                assert go
                tau += aij
                Bt += 1
            else:
                assert not go
                break


def test_survival_products_and_prefix_order():
    rng = np.random.default_rng(3)
    conf = rng.uniform(0.0, 1.0, (40, 7)).astype(np.float32)
    conf[3, 2] = 1.0      # equal consecutive survival values
    conf[3, 3] = 1.0
    conf[5, 4] = 0.0      # zero survival: not a candidate
    K_r = rng.integers(1, 8, 40)
    K_r[3] = 7
    K_r[5] = 7
    sps = np.array([0.0] + [1.0] * 400)
    out = oracle.schedule_survival(conf, K_r, sps)
    a = out["survival"]
    for r in range(40):
        prod = np.float32(1.0)
        for j in range(K_r[r]):
            prod = np.float32(prod * conf[r, j])
            assert a[r, j] == prod                      # sequential fp32 product
            if j:
                assert a[r, j] <= a[r, j - 1]           # non-increasing
    assert a[3, 2] == a[3, 1] == a[3, 3]
    pos = {int(i): n for n, i in enumerate(out["order"])}
    for r in range(40):
        for j in range(1, K_r[r]):
            i0, i1 = (j - 1) * 40 + r, j * 40 + r
            if i1 in pos:
                assert pos[i0] < pos[i1]                # (r, j) ranks before (r, j + 1)
    assert (4 * 40 + 5) not in pos and (5 * 40 + 5) not in pos
    assert out["n_cand"] == sum(int((a[r, :K_r[r]] > 0).sum()) for r in range(40))


def test_ties_rank_earlier_position_then_lower_request():
    conf = np.array([[0.5, 1.0], [0.5, 1.0]], np.float32)
    sps = np.ones(8)
    out = oracle.schedule_survival(conf, [2, 2], sps)
    # all four survivals equal 0.5: order (r0,j1) (r1,j1) (r0,j2) (r1,j2)
    assert out["order"].tolist() == [0, 1, 2, 3]


def test_errors():
    conf = np.full((2, 3), 0.5, np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_survival(conf, [3, 3], np.ones(8))          # needs R + N + 1 = 9 entries
    assert e.value.name == "ERR_SPS_TOO_SHORT"
    oracle.schedule_survival(conf, [3, 3], np.ones(9))
    bad = conf.copy()
    bad[1, 0] = 1.5
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_survival(bad, [3, 3], np.ones(9))
    assert e.value.name == "ERR_CONFIDENCE"
    with pytest.raises(oracle.OracleError) as e:
        oracle.schedule_survival(conf, [0, 3], np.ones(9))
    assert e.value.name == "ERR_LENGTHS"

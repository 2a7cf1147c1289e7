"""GPU scheduler variants vs the CPU oracle, bit for bit, through the C ABI.

The capacity of the asynchronous scheduler, dynamic top-K admission and the static
thresholds ("DSpark" S5.2 and S3.2.2 / S4.3.3) on every benchmark configuration at full
size, and on random small cases with ties, zero confidences and ragged lengths.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(name):
    cfg = wl.CONFIGS[name]
    return wl.confidences(cfg, "cpu"), wl.request_params(cfg, "cpu")["K_r"]


def _random_case(rng, trial):
    B = int(rng.integers(1, 300))
    K = int(rng.integers(1, 17))
    conf = rng.uniform(0, 1, (B, K)).astype(np.float32)
    conf[rng.uniform(size=(B, K)) < 0.05] = 1.0          # equal survival values: tie order
    conf[rng.uniform(size=(B, K)) < 0.02] = 0.0          # zero survival: not a candidate
    K_r = rng.integers(1, K + 1, B).astype(np.int32)
    n = B * (K + 1) + 2
    if trial % 3 == 0:
        sps = np.concatenate([[0.0], rng.uniform(0.5, 1.0, n - 1)])     # jagged
    elif trial % 3 == 1:
        step = int(rng.integers(2, 64))
        sps = np.array([0.0] + [1.0 / (1 + ((b + step - 1) // step) * step / 300.0) for b in range(1, n)])
    else:
        sps = np.concatenate([[0.0], 1.0 / (1.0 + np.arange(1, n) / rng.uniform(5, 500))])
    return conf, K_r, sps


def _check_capacity(conf, K_r, sps):
    o = oracle.schedule_capacity(conf, K_r, sps)
    g = ds.schedule_capacity(torch.from_numpy(np.ascontiguousarray(conf)).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(K_r, dtype=np.int32)).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(sps)).to(DEV))
    assert ds.check(g["status"]) == "DSPARK_OK"
    assert g["capacity"].item() == o["capacity"]
    assert g["theta_best"].item() == o["theta_best"]              # bit-exact fp64
    np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
    np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])
    return o


def _check_topk(conf, K_r, capacity):
    o = oracle.schedule_topk(conf, K_r, capacity)
    cap = torch.tensor([capacity], dtype=torch.int32, device=DEV)
    g = ds.schedule_topk(torch.from_numpy(np.ascontiguousarray(conf)).to(DEV),
                         torch.from_numpy(np.ascontiguousarray(K_r, dtype=np.int32)).to(DEV), cap)
    assert ds.check(g["status"]) == "DSPARK_OK"
    np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
    np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])
    np.testing.assert_array_equal(g["survival"].cpu().numpy(), o["survival"])
    assert g["b_star"].item() == conf.shape[0] + o["n_admitted"]
    return o


def _check_threshold(conf, K_r, theta, mode):
    o = oracle.schedule_threshold(conf, K_r, theta, mode)
    g = ds.schedule_threshold(torch.from_numpy(np.ascontiguousarray(conf)).to(DEV),
                              torch.from_numpy(np.ascontiguousarray(K_r, dtype=np.int32)).to(DEV), theta, mode)
    assert ds.check(g["status"]) == "DSPARK_OK"
    np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
    np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])
    np.testing.assert_array_equal(g["survival"].cpu().numpy(), o["survival"])
    assert g["b_star"].item() == int(o["tgt_off"][-1])


@pytest.mark.parametrize("name", list(wl.CONFIGS))
@pytest.mark.parametrize("variant", ["literal", "step"])
def test_capacity_full_size(name, variant):
    conf, K_r = _inputs(name)
    _check_capacity(conf.numpy(), K_r.numpy(), wl.sps_table(wl.CONFIGS[name], variant).numpy())


@pytest.mark.parametrize("name", list(wl.CONFIGS))
def test_topk_full_size(name):
    conf, K_r = _inputs(name)
    c, k = conf.numpy(), K_r.numpy()
    N = oracle.schedule_topk(c, k, 0)["n_cand"]
    alg1 = oracle.schedule_survival(c, k, wl.sps_table(wl.CONFIGS[name], "step").numpy())
    for capacity in sorted({0, 1, alg1["n_admitted"], N // 3, N - 1, N, N + 17}):
        if capacity >= 0:
            _check_topk(c, k, capacity)


@pytest.mark.parametrize("name", list(wl.CONFIGS))
def test_asynchronous_pipeline_on_device(name):
    # capacity from an earlier step's confidences feeds the top-K of the current step on the
    # device, with no host round trip in between
    cfg = wl.CONFIGS[name]
    conf, K_r = _inputs(name)
    old = torch.roll(conf, shifts=1, dims=0)                 # another step's confidences
    sps = wl.sps_table(cfg, "step")
    cap = ds.schedule_capacity(old.to(DEV), K_r.to(DEV), sps.to(DEV))
    g = ds.schedule_topk(conf.to(DEV), K_r.to(DEV), cap["capacity"], status=cap["status"])
    assert ds.check(g["status"]) == "DSPARK_OK"
    o_cap = oracle.schedule_capacity(old.numpy(), K_r.numpy(), sps.numpy())
    o = oracle.schedule_topk(conf.numpy(), K_r.numpy(), o_cap["capacity"])
    np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
    np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])


@pytest.mark.parametrize("name", list(wl.CONFIGS))
def test_threshold_full_size(name):
    conf, K_r = _inputs(name)
    c, k = conf.numpy(), K_r.numpy()
    for mode in (ds.THRESHOLD_CONFIDENCE, ds.THRESHOLD_SURVIVAL):
        for theta in (-1.0, 0.0, 0.3, 0.5, 0.8, float(c[0, 0]), 1.0, 1.5):
            _check_threshold(c, k, theta, mode)


def test_variants_random_small():
    rng = np.random.default_rng(5)
    for trial in range(30):
        conf, K_r, sps = _random_case(rng, trial)
        cap = _check_capacity(conf, K_r, sps)
        N = oracle.schedule_topk(conf, K_r, 0)["n_cand"]
        for capacity in {0, cap["capacity"], N // 2, N + 1}:
            _check_topk(conf, K_r, capacity)
        for mode in (ds.THRESHOLD_CONFIDENCE, ds.THRESHOLD_SURVIVAL):
            for theta in (0.0, 0.4, float(conf[0, 0])):
                _check_threshold(conf, K_r, theta, mode)


def test_variant_device_errors():
    conf = torch.full((4, 3), 0.5, device=DEV)
    K_r = torch.full((4,), 3, dtype=torch.int32, device=DEV)
    g = ds.schedule_topk(conf, K_r, torch.tensor([-1], dtype=torch.int32, device=DEV))
    assert ds.check(g["status"]) == "DSPARK_ERR_LENGTHS"
    g = ds.schedule_capacity(conf, K_r, torch.ones(16, dtype=torch.float64, device=DEV))   # needs 4 + 12 + 1
    assert ds.check(g["status"]) == "DSPARK_ERR_SPS_TOO_SHORT"
    bad = conf.clone()
    bad[2, 1] = 1.5
    g = ds.schedule_threshold(bad, K_r, 0.5)
    assert ds.check(g["status"]) == "DSPARK_ERR_CONFIDENCE"
    g = ds.schedule_threshold(conf, torch.tensor([3, 0, 3, 3], dtype=torch.int32, device=DEV), 0.5)
    assert ds.check(g["status"]) == "DSPARK_ERR_LENGTHS"
    with pytest.raises(ds.DsparkError):
        ds.schedule_threshold(conf, K_r, float("nan"))

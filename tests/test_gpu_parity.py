"""GPU path vs CPU oracle, element by element, through the C ABI.

Small cases span several tiles (requests across 128-row tiles, vocabularies
with a ragged last 64-wide tile), every temperature mode and both draft kernel
paths; the benchmark configurations are checked at full size on sampled
requests (the oracle recomputes those requests one by one with their own
request ids).  Tokens and lengths are bit-exact outside the oracle's near-tie
flags; normalisers are within 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_gb300 as ds
from speculative_decoding_draft_gb300 import workloads as wl

from parity_helpers import comparable, compare_draft, compare_verify, host, oracle_draft, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _to(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


def _run_draft(g, seed, **kw):
    out = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], seed, **kw)
    assert ds.check(out["status"]) == "DSPARK_OK"
    return out


# ---------------------------------------------------------------------------
# schedule: every benchmark configuration at full size, both SPS readings
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(wl.CONFIGS))
@pytest.mark.parametrize("variant", ["literal", "step"])
def test_schedule_full_size(name, variant):
    cfg = wl.CONFIGS[name]
    conf = wl.confidences(cfg, "cpu")
    K_r = wl.request_params(cfg, "cpu")["K_r"]
    sps = wl.sps_table(cfg, variant)
    o = oracle.schedule_survival(conf.numpy(), K_r.numpy(), sps.numpy())
    g = ds.schedule_survival(conf.to(DEV), K_r.to(DEV), sps.to(DEV))
    assert ds.check(g["status"]) == "DSPARK_OK"
    np.testing.assert_array_equal(g["survival"].cpu().numpy(), o["survival"])
    np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
    np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])
    assert g["theta_best"].item() == o["theta_best"]           # bit-exact fp64
    assert g["b_star"].item() == o["B_star"]


def test_schedule_worked_example_and_ties():
    conf = torch.tensor([[0.9, 0.6, 0.2], [0.8, 0.5, 0.1]])
    sps = torch.tensor([0, 1, 1, 1, 1, 1, 0.9, 0.9, 0.9], dtype=torch.float64)
    g = ds.schedule_survival(conf.to(DEV), torch.tensor([3, 3], dtype=torch.int32, device=DEV), sps.to(DEV))
    assert g["ell"].tolist() == [2, 1] and g["b_star"].item() == 5
    # equal survivals: earlier positions first (so the prefix property holds)
    conf = torch.tensor([[0.5, 1.0, 1.0], [0.5, 1.0, 0.4]])
    sps = torch.ones(9, dtype=torch.float64)
    sps[7:] = 0.5
    g = ds.schedule_survival(conf.to(DEV), torch.tensor([3, 3], dtype=torch.int32, device=DEV), sps.to(DEV))
    o = oracle.schedule_survival(conf.numpy(), [3, 3], sps.numpy())
    assert g["ell"].tolist() == o["ell"].tolist()


def test_schedule_random_small():
    rng = np.random.default_rng(0)
    for trial in range(40):
        B = int(rng.integers(1, 300))
        K = int(rng.integers(1, 17))
        conf = rng.uniform(0, 1, (B, K)).astype(np.float32)
        conf[rng.uniform(size=(B, K)) < 0.05] = 1.0
        conf[rng.uniform(size=(B, K)) < 0.02] = 0.0
        K_r = rng.integers(1, K + 1, B).astype(np.int32)
        n = B * (K + 1) + 2
        sps = np.concatenate([[0.0], 1.0 / (1.0 + np.arange(1, n) / rng.uniform(5, 500))])
        if trial % 3 == 0:
            sps = np.concatenate([[0.0], rng.uniform(0.5, 1.0, n - 1)])
        o = oracle.schedule_survival(conf, K_r, sps)
        g = ds.schedule_survival(torch.from_numpy(conf).to(DEV), torch.from_numpy(K_r).to(DEV),
                                 torch.from_numpy(sps).to(DEV))
        assert ds.check(g["status"]) == "DSPARK_OK"
        np.testing.assert_array_equal(g["ell"].cpu().numpy(), o["ell"])
        np.testing.assert_array_equal(g["tgt_off"].cpu().numpy(), o["tgt_off"])
        assert g["theta_best"].item() == o["theta_best"]


# ---------------------------------------------------------------------------
# draft: small cases through both kernel paths
# ---------------------------------------------------------------------------
DRAFT_CASES = {
    "tiny-fp32": (dict(name="tiny"), False),
    "bf16-tc-ragged": (dict(name="ragged", B=150, K_max=3, V=4104), False),
    "bf16-tc-qwen": (dict(name="qwen", B=40, K_max=4, V=2056), False),
    "bf16-tc-rank64": (dict(name="qwen", B=9, K_max=3, V=520, rank=64), False),
    "bf16-tc-single": (dict(name="qwen", B=1, K_max=1, V=1032), False),
    "bf16-tc-multiblock": (dict(name="qwen", B=64, K_max=2, V=64040), False),
    "bf16-tc-mixedF": (dict(name="ragged", B=150, K_max=2, V=64040), False),
    "bf16-simt-ragged": (dict(name="ragged", B=150, K_max=3, V=1048), True),
    "fp32-simt-oddV": (dict(name="tiny", B=5, K_max=4, V=1003, rank=7), False),
}


@pytest.mark.parametrize("case", list(DRAFT_CASES))
def test_draft_parity(case):
    kw, simt = DRAFT_CASES[case]
    cfg = wl.small_config(**kw)
    inp = wl.draft_inputs(cfg, "cpu")
    gpu = _run_draft(_to(inp), cfg.philox_seed, force_simt=simt)
    orc = oracle_draft(inp, cfg.philox_seed)
    n = compare_draft(gpu, orc, inp["K_r"].numpy(), cfg.dtype)
    assert n == comparable(orc["flags"], inp["K_r"].numpy())
    assert n >= 0.9 * int(inp["K_r"].sum())


def _pack_reference(W_bits, rank, V):
    # the packed layout as the header states it: block (c, t) = 64 rows of 128 bytes; row i
    # holds W[64c + i, 64t + 8 (u ^ (i & 7)) ...] in 16-byte unit u; columns past V are zero
    nb = (V + 63) // 64
    Wpad = np.zeros((rank, nb * 64), np.uint16)
    Wpad[:, :V] = W_bits
    out = np.zeros((rank // 64, nb, 64, 8, 8), np.uint16)
    for i in range(64):
        src = Wpad.reshape(rank // 64, 64, nb, 8, 8)[:, i]          # [c, t, unit, 8]
        perm = np.arange(8) ^ (i & 7)
        out[:, :, i] = src[:, :, perm]
    return out.reshape(-1)


@pytest.mark.parametrize("rank,V", [(256, 1032), (64, 4104), (128, 520)])
def test_pack_projection_layout(rank, V):
    W = (torch.randn(rank, V, device=DEV) * 0.1).to(torch.bfloat16)
    pk = ds.pack_projection(W)
    got = pk.data.cpu().numpy().view(np.uint16)
    want = _pack_reference(wl.bf16_bits(W), rank, V)
    assert got.shape == want.shape
    np.testing.assert_array_equal(got, want)


def test_draft_packed_equals_unpacked():
    # a pre-packed projection and the per-call packing into the workspace give identical bits
    cfg = wl.small_config("qwen", B=64, K_max=3, V=64040)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    a = _run_draft(g, 3)
    pk = ds.pack_projection(g["W"])
    b = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 3)
    assert ds.check(b["status"]) == "DSPARK_OK"
    assert torch.equal(a["draft_tok"], b["draft_tok"])
    assert torch.equal(a["draft_lse"], b["draft_lse"])
    K_r = g["K_r"].cpu()
    for r in range(cfg.B):
        k = int(K_r[r])
        assert torch.equal(a["draft_logits"][r, :k], b["draft_logits"][r, :k])
    # a packed projection cannot feed the CUDA-core path
    with pytest.raises(ds.DsparkError) as e:
        ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 3, force_simt=True)
    assert e.value.name == "DSPARK_ERR_UNSUPPORTED"


def test_draft_spare_sm_matches():
    # leaving one SM free changes only the split of the vocabulary over CTAs: the same
    # tokens and logits, normalisers equal up to the order of the partial sums
    cfg = wl.small_config("qwen", B=64, K_max=3, V=64040)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    pk = ds.pack_projection(g["W"])
    a = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 9)
    b = ds.draft_markov_sample(g["U"], g["E"], pk, g["anchor"], g["K_r"], g["temperature"], 9, spare_sm=True)
    assert ds.check(a["status"]) == "DSPARK_OK" and ds.check(b["status"]) == "DSPARK_OK"
    assert torch.equal(a["draft_tok"], b["draft_tok"])
    K_r = g["K_r"].cpu()
    for r in range(cfg.B):
        k = int(K_r[r])
        assert torch.equal(a["draft_logits"][r, :k], b["draft_logits"][r, :k])
        assert torch.allclose(a["draft_lse"][r, :k], b["draft_lse"][r, :k], rtol=1e-6, atol=0)


def test_draft_paths_agree():
    # the tensor-core and CUDA-core kernels sample the same tokens (fp32 rounding aside)
    cfg = wl.small_config("ragged", B=130, K_max=3, V=2048)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    a = _run_draft(g, 5)
    b = _run_draft(g, 5, force_simt=True)
    ta, tb = a["draft_tok"].cpu().numpy(), b["draft_tok"].cpu().numpy()
    assert (ta == tb).mean() > 0.999
    # rows past K_r are not written; compare the written ones where both paths drew the same prefix
    K_r = g["K_r"].cpu().numpy()
    La, Lb = a["draft_logits"].float().cpu().numpy(), b["draft_logits"].float().cpu().numpy()
    for r in range(cfg.B):
        for k in range(K_r[r]):
            if k > 0 and ta[r, k - 1] != tb[r, k - 1]:
                break
            assert np.abs(La[r, k] - Lb[r, k]).max() <= 0.07, (r, k)


def test_draft_deterministic_and_seeded():
    cfg = wl.small_config("qwen", B=8, K_max=3, V=1024)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    a = _run_draft(g, 11)["draft_tok"].cpu()
    b = _run_draft(g, 11)["draft_tok"].cpu()
    c = _run_draft(g, 12)["draft_tok"].cpu()
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


# ---------------------------------------------------------------------------
# verify: small cases, with and without the draft normaliser
# ---------------------------------------------------------------------------
VERIFY_CASES = {
    "fp32-tiny": dict(name="tiny"),
    "bf16-qwen": dict(name="qwen", B=24, K_max=7, V=4104),
    "bf16-ragged": dict(name="ragged", B=60, K_max=5, V=2056),
    "bf16-odd": dict(name="qwen", B=5, K_max=3, V=1003),
    "fp32-odd": dict(name="tiny", B=7, K_max=4, V=997, rank=5),
}


@pytest.mark.parametrize("case", list(VERIFY_CASES))
@pytest.mark.parametrize("with_lse", [True, False])
def test_verify_parity(case, with_lse):
    cfg = wl.small_config(**VERIFY_CASES[case])
    inp = wl.draft_inputs(cfg, "cpu")
    od = oracle_draft(inp, cfg.philox_seed)
    rng = np.random.default_rng(cfg.index + 7)
    K_r = inp["K_r"].numpy()
    ell = np.array([rng.integers(0, k + 1) for k in K_r], np.int32)
    ell[: max(1, cfg.B // 4)] = K_r[: max(1, cfg.B // 4)]        # some requests verify everything
    tgt_dense = wl.target_dense(cfg, inp["U"], inp["K_r"])
    flat, off = wl.flatten_targets(tgt_dense, torch.from_numpy(ell))
    D = torch.from_numpy(od["draft_logits"])
    if cfg.dtype == "bf16":
        D = D.view(torch.bfloat16)
    lse = None
    if with_lse:
        lse = torch.from_numpy(oracle.row_lse(od["draft_logits"], np.repeat(inp["temperature"].numpy(), cfg.K_max)
                                              ).astype(np.float32)).to(DEV)
    seed = 1000 + cfg.index
    g = ds.verify_ragged(D.to(DEV), flat.to(DEV), off.to(DEV), torch.from_numpy(ell).to(DEV),
                         torch.from_numpy(od["draft_tok"]).to(DEV), inp["temperature"].to(DEV), seed, draft_lse=lse)
    assert ds.check(g["status"]) == "DSPARK_OK"
    o = oracle.verify_ragged(host(D), host(flat), off.numpy(), ell, od["draft_tok"], inp["temperature"].numpy(), seed)
    assert compare_verify(g, o) >= 0.9 * cfg.B


@pytest.mark.parametrize("B,K,V,greedy", [(6, 3, 40000, False), (5, 3, 30000, False), (120, 3, 64040, False),
                                           (8, 3, 40000, True), (4, 15, 40000, False), (4, 16, 40000, False)])
def test_verify_bonus_draw_in_parts(B, K, V, greedy):
    # the target rows of the verified positions are the draft's own rows, so every draft token
    # is accepted and every request draws its bonus token; with few requests and several
    # vocabulary slices per row the scan splits each T > 0 bonus draw into parts over slice
    # ranges (4, 3 and 2 parts here), whose winners merge in one packed maximum; with every
    # other request greedy, the whole greedy bonus rows (argmax) share the list with the parts;
    # at K_max = 15 and 16 the row list's capacity B (K_max + 1) allows 2 parts and 1
    cfg = wl.small_config("qwen", B=B, K_max=K, V=V)
    inp = wl.draft_inputs(cfg, "cpu")
    if greedy:
        inp["temperature"][::2] = 0.0
    od = oracle_draft(inp, cfg.philox_seed)
    ell = inp["K_r"].numpy().astype(np.int32)
    tgt_dense = wl.target_dense(cfg, inp["U"], inp["K_r"])
    D = torch.from_numpy(od["draft_logits"]).view(torch.bfloat16)
    tgt_dense[:, : cfg.K_max] = D
    flat, off = wl.flatten_targets(tgt_dense, torch.from_numpy(ell))
    T = inp["temperature"].numpy()
    lse = torch.from_numpy(oracle.row_lse(od["draft_logits"], np.repeat(T, cfg.K_max)).astype(np.float32)).to(DEV)
    seed = 31
    g = ds.verify_ragged(D.to(DEV), flat.to(DEV), off.to(DEV), torch.from_numpy(ell).to(DEV),
                         torch.from_numpy(od["draft_tok"]).to(DEV), inp["temperature"].to(DEV), seed, draft_lse=lse)
    assert ds.check(g["status"]) == "DSPARK_OK"
    o = oracle.verify_ragged(host(D), host(flat), off.numpy(), ell, od["draft_tok"], T, seed)
    assert (o["n_acc"] == ell).sum() >= B - 1        # (nearly) everything accepted
    assert compare_verify(g, o) >= B - 1


def test_verify_output_law_on_gpu():
    # two-token example: lossless output law (0.7, 0.3), acceptance 0.8
    N = 100000
    q = np.array([0.5, 0.5])
    p = np.array([0.7, 0.3])
    U = torch.from_numpy(np.log(q).astype(np.float32)).view(1, 1, 2).expand(N, 1, 2).contiguous().to(DEV)
    E = torch.zeros(2, 1, device=DEV)
    W = torch.zeros(1, 2, device=DEV)
    ones = torch.ones(N, device=DEV)
    d = ds.draft_markov_sample(U, E, W, torch.zeros(N, dtype=torch.int32, device=DEV),
                               torch.ones(N, dtype=torch.int32, device=DEV), ones, 3)
    rows = torch.from_numpy(np.log(np.stack([p, [0.2, 0.8]])).astype(np.float32)).repeat(N, 1).to(DEV)
    off = (torch.arange(N + 1, dtype=torch.int32, device=DEV) * 2)
    v = ds.verify_ragged(d["draft_logits"], rows, off, torch.ones(N, dtype=torch.int32, device=DEV),
                         d["draft_tok"], ones, 4, draft_lse=d["draft_lse"], status=d["status"])
    assert ds.check(d["status"]) == "DSPARK_OK"
    y = v["out_tok"][:, 0].cpu().numpy()
    acc = v["n_acc"].cpu().numpy() == 1
    sd = np.sqrt(0.25 / N)
    assert abs(np.mean(y == 0) - 0.7) < 5 * sd
    assert abs(np.mean(acc) - 0.8) < 5 * sd
    assert (y[~acc] == 0).all()


# ---------------------------------------------------------------------------
# full-size benchmark configurations on sampled requests
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["qwen", "highc", "ragged", "dsv4"])
def test_draft_full_size_sampled(name):
    cfg = wl.CONFIGS[name]
    g = wl.draft_inputs(cfg, DEV)
    if name == "qwen":      # the benchmark's call: W2 packed once
        gpu = ds.draft_markov_sample(g["U"], g["E"], ds.pack_projection(g["W"]), g["anchor"], g["K_r"],
                                     g["temperature"], cfg.philox_seed)
        assert ds.check(gpu["status"]) == "DSPARK_OK"
    else:
        gpu = _run_draft(g, cfg.philox_seed)
    rows = sample_rows(cfg, 16)
    sub = {k: (v[torch.from_numpy(rows).to(DEV)] if k not in ("E", "W") else v) for k, v in g.items()}
    orc = oracle_draft(sub, cfg.philox_seed, req_id=rows.astype(np.int64))
    st = {}
    n = compare_draft(gpu, orc, sub["K_r"].cpu().numpy(), cfg.dtype, rows=rows, stats=st)
    assert n == comparable(orc["flags"], sub["K_r"].cpu().numpy()), (n, st)
    assert n >= 0.8 * int(sub["K_r"].sum()), (n, st)
    del g, gpu
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["qwen", "highc", "ragged", "dsv4"])
def test_verify_full_size_sampled(name):
    cfg = wl.CONFIGS[name]
    g = wl.draft_inputs(cfg, DEV)
    K_r = g["K_r"].cpu()
    conf = wl.confidences(cfg, "cpu")
    o_s = oracle.schedule_survival(conf.numpy(), K_r.numpy(), wl.sps_table(cfg, "literal").numpy())
    ell = torch.from_numpy(o_s["ell"])
    tgt = wl.target_dense(cfg, g["U"], g["K_r"])
    flat, off = wl.flatten_targets(tgt, ell)
    del tgt
    # draft rows: the base logits, draft tokens: uniform ids (inputs independent of any kernel)
    D = g["U"]
    gen = torch.Generator(device="cpu").manual_seed(77)
    tok = torch.randint(0, cfg.V, (cfg.B, cfg.K_max), generator=gen, dtype=torch.int32)
    T = g["temperature"].cpu()
    rows = np.sort(np.random.default_rng(2).choice(cfg.B, size=6, replace=False))
    # normalisers only for the sampled requests (the others are not compared)
    lse = torch.zeros(cfg.B, cfg.K_max)
    for r in rows:
        lse[r] = torch.from_numpy(oracle.row_lse(host(D[int(r)]), np.full(cfg.K_max, T[r].item(), np.float32)))
    v = ds.verify_ragged(D, flat, off.to(DEV), ell.to(torch.int32).to(DEV), tok.to(DEV), g["temperature"], 55,
                         draft_lse=lse.to(DEV))
    assert ds.check(v["status"]) == "DSPARK_OK"
    rsel = torch.from_numpy(rows)
    sub_ell = ell[rsel]
    parts = [flat[int(off[r]):int(off[r + 1])].cpu() for r in rows]
    sub_flat = torch.cat(parts)
    sub_off = torch.zeros(len(rows) + 1, dtype=torch.int32)
    sub_off[1:] = torch.cumsum(sub_ell + 1, 0)
    o = oracle.verify_ragged(host(D[rsel.to(DEV)]), host(sub_flat), sub_off.numpy(), sub_ell.numpy(),
                             tok[rsel].numpy(), T[rsel].numpy(), 55, req_id=rows.astype(np.int64))
    assert compare_verify(v, o, rows=rows) >= 4


# ---------------------------------------------------------------------------
# device-side validation
# ---------------------------------------------------------------------------
def test_device_errors_and_sticky_status():
    cfg = wl.small_config("qwen", B=4, K_max=3, V=1024)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    bad = dict(g)
    bad["anchor"] = g["anchor"].clone()
    bad["anchor"][2] = cfg.V
    out = ds.draft_markov_sample(bad["U"], bad["E"], bad["W"], bad["anchor"], bad["K_r"], bad["temperature"], 0)
    # a later call on the same status word does nothing until the error is read
    st = out["status"]
    ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 0, status=st)
    assert ds.check(st) == "DSPARK_ERR_TOKEN_RANGE"
    assert ds.check(st) == "DSPARK_OK"
    bad = dict(g)
    bad["temperature"] = g["temperature"].clone()
    bad["temperature"][0] = 1e-5
    out = ds.draft_markov_sample(bad["U"], bad["E"], bad["W"], bad["anchor"], bad["K_r"], bad["temperature"], 0)
    assert ds.check(out["status"]) == "DSPARK_ERR_TEMPERATURE"
    bad = dict(g)
    bad["K_r"] = g["K_r"].clone()
    bad["K_r"][1] = 0
    out = ds.draft_markov_sample(bad["U"], bad["E"], bad["W"], bad["anchor"], bad["K_r"], bad["temperature"], 0)
    assert ds.check(out["status"]) == "DSPARK_ERR_LENGTHS"
    conf = torch.full((4, 3), 0.5, device=DEV)
    K_r = torch.full((4,), 3, dtype=torch.int32, device=DEV)
    s = ds.schedule_survival(conf, K_r, torch.ones(16, dtype=torch.float64, device=DEV))
    assert ds.check(s["status"]) == "DSPARK_ERR_SPS_TOO_SHORT"
    conf2 = conf.clone()
    conf2[0, 0] = 1.5
    s = ds.schedule_survival(conf2, K_r, torch.ones(64, dtype=torch.float64, device=DEV))
    assert ds.check(s["status"]) == "DSPARK_ERR_CONFIDENCE"
    D = torch.zeros(4, 3, 1024, dtype=torch.bfloat16, device=DEV)
    tgt = torch.zeros(8, 1024, dtype=torch.bfloat16, device=DEV)
    ell = torch.ones(4, dtype=torch.int32, device=DEV)
    off = torch.arange(5, dtype=torch.int32, device=DEV) * 2
    tok = torch.zeros(4, 3, dtype=torch.int32, device=DEV)
    T = torch.ones(4, device=DEV)
    v = ds.verify_ragged(D, tgt, off, ell, tok, T, 0)
    assert ds.check(v["status"]) == "DSPARK_OK"
    v = ds.verify_ragged(D, tgt, off + torch.tensor([0, 1, 0, 0, 0], dtype=torch.int32, device=DEV), ell, tok, T, 0)
    assert ds.check(v["status"]) == "DSPARK_ERR_OFFSETS"
    tok2 = tok.clone()
    tok2[3, 0] = -1
    v = ds.verify_ragged(D, tgt, off, ell, tok2, T, 0)
    assert ds.check(v["status"]) == "DSPARK_ERR_TOKEN_RANGE"


def test_host_errors():
    cfg = wl.small_config("qwen", B=4, K_max=3, V=1024)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    with pytest.raises(TypeError):
        ds.draft_markov_sample(g["U"].float(), g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 0)
    with pytest.raises(TypeError):
        ds.draft_markov_sample(g["U"].cpu(), g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 0)
    L = ds.lib()
    small = torch.empty(256, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dims = ds.Dims(4, 3, 1024, 256, ds.BF16, 0)
    tok = torch.empty(4, 3, dtype=torch.int32, device=DEV)
    p = lambda t: __import__("ctypes").c_void_p(t.data_ptr())
    code = L.dspark_draft_markov_sample(p(g["U"]), p(g["E"]), p(g["W"]), p(g["anchor"]), p(g["K_r"]),
                                        p(g["temperature"]), 0, dims, p(tok), None, None, None, p(small), 256, p(st),
                                        None)
    assert ds.STATUS_NAMES[code] == "DSPARK_ERR_WORKSPACE"


@pytest.mark.parametrize("case,simt", [("bf16-tc", False), ("bf16-simt", True), ("fp32-simt", False)])
def test_draft_tok_logit_is_the_stored_logit(case, simt):
    # the drawn token's logit output equals the stored logit row at that token, bit for bit,
    # on both kernel paths and for greedy rows; and it is the same with no logits stored
    kw = dict(name="ragged", B=150, K_max=4, V=4104) if case.startswith("bf16") else dict(name="tiny", B=9)
    cfg = wl.small_config(**kw)
    g = _to(wl.draft_inputs(cfg, "cpu"))
    d = _run_draft(g, 21, force_simt=simt)
    tok = d["draft_tok"].long()
    K_r = g["K_r"].cpu()
    live = torch.arange(cfg.K_max, device=DEV)[None, :] < g["K_r"][:, None].long()
    at = torch.gather(d["draft_logits"].float(), 2, tok.clamp(min=0)[..., None])[..., 0]
    assert torch.equal(at[live], d["draft_tok_logit"][live])
    assert int(K_r.sum()) == int(live.sum())
    n = ds.draft_markov_sample(g["U"], g["E"], g["W"], g["anchor"], g["K_r"], g["temperature"], 21,
                               want_logits=False, force_simt=simt)
    assert ds.check(n["status"]) == "DSPARK_OK"
    assert torch.equal(n["draft_tok"], d["draft_tok"])
    assert torch.equal(n["draft_tok_logit"][live], d["draft_tok_logit"][live])

"""Pins for the oracle's random stream (Philox4x32-10, uniforms, Gumbel noise).

The generator is checked against the published known-answer vectors; the
uniform and Gumbel conversions against their exact ranges and laws.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answer_vectors():
    kat = json.load(open(os.path.join(GOLDEN, "philox_kat.json")))
    for vec in kat["vectors"]:
        ctr = [int(x, 16) for x in vec["counter"]]
        key = [int(x, 16) for x in vec["key"]]
        want = [int(x, 16) for x in vec["out"]]
        assert list(map(int, oracle.philox4x32_10(ctr, key))) == want


def test_stream_word_layout():
    # element v uses word v & 3 of the block with counter (v >> 2, position, request, tag);
    # key = (seed lo, seed hi)
    seed = 0x0123456789ABCDEF
    for v in (0, 1, 2, 3, 4, 7, 151935):
        blk = oracle.philox4x32_10([v >> 2, 5, 9, 2], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.stream_word(seed, v, 5, 9, 2) == int(blk[v & 3])


def test_uniform_ranges_and_exactness():
    # gumbel uniform ((w >> 9) + 0.5) * 2^-23 spans (0, 1) and is exact in fp32
    assert oracle.uniform_open(0) == 2.0 ** -24
    assert oracle.uniform_open(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform_accept(0) == 0.0
    assert oracle.uniform_accept(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    rng = np.random.default_rng(0)
    for w in rng.integers(0, 2 ** 32, 2000, dtype=np.uint64):
        u = oracle.uniform_open(int(w))
        assert float(np.float32(u)) == u and 0.0 < u < 1.0
        a = oracle.uniform_accept(int(w))
        assert float(np.float32(a)) == a and 0.0 <= a < 1.0


def test_gumbel_extremes_closed_form():
    # g = -log(-log(u)) at the two ends of the uniform grid
    assert oracle.gumbel(0) == pytest.approx(-math.log(-math.log(2.0 ** -24)), rel=1e-15)
    assert oracle.gumbel(0xFFFFFFFF) == pytest.approx(-math.log(-math.log1p(-(2.0 ** -24))), rel=1e-12)


def test_stream_uniformity_and_independence():
    # words of one stream: uniform (chi-square on 256 bins of the top byte),
    # lag-1 correlation near zero, different tags/requests/positions decorrelated
    n = 40000
    w = np.array([oracle.stream_word(7, v, 3, 11, 0) for v in range(n)], dtype=np.uint64)
    top = (w >> 24).astype(np.int64)
    counts = np.bincount(top, minlength=256)
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4
    u = (w.astype(np.float64) + 0.5) / 2 ** 32
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.03
    w2 = np.array([oracle.stream_word(7, v, 3, 11, 1) for v in range(2000)], dtype=np.float64)
    w3 = np.array([oracle.stream_word(7, v, 3, 12, 0) for v in range(2000)], dtype=np.float64)
    w4 = np.array([oracle.stream_word(7, v, 4, 11, 0) for v in range(2000)], dtype=np.float64)
    for other in (w2, w3, w4):
        assert abs(np.corrcoef(u[:2000], other)[0, 1]) < 0.08
        assert not np.array_equal(w[:2000].astype(np.float64), other)


def test_gumbel_law():
    # g = -log(-log u) with u uniform is standard Gumbel: P(g <= x) = exp(-exp(-x))
    g = np.array([oracle.gumbel(oracle.stream_word(3, v, 1, 0, 0)) for v in range(20000)])
    ks = stats.kstest(g, stats.gumbel_r.cdf)
    assert ks.pvalue > 1e-4
    assert g.mean() == pytest.approx(np.euler_gamma, abs=0.03)

"""Pins of the oracle's per-position acceptance rate beta = sum min(p, q) and
total-variation distance TV = (1/2) sum |p - q| (CPU only).

beta is pinned to the pages' printed values, to the accept rule itself (the
exact acceptance mass of the oracle's verify step, found by enumerating its
decision cells), and to closed forms: q = p, disjoint supports, a top-p case
worked by hand, the TV identity and symmetry.
"""
import os

import numpy as np
import pytest

import oracle
import workloads
from enumeration import cells, processed, softmax_T


def _golden(name):
    rows = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = vals
    return rows


def _logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _pair(p, q):
    """[1, 2, V] target (row 0 = p, row 1 unused) and [1, 1, V] draft."""
    lp = _logits_of(p)
    return np.stack([lp, lp])[None], _logits_of(q)[None, None]


def test_quiz_value():
    """"3.5 Speculative Decoding", "Check your understanding": beta = 0.7."""
    g = _golden("lz_quiz_residual.txt")
    tgt, drf = _pair(np.array(g["p"], float), np.array(g["q"], float))
    r = oracle.acceptance(tgt, drf)
    assert r["errors"] == 0
    assert abs(r["beta"][0, 0] - float(g["beta"][0])) < 1e-6
    assert abs(r["tv"][0, 0] - (1 - float(g["beta"][0]))) < 1e-6


def test_misaligned_pair_printed_rate():
    """"246 Speculative Decoding", 3.2: sum min(p, q) = 0.55 for the page's
    pair, and the page's measured rate over 200,000 trials lies within four
    standard errors of it."""
    g = _golden("mn_exactness_v6.txt")
    tgt, drf = _pair(np.array(g["p"], float), np.array(g["q"], float))
    beta = oracle.acceptance(tgt, drf)["beta"][0, 0]
    assert abs(beta - float(g["beta_exact"][0])) < 1e-6
    n = int(g["trials"][0])
    assert abs(float(g["printed_accept_rate"][0]) - beta) < 4 * np.sqrt(beta * (1 - beta) / n)


@pytest.mark.parametrize("seed,T,top_p", [(0, 1.0, 1.0), (1, 0.7, 1.0), (2, 1.3, 0.8),
                                          (3, 1.0, 0.5), (4, 0.6, 0.95)])
def test_beta_is_the_accept_mass_of_the_rule(seed, T, top_p):
    """beta_1 equals the probability that the accept test u*Q < P passes when
    x~ ~ q: the weight of the cells where the oracle's verify step accepts."""
    rng = np.random.default_rng(seed)
    V = 5
    tgt = rng.normal(0, 1.5, (1, 2, V)).astype(np.float32)
    drf = (tgt[:, :1] + rng.normal(0, 1.0, (1, 1, V))).astype(np.float32)
    P = [processed(tgt[0, 0], T, top_p), processed(tgt[0, 1], T, top_p)]
    Q = [processed(drf[0, 0], T, top_p)]
    cl = list(cells(P, Q))
    n = len(cl)
    res = oracle.verify_sample(np.repeat(tgt, n, 0), np.repeat(drf, n, 0),
                               np.array([c[0] for c in cl], np.int32).reshape(n, 1),
                               np.array([c[1] for c in cl], np.float32), T=T, top_p=top_p)
    w = np.array([c[2] for c in cl])
    accept_mass = w[res["num_accepted"] == 1].sum()
    r = oracle.acceptance(tgt, drf, T=T, top_p=top_p)
    assert abs(r["beta"][0, 0] - accept_mass) < 1e-9


def test_identical_rows():
    """q = p: beta = 1 and TV = 0 ("Acceptance Rate and Total Variation
    Distance": a perfect draft gives alpha = 1)."""
    rng = np.random.default_rng(5)
    tgt = rng.normal(0, 2, (3, 4, 700)).astype(np.float32)
    for top_p in (1.0, 0.9):
        r = oracle.acceptance(tgt, tgt[:, :3].copy(), T=0.8, top_p=top_p)
        np.testing.assert_allclose(r["beta"], 1.0, atol=1e-12)
        np.testing.assert_allclose(r["tv"], 0.0, atol=1e-12)


def test_disjoint_supports():
    p = np.array([0.6, 0.4, 0.0, 0.0])
    q = np.array([0.0, 0.0, 0.5, 0.5])
    tgt, drf = _pair(p, q)
    r = oracle.acceptance(tgt, drf)
    assert r["beta"][0, 0] == 0.0
    assert abs(r["tv"][0, 0] - 1.0) < 1e-15


def test_top_p_by_hand():
    """p = (.5, .3, .2), q = (.2, .3, .5), top_p = 0.7: the nuclei are {0, 1}
    and {2, 1}, so p -> (.625, .375, 0), q -> (0, .375, .625): beta = .375,
    TV = .625."""
    tgt, drf = _pair([0.5, 0.3, 0.2], [0.2, 0.3, 0.5])
    r = oracle.acceptance(tgt, drf, top_p=0.7)
    assert abs(r["beta"][0, 0] - 0.375) < 1e-7
    assert abs(r["tv"][0, 0] - 0.625) < 1e-7


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tv_identity_and_symmetry(dtype):
    """TV = 1 - beta for any two distributions, beta(p, q) = beta(q, p), and
    beta matches numpy's sum of minima over the enumeration helpers' rows."""
    rng = np.random.default_rng(7)
    B, k, V = 2, 3, 257
    t32 = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    d32 = (t32[:, :k] + rng.normal(0, 1, (B, k, V))).astype(np.float32)
    if dtype == "bf16":
        tgt, drf = workloads.to_bf16_bits(t32), workloads.to_bf16_bits(d32)
    else:
        tgt, drf = t32, d32
    r = oracle.acceptance(tgt, drf, T=0.9)
    np.testing.assert_allclose(r["beta"] + r["tv"], 1.0, atol=1e-12)
    swapped_t = np.concatenate([drf, tgt[:, k:]], axis=1)
    swapped_d = tgt[:, :k].copy()
    np.testing.assert_allclose(oracle.acceptance(swapped_t, swapped_d, T=0.9)["beta"], r["beta"],
                               atol=1e-14)
    tf, df = workloads.as_f32(tgt), workloads.as_f32(drf)
    for b in range(B):
        for i in range(k):
            want = np.minimum(softmax_T(tf[b, i], 0.9), softmax_T(df[b, i], 0.9)).sum()
            assert abs(r["beta"][b, i] - want) < 1e-12


def test_data_errors_give_nan():
    rng = np.random.default_rng(9)
    tgt = rng.normal(0, 1, (2, 3, 16)).astype(np.float32)
    drf = rng.normal(0, 1, (2, 2, 16)).astype(np.float32)
    tgt[0, 1, 3] = np.nan
    drf[1, 0, :] = -np.inf
    r = oracle.acceptance(tgt, drf)
    assert np.isnan(r["beta"][0, 1]) and np.isnan(r["tv"][0, 1])
    assert np.isnan(r["beta"][1, 0])
    assert np.isfinite(r["beta"][0, 0]) and np.isfinite(r["beta"][1, 1])
    assert r["errors"] == (1 << oracle.ROW_NONFINITE) | (1 << oracle.ROW_ALL_NEG_INF)

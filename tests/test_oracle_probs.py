"""Pins of the oracle's verify step with the draft given as probabilities
(CPU only).

The pages' own worked pairs are stated as probability vectors, so here they
enter exactly as printed: the exact law of the step (enumerated over its
decision cells) must give the page's acceptance rate and residual, and emit
p -- the exactness theorem holds for any q.
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


def _cells_in_range(P, Q):
    """The decision cells whose midpoint uniforms stay below 1 in fp32.  A
    reject cell of width ~1e-8 (p/q a hair under 1 after fp32 rounding) has
    its midpoint round up to 1.0; it is dropped and its weight returned."""
    keep, dropped = [], 0.0
    for c in cells(P, Q):
        if np.all(np.asarray(c[1], np.float32) < 1.0):
            keep.append(c)
        else:
            dropped += c[2]
    return keep, dropped


def _exact_law(p, q, top_p=1.0):
    """One position (k = 1) with target logits log p and draft probabilities
    q (fp32): (acceptance mass, law of the emitted token, residual law)."""
    lp = _logits_of(p)
    tgt = np.stack([lp, lp])[None]
    qf = np.asarray(q, np.float32)[None, None]
    P = [processed(lp, 1.0, top_p)] * 2
    Q = [qf[0, 0].astype(np.float64)]
    cl, dropped = _cells_in_range(P, Q)
    assert dropped < 1e-6
    n = len(cl)
    res = oracle.verify_sample_probs(np.repeat(tgt, n, 0), np.repeat(qf, n, 0),
                                     np.array([c[0] for c in cl], np.int32).reshape(n, 1),
                                     np.array([c[1] for c in cl], np.float32), T=1.0, top_p=top_p)
    assert res["errors"] == 0
    w = np.array([c[2] for c in cl])
    acc = res["num_accepted"] == 1
    V = len(p)
    law = np.zeros(V)
    np.add.at(law, res["tokens"][:, 0], w)
    resid = np.zeros(V)
    np.add.at(resid, res["tokens"][~acc, 0], w[~acc])
    return w[acc].sum(), law, resid / resid.sum(), P[0]


def test_quiz_pair_as_probabilities():
    """"3.5 Speculative Decoding", "Check your understanding": beta = 0.7,
    residual all on a, and a keeps probability 0.6."""
    g = _golden("lz_quiz_residual.txt")
    p, q = np.array(g["p"], float), np.array(g["q"], float)
    beta, law, resid, _ = _exact_law(p, q)
    assert abs(beta - float(g["beta"][0])) < 1e-6
    np.testing.assert_allclose(resid, np.array(g["residual"], float), atol=1e-6)
    assert abs(law[0] - float(g["p_emit_a"][0])) < 1e-6
    np.testing.assert_allclose(law, p, atol=1e-6)


def test_misaligned_pair_as_probabilities():
    """"246 Speculative Decoding", 3.2: the page's (p, q) entered as printed;
    acceptance 0.55, residual (2/3, 1/3, 0, 0, 0, 0), emitted law p."""
    g = _golden("mn_exactness_v6.txt")
    p, q = np.array(g["p"], float), np.array(g["q"], float)
    beta, law, resid, _ = _exact_law(p, q)
    assert abs(beta - float(g["beta_exact"][0])) < 1e-6
    np.testing.assert_allclose(resid, [2 / 3, 1 / 3, 0, 0, 0, 0], atol=1e-6)
    np.testing.assert_allclose(law, p, atol=1e-6)


def test_top_p_processes_the_target_only():
    """p = (.5, .3, .2) with top-p 0.7 -> p' = (.625, .375, 0); q = (.2, .3,
    .5) is used as given.  Acceptance = sum min(p', q) = .2 + .3 = .5, the
    residual max(0, p' - q) = (.425, .075, 0) normalises to (.85, .15, 0),
    and the emitted law is p'."""
    beta, law, resid, pp = _exact_law([0.5, 0.3, 0.2], [0.2, 0.3, 0.5], top_p=0.7)
    np.testing.assert_allclose(pp, [0.625, 0.375, 0.0], atol=1e-7)
    assert abs(beta - 0.5) < 1e-6
    np.testing.assert_allclose(resid, [0.85, 0.15, 0.0], atol=1e-6)
    np.testing.assert_allclose(law, [0.625, 0.375, 0.0], atol=1e-6)


@pytest.mark.parametrize("seed", range(4))
def test_exactness_for_arbitrary_q(seed):
    """Random tiny steps (V = 5, k = 2) with q drawn independently of p: the
    law of every emitted position is p_n (exactness needs no relation
    between q and p)."""
    rng = np.random.default_rng(seed)
    V, k, T = 5, 2, 0.8
    tgt = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    qf = rng.dirichlet(np.ones(V), k).astype(np.float32)
    P = [processed(tgt[i], T, 1.0) for i in range(k + 1)]
    Q = [qf[i].astype(np.float64) for i in range(k)]
    cl, dropped = _cells_in_range(P, Q)
    assert dropped < 1e-6
    n = len(cl)
    res = oracle.verify_sample_probs(np.broadcast_to(tgt, (n, k + 1, V)).copy(),
                                     np.broadcast_to(qf, (n, k, V)).copy(),
                                     np.array([c[0] for c in cl], np.int32).reshape(n, k),
                                     np.array([c[1] for c in cl], np.float32), T=T)
    w = np.array([c[2] for c in cl])
    jn, tok = res["num_accepted"], res["tokens"]
    assert np.all(jn >= 0)
    # Position n emits a token iff the first n-1 drafts were accepted; its
    # law, conditioned on being reached, is p_n.
    for pos in range(k + 1):
        reach = jn >= pos
        law = np.zeros(V)
        np.add.at(law, tok[reach, pos], w[reach])
        np.testing.assert_allclose(law / w[reach].sum(), P[pos], atol=1e-9)


def test_matches_the_logits_form():
    """q given as the oracle's own processed draft rows (rounded to fp32)
    gives the logits form's outcome wherever neither run is within 1e-5 of
    a decision boundary."""
    wl = workloads.c2()
    q = np.stack([[oracle.process_row(wl.draft[b, i], wl.T, wl.top_p)[1]
                   for i in range(wl.k)] for b in range(wl.B)]).astype(np.float32)
    a = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T,
                             debug=True)
    b = oracle.verify_sample_probs(wl.target, q, wl.draft_tokens, wl.uniforms, T=wl.T,
                                   debug=True)
    near = oracle.boundary_flags(a, wl.uniforms) | oracle.boundary_flags(b, wl.uniforms)
    same = (a["num_accepted"] == b["num_accepted"]) & np.all(a["tokens"] == b["tokens"], axis=1)
    assert np.all(same | near)
    np.testing.assert_allclose(b["dbg"][:, wl.k:2 * wl.k], a["dbg"][:, wl.k:2 * wl.k], rtol=1e-6)


def test_gathered_probability_checks():
    rng = np.random.default_rng(3)
    B, k, V = 5, 2, 16
    tgt = rng.normal(0, 1, (B, k + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, k)).astype(np.float32)
    toks = rng.integers(0, V, (B, k)).astype(np.int32)
    u = workloads.uniforms(rng, (B, k + 1))
    q[0, 1, toks[0, 1]] = np.nan
    q[1, 0, toks[1, 0]] = -0.25
    q[2, 1, toks[2, 1]] = 1.5
    q[3, 0, (toks[3, 0] + 1) % V] = np.nan  # not gathered: not checked
    res = oracle.verify_sample_probs(tgt, q, toks, u)
    assert list(res["num_accepted"][:3]) == [-1, -1, -1]
    assert np.all(res["tokens"][:3] == -1)
    assert res["num_accepted"][4] >= 0
    assert res["errors"] == 1 << oracle.PROB_RANGE


def test_invariants_on_c3_rows():
    """Every sequence emits 1..k+1 tokens, all in [0, V), on a c3-shaped
    batch with Dirichlet-drawn probability rows."""
    rng = np.random.default_rng(8)
    wl = workloads.c3(B=3)
    q = rng.dirichlet(np.full(wl.V, 0.05), (wl.B, wl.k)).astype(np.float32)
    toks = np.array([[rng.choice(wl.V, p=q[b, i] / q[b, i].sum(dtype=np.float64))
                      for i in range(wl.k)] for b in range(wl.B)], np.int32)
    res = oracle.verify_sample_probs(wl.target, q, toks, wl.uniforms, T=wl.T)
    j = res["num_accepted"]
    assert np.all((j >= 0) & (j <= wl.k))
    for b in range(wl.B):
        emitted = res["tokens"][b, :j[b] + 1]
        assert np.all((emitted >= 0) & (emitted < wl.V))
        assert np.all(res["tokens"][b, j[b] + 1:] == -1)
        np.testing.assert_array_equal(emitted[:j[b]], toks[b, :j[b]])

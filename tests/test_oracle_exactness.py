"""Pins of the CPU oracle against the exactness theorem, by exact enumeration.

"3.5 Speculative Decoding", "Proof that the output distribution is exactly
p", and "246 Speculative Decoding", 2.3 "Proof of exactness": whatever the
draft, the token emitted at each position is distributed exactly as the
(processed) target p.  For V <= 8 and k <= 3 the oracle is evaluated at the
midpoint of every cell of its piecewise-constant dependence on the uniforms
(tests/enumeration.py); the resulting law must equal p_n within 1e-12, and
the chance of reaching position n must be prod_{i<n} beta_i.
"""
import numpy as np
import pytest

import oracle
import workloads
from enumeration import acceptance_probability, cells, laws, processed


def _run_cells(target_rows, draft_rows, T, top_p, storage):
    """target_rows [k+1, V], draft_rows [k, V] in storage dtype; returns the
    expected distributions, the cells and the oracle's outputs on them."""
    vals_t = workloads.as_f32(target_rows).astype(np.float64)
    vals_d = workloads.as_f32(draft_rows).astype(np.float64)
    k = draft_rows.shape[0]
    P = [processed(vals_t[i], T, top_p) for i in range(k + 1)]
    Q = [processed(vals_d[i], T, top_p) for i in range(k)]
    cl = list(cells(P, Q))
    B = len(cl)
    toks = np.array([c[0] for c in cl], np.int32).reshape(B, k)
    unis = np.array([c[1] for c in cl], np.float32)
    weights = np.array([c[2] for c in cl])
    tgt = np.ascontiguousarray(np.broadcast_to(target_rows, (B,) + target_rows.shape))
    drf = np.ascontiguousarray(np.broadcast_to(draft_rows, (B,) + draft_rows.shape))
    res = oracle.verify_sample(tgt, drf, toks, unis, T=T, top_p=top_p)
    assert res["errors"] == 0
    return P, Q, cl, toks, weights, res


CASES = [
    # (V, k, T, top_p, dtype, seed)
    (3, 1, 1.0, 1.0, "f32", 1),
    (5, 2, 1.0, 1.0, "f32", 2),
    (6, 3, 0.7, 1.0, "f32", 3),
    (8, 3, 1.3, 1.0, "bf16", 4),
    (8, 2, 1.0, 0.8, "f32", 5),
    (7, 3, 0.9, 0.7, "bf16", 6),
]


@pytest.mark.parametrize("V,k,T,top_p,dt,seed", CASES)
def test_emitted_law_equals_target(V, k, T, top_p, dt, seed):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    if top_p < 1.0:
        # a related draft, so the two nuclei overlap and later positions are
        # reached
        drf = (tgt[:k] + rng.normal(0, 0.5, (k, V))).astype(np.float32)
        # force exact ties so the tie rule is exercised
        tgt[:, 1] = tgt[:, 0]
        drf[:, 2] = drf[:, 0]
    else:
        drf = rng.normal(0, 1.5, (k, V)).astype(np.float32)  # unrelated draft
    store = workloads.to_bf16_bits if dt == "bf16" else (lambda a: a)
    tgt, drf = store(tgt), store(drf)
    P, Q, cl, toks, w, res = _run_cells(tgt, drf, T, top_p, dt)

    # The oracle lands in the cell it was evaluated in.
    exp_j = np.array([c[3] for c in cl])
    exp_x = np.array([c[4] for c in cl])
    np.testing.assert_array_equal(res["num_accepted"], exp_j)
    np.testing.assert_array_equal(res["tokens"][np.arange(len(cl)), exp_j], exp_x)

    law, reach = laws(P, Q, toks, res["num_accepted"], res["tokens"], w)
    assert abs(w.sum() - 1.0) < 1e-12
    beta = [acceptance_probability(P[i], Q[i]) for i in range(k)]
    for n in range(k + 1):
        assert abs(reach[n] - np.prod(beta[:n])) < 1e-12
        assert reach[n] > 1e-6
        np.testing.assert_allclose(law[n] / reach[n], P[n], rtol=0, atol=1e-12)


def test_expected_tokens_is_sum_of_reach_probabilities():
    """E[emitted] = sum_{n=0}^{k} prod_{i<=n} beta_i with per-position beta
    (the closed form's derivation in "3.5 Speculative Decoding", "Expected
    tokens per step", without the equal-alpha assumption)."""
    rng = np.random.default_rng(11)
    V, k, T = 6, 3, 1.0
    tgt = rng.normal(0, 2, (k + 1, V)).astype(np.float32)
    drf = (tgt[:k] + rng.normal(0, 0.7, (k, V))).astype(np.float32)
    P, Q, cl, toks, w, res = _run_cells(tgt, drf, T, 1.0, "f32")
    emitted = res["num_accepted"] + 1
    beta = [acceptance_probability(P[i], Q[i]) for i in range(k)]
    closed = sum(np.prod(beta[:n]) for n in range(k + 1))
    assert abs((w * emitted).sum() - closed) < 1e-12


@pytest.mark.parametrize("alpha,k", [(0.7, 3), (0.8, 1), (0.8, 2), (0.8, 3), (0.6, 3)])
def test_closed_form_exact_with_equal_alpha(alpha, k):
    """With the same (p, q) at every position and sum min(p, q) = alpha,
    acceptance is independent at rate alpha and E[tokens per step] =
    (1 - alpha^(k+1)) / (1 - alpha) exactly ("3.5 Speculative Decoding",
    "Expected tokens per step"; "246 Speculative Decoding", 2.4)."""
    d = (1 - alpha) / 2
    p = np.array([0.5 + d, 0.5 - d])
    q = np.array([0.5 - d, 0.5 + d])
    tgt = np.log(np.tile(p, (k + 1, 1))).astype(np.float32)
    drf = np.log(np.tile(q, (k, 1))).astype(np.float32)
    P, Q, cl, toks, w, res = _run_cells(tgt, drf, 1.0, 1.0, "f32")
    beta = acceptance_probability(P[0], Q[0])
    assert abs(beta - alpha) < 1e-6  # fp32 logits of p, q
    closed = (1 - beta ** (k + 1)) / (1 - beta)
    assert abs((w * (res["num_accepted"] + 1)).sum() - closed) < 1e-12


def test_one_hot_stochastic_equals_greedy():
    """Point-mass p and q: the stochastic rule reduces to the greedy rule
    ("3.5 Speculative Decoding", end of the proof; "246 Speculative
    Decoding", end of 2.3)."""
    rng = np.random.default_rng(5)
    B, k, V = 200, 3, 9
    top = rng.integers(0, V, (B, k + 1))
    dtop = np.where(rng.random((B, k)) < 0.6, top[:, :k], rng.integers(0, V, (B, k)))
    tgt = np.full((B, k + 1, V), -1000.0, np.float32)
    drf = np.full((B, k, V), -1000.0, np.float32)
    np.put_along_axis(tgt, top[..., None], 0.0, axis=2)
    np.put_along_axis(drf, dtop[..., None], 0.0, axis=2)
    toks = dtop.astype(np.int32)  # drafts sampled from a point mass
    u = workloads.uniforms(rng, (B, k + 1))
    s = oracle.verify_sample(tgt, drf, toks, u, T=1.0)
    g = oracle.verify_sample(tgt, None, toks, None, mode=oracle.GREEDY)
    np.testing.assert_array_equal(s["tokens"], g["tokens"])
    np.testing.assert_array_equal(s["num_accepted"], g["num_accepted"])


def test_identical_draft_always_accepts():
    """q = p: every draft is accepted (u*Q < P for u < 1) and the bonus is
    drawn from p_{k+1} ("3.5 Speculative Decoding", step 4 "Bonus token")."""
    rng = np.random.default_rng(6)
    V, k = 5, 3
    tgt = rng.normal(0, 1, (k + 1, V)).astype(np.float32)
    P, Q, cl, toks, w, res = _run_cells(tgt, tgt[:k].copy(), 1.0, 1.0, "f32")
    assert np.all(res["num_accepted"] == k)
    law, reach = laws(P, Q, toks, res["num_accepted"], res["tokens"], w)
    np.testing.assert_allclose(law[k], P[k], atol=1e-12)

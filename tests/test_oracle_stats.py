"""Statistical pin of the CPU oracle on the tiny exactness workload (c1):
10^5 seeded verify steps, B=1, k=3, V=32, fp32, target ~ N(0, 2^2), draft =
target + N(0, 0.7^2), drafts drawn from q.

* Exactness ("3.5 Speculative Decoding", "Proof that the output distribution
  is exactly p"; "246 Speculative Decoding", 3.2): at every output position
  the emitted token, among the steps that reach it, follows p_n -- Pearson
  chi-square, bins with expected count < 5 pooled, pass at p > 0.001.
* Tokens per step: the mean equals sum_{n=0}^{k} prod_{i<=n} beta_i (the
  closed form with the per-position beta of these rows) within 4 standard
  errors.
* Invariant: every step emits between 1 and k+1 tokens.
"""
import numpy as np

import oracle
import workloads
from enumeration import acceptance_probability, softmax_T
from stats import position_fits


def test_c1_chi_square_and_tokens_per_step():
    wl = workloads.c1()
    res = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T)
    assert res["errors"] == 0
    j = res["num_accepted"]
    assert np.all((j >= 0) & (j <= wl.k))
    P = [softmax_T(wl.target[0, n].astype(np.float64), wl.T) for n in range(wl.k + 1)]
    Q = [softmax_T(wl.draft[0, n].astype(np.float64), wl.T) for n in range(wl.k)]
    pvals = position_fits(res["tokens"], j, P, wl.V)
    assert min(pvals) > 1e-3, pvals
    beta = [acceptance_probability(P[i], Q[i]) for i in range(wl.k)]
    exact = sum(np.prod(beta[:n]) for n in range(wl.k + 1))
    emitted = j + 1
    se = emitted.std() / np.sqrt(emitted.size)
    assert abs(emitted.mean() - exact) < 4 * se


def test_chi_square_detects_a_wrong_law():
    """Power check of the test itself: the same draws judged against a
    different distribution fail."""
    wl = workloads.c1()
    res = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T)
    P = [softmax_T(wl.target[0, n].astype(np.float64), wl.T) for n in range(wl.k + 1)]
    wrong = [softmax_T(wl.draft[0, 0].astype(np.float64), wl.T)] + P[1:]
    assert position_fits(res["tokens"], res["num_accepted"], wrong, wl.V)[0] < 1e-6

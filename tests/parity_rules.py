"""The stochastic parity rule, shared by the GPU tests.

  * accept counts are bit-exact, except on a sequence the oracle flags at an
    accept-ratio boundary (|u_i - P_i/Q_i| < 1e-5 at a test it ran) or at a
    top-p boundary (a row's cumulative mass within 1e-5 of top_p, which can
    change its kept set);
  * emitted tokens are exact, except that a sequence flagged only at a
    final-draw CDF edge may differ in the drawn token alone (the token at
    position j), and a sequence flagged at an accept-ratio or top-p boundary
    may differ anywhere;
  * mismatches (of any kind) are counted and stay within a budget.

Every call prints one line with the counts, so that a run with -s (or the
smoke test) reports them.
"""
import numpy as np

import oracle


def check(label, gpu_t, gpu_n, ref, uniforms, top_p, budget):
    """Apply the rule; returns the union of the flags.  `ref` is the oracle's
    verify_sample / verify_sample_probs result with debug=True."""
    acc, cdf, nuc = oracle.boundary_kinds(ref, uniforms, top_p)
    ref_t, ref_n = ref["tokens"], ref["num_accepted"]
    B, W = ref_t.shape
    same_n = gpu_n == ref_n
    same_t = np.all(gpu_t == ref_t, axis=1)
    same = same_n & same_t
    loose = acc | nuc  # anything may differ
    cdf_only = cdf & ~loose
    # only the drawn token (position j) may differ on a CDF-edge sequence
    other = np.arange(W)[None, :] != np.maximum(ref_n, 0)[:, None]
    bad_n = ~same_n & ~loose
    bad_cdf = cdf_only & same_n & np.any((gpu_t != ref_t) & other, axis=1)
    bad_t = ~same & ~(loose | cdf)
    print("%s: B=%d flagged=%d (accept %d, cdf %d, nucleus %d) mismatched=%d "
          "(accept counts %d)" % (label, B, (acc | cdf | nuc).sum(), acc.sum(), cdf.sum(),
                                  nuc.sum(), (~same).sum(), (~same_n).sum()))
    assert not bad_n.any(), "accept counts differ off an accept/top-p boundary at %s" % (
        np.nonzero(bad_n)[0][:10])
    assert not bad_cdf.any(), "a CDF-edge sequence differs beyond its drawn token at %s" % (
        np.nonzero(bad_cdf)[0][:10])
    assert not bad_t.any(), "unflagged mismatches at %s" % np.nonzero(bad_t)[0][:10]
    assert (~same).sum() <= budget, "%d mismatches > budget %d" % ((~same).sum(), budget)
    return acc | cdf | nuc

"""Goodness-of-fit helpers shared by the oracle and GPU statistical tests."""
import numpy as np
from scipy import stats


def chi_square_pvalue(counts, probs, min_expected=5.0):
    """Pearson chi-square p-value of observed counts against probabilities.

    Bins whose expected count is below min_expected are pooled (smallest
    first) until every bin reaches it; df = (number of bins) - 1.
    """
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    n = counts.sum()
    order = np.argsort(probs * n)
    obs, exp, pool_o, pool_e = [], [], 0.0, 0.0
    for i in order:
        e = probs[i] * n
        if pool_e + e < min_expected or (pool_e > 0 and pool_e < min_expected):
            pool_o += counts[i]
            pool_e += e
            if pool_e >= min_expected:
                obs.append(pool_o)
                exp.append(pool_e)
                pool_o = pool_e = 0.0
        else:
            obs.append(counts[i])
            exp.append(e)
    if pool_e > 0:
        if exp:
            obs[0] += pool_o
            exp[0] += pool_e
        else:
            obs.append(pool_o)
            exp.append(pool_e)
    obs, exp = np.array(obs), np.array(exp)
    if len(exp) < 2:
        return 1.0
    stat = ((obs - exp) ** 2 / exp).sum()
    return float(stats.chi2.sf(stat, len(exp) - 1))


def position_fits(tokens, num_accepted, P, V):
    """p-values of the emitted token at each output position n, among the
    steps that reach n, against the exact target distribution P[n]."""
    out = []
    for n in range(len(P)):
        reached = num_accepted >= n
        counts = np.bincount(tokens[reached, n], minlength=V)
        out.append(chi_square_pvalue(counts, P[n]))
    return out

"""Exact enumeration of one verification step on tiny inputs (test helper).

The step is a deterministic function of (draft tokens, uniforms) once the
logits are fixed, and it is piecewise constant in the uniforms: position i
accepts on u_i in [0, min(1, p_i/q_i)) and rejects on the rest, and the final
draw returns token x on u in [C(x-1)/S, C(x)/S).  Evaluating an
implementation once at the midpoint of every such cell, and weighting each
cell by its volume times prod_i q_i(x~_i), gives the exact law of its
output -- which the exactness theorem says must be p_n at every emitted
position n ("3.5 Speculative Decoding", "Proof that the output distribution
is exactly p"; "246 Speculative Decoding", 2.3 "Proof of exactness").

The expected distributions come from this module's own numpy softmax and a
brute-force nucleus over upper sets, never from the implementation under
test.
"""
from __future__ import annotations

import itertools

import numpy as np


def softmax_T(logits, T):
    """Plain numpy softmax of logits / T in fp64 (-inf -> 0)."""
    z = np.asarray(logits, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def nucleus_upper_set(p, top_p):
    """Top-p by brute force: among all token sets S that are closed upward
    (y in S and p(x) >= p(y) imply x in S), take the smallest whose mass is
    >= top_p; return p restricted to it and renormalised."""
    p = np.asarray(p, np.float64)
    V = p.shape[0]
    best = None
    for bits in range(1, 1 << V):
        S = [x for x in range(V) if bits >> x & 1]
        lowest = min(p[x] for x in S)
        if any(p[x] >= lowest and x not in S for x in range(V)):
            continue
        if p[S].sum() >= top_p and (best is None or len(S) < len(best)):
            best = S
    out = np.zeros(V)
    out[best] = p[best]
    return out / out.sum()


def processed(logits, T, top_p):
    p = softmax_T(logits, T)
    return nucleus_upper_set(p, top_p) if top_p < 1.0 else p


def cells(P, Q):
    """All cells of one step.  P: k+1 target distributions, Q: k draft ones.

    Yields (draft_tokens, uniforms[k+1], weight, j, token) where j is the
    number of accepted drafts and token the final draw in that cell."""
    k, V = len(Q), len(P[0])
    for xt in itertools.product(range(V), repeat=k):
        wq = float(np.prod([Q[i][xt[i]] for i in range(k)]))
        if wq == 0.0:
            continue
        for j in range(k + 1):
            u = [0.5] * (k + 1)
            vol = 1.0
            feasible = True
            for i in range(j):
                a = min(1.0, P[i][xt[i]] / Q[i][xt[i]])
                if a == 0.0:
                    feasible = False
                    break
                vol *= a
                u[i] = a / 2
            if not feasible:
                continue
            if j < k:
                a = min(1.0, P[j][xt[j]] / Q[j][xt[j]])
                if a >= 1.0:
                    continue
                vol *= 1.0 - a
                u[j] = (a + 1.0) / 2
                w = np.maximum(P[j] - Q[j], 0.0)
                if w.sum() <= 0.0:
                    w = P[j].copy()
            else:
                w = P[k].copy()
            S = w.sum()
            C = np.cumsum(w)
            for x in range(V):
                if w[x] <= 0.0:
                    continue
                u_final = (C[x] - w[x] / 2) / S
                uu = list(u)
                uu[k] = u_final
                yield xt, uu, wq * vol * w[x] / S, j, x


def laws(P, Q, draft_tokens, num_accepted, tokens, weights):
    """Exact law of the emitted token at each output position, from an
    implementation's outputs on the cells.  Returns (law[k+1][V],
    reach[k+1]) with reach[n] = P(position n is emitted)."""
    k, V = len(Q), len(P[0])
    law = np.zeros((k + 1, V))
    for n in range(k + 1):
        emitted = num_accepted >= n
        np.add.at(law[n], tokens[emitted, n], weights[emitted])
    reach = law.sum(axis=1)
    return law, reach


def acceptance_probability(p, q):
    """beta = sum_x min(p(x), q(x)) ("3.5 Speculative Decoding", by-product
    of the proof)."""
    return float(np.minimum(p, q).sum())

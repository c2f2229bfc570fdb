"""Pins of the oracle's stochastic tree verification (reading R11), CPU only:
the chain special case against the pinned chain rule, the exactness claim
by chi-square over 10^5 seeded trials on a tiny vocabulary (the method the
verification contract prescribes), a perfect draft, and data errors."""
import numpy as np
import pytest

import oracle
import workloads
from enumeration import processed
from stats import chi_square_pvalue


def fits(tokens, P):
    """The tokens follow P: none outside its support, chi-square p > 1e-4."""
    counts = np.bincount(tokens, minlength=len(P))
    return counts[np.asarray(P) == 0].sum() == 0 and chi_square_pvalue(counts, P) > 1e-4


def test_chain_tree_is_the_chain_rule():
    """A tree whose nodes have one child each is ordinary speculative
    decoding: same tokens and counts as the chain oracle, except sequences
    within 1e-9 of a decision boundary (the tree draws from the normalised
    residual, the chain from the raw one)."""
    wl = workloads.c2()
    B, k, V = wl.B * 40, wl.k, 64
    rng = np.random.default_rng(3)
    tgt = rng.normal(0, 1.5, (B, k + 1, V)).astype(np.float32)
    drf = (tgt[:, :k] + rng.normal(0, 1.0, (B, k, V))).astype(np.float32)
    toks = workloads.gumbel_draw(rng, drf.astype(np.float64), 0.8).astype(np.int32)
    u = workloads.uniforms(rng, (B, k + 1))
    chain = oracle.verify_sample(tgt, drf, toks, u, T=0.8)
    parents = np.arange(-1, k, dtype=np.int32)
    tree_draft = np.concatenate([drf, drf[:, :1]], axis=1)  # the leaf's row is unused
    node_tokens = np.concatenate([np.zeros((B, 1), np.int32), toks], axis=1)
    tu = np.concatenate([u[:, k:], u[:, :k]], axis=1)  # entry 0: the final draw
    tree = oracle.verify_tree_sample(tgt, tree_draft, parents, node_tokens, tu, k, T=0.8)
    same = (tree["num_accepted"] == chain["num_accepted"]) & np.all(
        tree["tokens"] == chain["tokens"], axis=1)
    assert np.all(same | (tree["margin"] < 1e-9))
    assert same.mean() > 0.99
    np.testing.assert_array_equal(tree["path"][0, :tree["num_accepted"][0] + 1],
                                  np.arange(tree["num_accepted"][0] + 1))


def _mc_tree(rng, parents, P, Q, n, T=1.0, top_p=1.0, top_k=0, tgt=None, drf=None):
    """n trials: children drawn i.i.d. from their parent's draft law."""
    N = len(parents)
    V = P[0].shape[0]
    tok = np.zeros((n, N), np.int32)
    for c in range(1, N):
        tok[:, c] = rng.choice(V, size=n, p=Q[parents[c]])
    u = workloads.uniforms(rng, (n, N))
    D = int(max(depth_of(parents)))
    res = oracle.verify_tree_sample(np.broadcast_to(tgt, (n,) + tgt.shape).copy(),
                                    np.broadcast_to(drf, (n,) + drf.shape).copy(), parents, tok, u,
                                    D, T=T, top_p=top_p, top_k=top_k)
    return res


def depth_of(parents):
    d = np.zeros(len(parents), np.int64)
    for c in range(1, len(parents)):
        d[c] = d[parents[c]] + 1
    return d


@pytest.mark.parametrize("T,top_p,top_k", [(1.0, 1.0, 0), (0.8, 0.85, 0), (1.2, 1.0, 3)])
def test_exactness_chi_square(T, top_p, top_k):
    """10^5 trials on a tree with three i.i.d. candidates at the root and
    two under the first of them (V = 5): the first emitted token follows
    p_root, and the token after an accepted node c follows p_c."""
    rng = np.random.default_rng(11)
    V = 5
    parents = np.array([-1, 0, 0, 0, 1, 1, 2], np.int32)
    N = len(parents)
    tgt = rng.normal(0, 1.5, (N, V)).astype(np.float32)
    drf = (tgt + rng.normal(0, 1.2, (N, V))).astype(np.float32)
    P = [processed_k(tgt[i], T, top_p, top_k) for i in range(N)]
    Q = [processed_k(drf[i], T, top_p, top_k) for i in range(N)]
    n = 100_000
    res = _mc_tree(rng, parents, P, Q, n, T, top_p, top_k, tgt, drf)
    assert res["errors"] == 0
    first = res["tokens"][:, 0]
    assert fits(first, P[0])
    for c in (1, 2, 3):
        at = res["path"][:, 1] == c
        if at.sum() > 2000:
            assert fits(res["tokens"][at, 1], P[c])
    # every trial emits depth + 1 tokens, the path follows parents
    d = res["num_accepted"]
    assert np.all(d >= 0) and np.all(d <= 2)
    for i in np.nonzero(d >= 1)[0][:500]:
        path = res["path"][i, :d[i] + 1]
        assert path[0] == 0 and all(parents[path[j + 1]] == path[j] for j in range(d[i]))


def processed_k(logits, T, top_p, top_k):
    l = np.asarray(logits, np.float64)
    if 0 < top_k < l.shape[0]:
        kth = np.sort(l)[::-1][top_k - 1]
        l = np.where(l >= kth, l, -np.inf)
    return processed(l.astype(np.float32), T, top_p)


def test_perfect_draft_takes_first_children():
    rng = np.random.default_rng(2)
    V, B = 16, 50
    parents = np.array([-1, 0, 0, 1, 1, 3], np.int32)
    N = len(parents)
    tgt = rng.normal(0, 1.0, (B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    res = oracle.verify_tree_sample(tgt, tgt, parents, tok, workloads.uniforms(rng, (B, N)), 3)
    # with q = p every test u q(x) < p(x) passes: the walk is 0 -> 1 -> 3 -> 5
    np.testing.assert_array_equal(res["num_accepted"], 3)
    np.testing.assert_array_equal(res["path"], np.tile([0, 1, 3, 5], (B, 1)))


def test_data_errors():
    rng = np.random.default_rng(4)
    V, B = 8, 5
    parents = np.array([-1, 0, 0, 1], np.int32)
    tgt = rng.normal(0, 1.0, (B, 4, V)).astype(np.float32)
    drf = rng.normal(0, 1.0, (B, 4, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, 4)).astype(np.int32)
    u = workloads.uniforms(rng, (B, 4))
    tgt[0, 2, 1] = np.nan
    tok[1, 3] = V
    u[2, 0] = 1.0
    drf[3, 1, :] = -np.inf
    res = oracle.verify_tree_sample(tgt, drf, parents, tok, u, 2)
    assert list(res["num_accepted"][:4]) == [-1] * 4 and res["num_accepted"][4] >= 0
    assert res["errors"] == ((1 << oracle.ROW_NONFINITE) | (1 << oracle.TOKEN_RANGE) |
                             (1 << oracle.UNIFORM_RANGE) | (1 << oracle.ROW_ALL_NEG_INF))
    bad = oracle.verify_tree_sample(tgt[4:], drf[4:], np.array([-1, 0, 3, 1], np.int32),
                                    tok[4:], u[4:], 2)
    assert bad["num_accepted"][0] == -1 and bad["errors"] == 1 << oracle.TREE_SHAPE

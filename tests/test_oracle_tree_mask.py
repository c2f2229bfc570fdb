"""Pins of the oracle's tree attention mask and position builder (CPU only):
the page's 6-node tree, a transitive-closure brute force on random trees,
the tie to the tree verify rule, and malformed trees."""
import os

import numpy as np
import pytest

import oracle


def _golden(name):
    rows = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = vals
    return rows


def random_tree(rng, N, max_children=None):
    """parents in topological (not necessarily breadth-first) order."""
    par = np.empty(N, np.int32)
    par[0] = -1
    for n in range(1, N):
        par[n] = rng.integers(0, n) if max_children is None else max(0, n - 1 - rng.integers(0, max_children))
    return par


def closure(par):
    """Ancestor-or-self relation by repeated boolean squaring of the
    parent adjacency (no walk up the tree)."""
    N = len(par)
    A = np.eye(N, dtype=bool)
    for n in range(1, N):
        A[n, par[n]] = True
    R = A.copy()
    while True:
        R2 = (R.astype(np.int64) @ R.astype(np.int64)) > 0
        if np.array_equal(R2, R):
            return R.astype(np.uint8)
        R = R2


def bfs_depth(par):
    N = len(par)
    kids = [[] for _ in range(N)]
    for n in range(1, N):
        kids[par[n]].append(n)
    depth = np.full(N, -1, np.int64)
    depth[0] = 0
    frontier = [0]
    while frontier:
        nxt = []
        for u in frontier:
            for v in kids[u]:
                depth[v] = depth[u] + 1
                nxt.append(v)
        frontier = nxt
    return depth


def test_page_tree():
    """"3.5 Speculative Decoding", "Tree verification": the mask of the
    flattened [a, b, a1, a2, b1, b2] tree, every node seeing the context,
    and a1 / b1 sharing one position index."""
    g = _golden("lz_tree_mask.txt")
    par = np.array(g["parents"], np.int32)
    res = oracle.tree_mask(par[None], pos0=[100])
    assert res["errors"] == 0
    page = np.array([[int(v) for v in g[name]] for name in g["names"]], np.uint8)
    np.testing.assert_array_equal(res["mask"][0, 1:, 1:], page)
    assert np.all(res["mask"][0, :, 0] == 1)
    np.testing.assert_array_equal(res["pos"][0], 100 + np.array(g["depth"], np.int32))
    names = ["root"] + g["names"]
    assert res["pos"][0, names.index("a1")] == res["pos"][0, names.index("b1")]


@pytest.mark.parametrize("seed", range(6))
def test_random_trees_against_closure(seed):
    rng = np.random.default_rng(seed)
    B, N = 4, int(rng.integers(1, 60))
    par = np.stack([random_tree(rng, N) for _ in range(B)])
    pos0 = rng.integers(0, 1000, B).astype(np.int32)
    res = oracle.tree_mask(par, pos0)
    assert res["errors"] == 0
    for b in range(B):
        np.testing.assert_array_equal(res["mask"][b], closure(par[b]))
        np.testing.assert_array_equal(res["pos"][b], pos0[b] + bfs_depth(par[b]))
        # lower triangular with a unit diagonal; each row holds depth + 1 ones
        assert np.all(np.triu(res["mask"][b], 1) == 0)
        assert np.all(np.diag(res["mask"][b]) == 1)
        np.testing.assert_array_equal(res["mask"][b].sum(1), bfs_depth(par[b]) + 1)


def test_mask_agrees_with_tree_verification():
    """The node the greedy tree rule keeps is the deepest one whose masked
    ancestors (the path the mask exposes) all match their parent's argmax."""
    rng = np.random.default_rng(3)
    B, N, V = 40, 21, 6
    par = random_tree(rng, N, max_children=3)
    tgt = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    g = tgt.argmax(-1)
    tok = np.where(rng.random((B, N)) < 0.7, g[:, par.clip(0)], rng.integers(0, V, (B, N)))
    tok = tok.astype(np.int32)
    D = int(bfs_depth(par).max())
    ref = oracle.verify_tree(tgt, par, tok, D)
    m = oracle.tree_mask(par[None])["mask"][0]
    depth = bfs_depth(par)
    for b in range(B):
        ok = [all(tok[b, j] == g[b, par[j]] for j in range(1, N) if m[n, j]) for n in range(N)]
        best = max((depth[n], -n) for n in range(N) if ok[n])
        assert ref["num_accepted"][b] == best[0]
        assert ref["path"][b, best[0]] == -best[1]


def test_malformed_trees():
    good = np.array([-1, 0, 0, 1], np.int32)
    par = np.stack([good, [0, 0, 0, 1], [-1, 0, 2, 1], [-1, 0, -1, 1], good]).astype(np.int32)
    res = oracle.tree_mask(par, pos0=[5] * 5)
    assert res["errors"] == 1 << oracle.TREE_SHAPE
    for b in (1, 2, 3):
        assert np.all(res["mask"][b] == 0) and np.all(res["pos"][b] == -1)
    for b in (0, 4):
        np.testing.assert_array_equal(res["pos"][b], [5, 6, 6, 7])

"""Pins of the CPU oracle against the pages' worked examples, closed forms,
special cases and the readings' own edge cases (CPU only).

Golden fixtures live in tests/golden/, each citing its page and section.
"""
import os

import numpy as np
import pytest

import oracle
import workloads
from enumeration import acceptance_probability, cells, laws, nucleus_upper_set, softmax_T


def _golden(golden_dir, name):
    rows = {}
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = vals
    return rows


def _logits_of(p):
    """fp32 logits whose softmax is p (up to fp32 rounding of log p)."""
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _exact_single_position(p, q):
    """Exact law of one verify position (k = 1) by cell enumeration:
    returns (acceptance probability, law of the emitted token, residual)."""
    tgt = np.stack([_logits_of(p), _logits_of(p)])[None]
    drf = _logits_of(q)[None, None]
    P = [softmax_T(tgt[0, 0], 1.0), softmax_T(tgt[0, 1], 1.0)]
    Q = [softmax_T(drf[0, 0], 1.0)]
    cl = list(cells(P, Q))
    B = len(cl)
    res = oracle.verify_sample(
        np.repeat(tgt, B, 0), np.repeat(drf, B, 0),
        np.array([c[0] for c in cl], np.int32).reshape(B, 1),
        np.array([c[1] for c in cl], np.float32), T=1.0)
    w = np.array([c[2] for c in cl])
    law, reach = laws(P, Q, None, res["num_accepted"], res["tokens"], w)
    accept = w[res["num_accepted"] == 1].sum()
    rejected = res["num_accepted"] == 0
    resid = np.zeros(len(p))
    np.add.at(resid, res["tokens"][rejected, 0], w[rejected])
    return accept, law[0], resid / resid.sum()


def test_quiz_acceptance_and_residual(golden_dir):
    g = _golden(golden_dir, "lz_quiz_residual.txt")
    p = np.array(g["p"], float)
    q = np.array(g["q"], float)
    beta, law, resid = _exact_single_position(p, q)
    assert abs(beta - float(g["beta"][0])) < 1e-6
    np.testing.assert_allclose(resid, np.array(g["residual"], float), atol=1e-6)
    assert abs(law[0] - float(g["p_emit_a"][0])) < 1e-6
    np.testing.assert_allclose(law, p, atol=1e-6)


def test_misaligned_pair_v6(golden_dir):
    """Exact acceptance 0.55 and residual (2/3, 1/3, 0, ...), then the page's
    200,000-trial experiment re-run through the oracle: the acceptance rate
    and histogram agree with the exact values within 4 standard errors, and
    the page's own printed figures sit inside the same band."""
    g = _golden(golden_dir, "mn_exactness_v6.txt")
    p = np.array(g["p"], float)
    q = np.array(g["q"], float)
    beta, law, resid = _exact_single_position(p, q)
    assert abs(beta - float(g["beta_exact"][0])) < 1e-6
    np.testing.assert_allclose(resid, [2 / 3, 1 / 3, 0, 0, 0, 0], atol=1e-6)

    n = int(g["trials"][0])
    rng = np.random.default_rng(2024)
    tgt = np.broadcast_to(np.stack([_logits_of(p)] * 2), (n, 2, 6)).copy()
    drf = np.broadcast_to(_logits_of(q), (n, 1, 6)).copy()
    toks = workloads.gumbel_draw(rng, drf.astype(np.float64), 1.0).astype(np.int32)
    u = workloads.uniforms(rng, (n, 2))
    res = oracle.verify_sample(tgt, drf, toks, u, T=1.0)
    se = np.sqrt(0.55 * 0.45 / n)
    rate = (res["num_accepted"] == 1).mean()
    assert abs(rate - 0.55) < 4 * se
    assert abs(float(g["printed_accept_rate"][0]) - 0.55) < 4 * se
    emp = np.bincount(res["tokens"][:, 0], minlength=6) / n
    band = 4 * np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(emp - p) < band)
    printed = np.array(g["printed_empirical"], float)
    assert np.all(np.abs(printed - p) < band + 5e-5)  # printed to 4 decimals


def _closed_form(alpha, k):
    return (1 - alpha ** (k + 1)) / (1 - alpha)


def test_closed_form_table_matches_pages(golden_dir):
    """The printed values are the closed form, rounded as printed; and
    Bernoulli(alpha) acceptance chains reproduce the closed form."""
    rng = np.random.default_rng(3)
    with open(os.path.join(golden_dir, "expected_tokens_per_step.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for src, a, k, printed, tol in rows:
        a, k, printed, tol = float(a), int(k), float(printed), float(tol)
        assert abs(_closed_form(a, k) - printed) <= tol + 1e-12, (src, a, k)
        chains = rng.random((200_000, k)) < a
        emitted = 1 + np.cumprod(chains, axis=1).sum(axis=1)
        se = emitted.std() / np.sqrt(emitted.size)
        assert abs(emitted.mean() - _closed_form(a, k)) < 4 * se + 1e-12


@pytest.mark.parametrize("alpha,k", [(0.7, 3), (0.8, 4), (0.8, 10), (0.85, 5), (0.7, 8)])
def test_closed_form_through_oracle(alpha, k):
    """Real (p, q) with sum min(p, q) = alpha at every position, drafts drawn
    from q: the oracle's mean tokens per step matches (1 - alpha^(k+1)) /
    (1 - alpha) within 4 standard errors ("3.5 Speculative Decoding",
    "Expected tokens per step"; "Speculative Decoding from First Principles":
    alpha = 0.7, k = 3 -> 2.5 tokens per pass)."""
    d = (1 - alpha) / 2
    p = np.array([0.5 + d, 0.5 - d])
    q = np.array([0.5 - d, 0.5 + d])
    n = 100_000
    rng = np.random.default_rng(int(alpha * 100) + k)
    tgt = np.broadcast_to(_logits_of(p), (n, k + 1, 2)).copy()
    drf = np.broadcast_to(_logits_of(q), (n, k, 2)).copy()
    toks = workloads.gumbel_draw(rng, drf.astype(np.float64), 1.0).astype(np.int32)
    u = workloads.uniforms(rng, (n, k + 1))
    res = oracle.verify_sample(tgt, drf, toks, u, T=1.0)
    emitted = res["num_accepted"] + 1
    beta = acceptance_probability(softmax_T(tgt[0, 0], 1.0), softmax_T(drf[0, 0], 1.0))
    se = emitted.std() / np.sqrt(n)
    assert abs(emitted.mean() - _closed_form(beta, k)) < 4 * se


def test_greedy_worked_example(golden_dir):
    """"3.5 Speculative Decoding", "Worked example": accept, accept, reject
    -> emit the target's token; 3 tokens, no bonus."""
    rows = []
    with open(os.path.join(golden_dir, "lz_greedy_trace.txt")) as f:
        for line in f:
            if line.startswith("pos") or line.startswith("emitted"):
                rows.append([c.strip().strip('"') for c in line.split("|")])
            elif line.startswith("accepted"):
                accepted = int(line.split()[1])
    vocab = sorted({c for r in rows for c in r[1:] if c not in ("-",)})
    ids = {t: i for i, t in enumerate(vocab)}
    trace = [r for r in rows if r[0].startswith("pos")]
    k, V = len(trace) - 1, len(vocab)
    tgt = np.zeros((1, k + 1, V), np.float32)
    for i, r in enumerate(trace):
        tgt[0, i, ids[r[2]]] = 5.0
    drafts = np.array([[ids[r[1]] for r in trace[:k]]], np.int32)
    res = oracle.verify_sample(tgt, None, drafts, None, mode=oracle.GREEDY)
    emitted = [r for r in rows if r[0] == "emitted"][0][1:]
    assert res["num_accepted"][0] == accepted
    n = accepted + 1
    assert [vocab[t] for t in res["tokens"][0, :n]] == emitted
    assert np.all(res["tokens"][0, n:] == -1)


def test_tree_mask_from_parents(golden_dir):
    """The ancestor relation of the page's 6-node tree reproduces its tree
    attention mask ("3.5 Speculative Decoding", "Tree verification")."""
    g = _golden(golden_dir, "lz_tree_mask.txt")
    parents = np.array(g["parents"], np.int32)
    st, mask = oracle.ancestor_mask(parents)
    assert st == 0
    page = np.array([[int(v) for v in g[name]] for name in g["names"]], np.uint8)
    np.testing.assert_array_equal(mask[1:, 1:], page)
    assert np.all(mask[:, 0] == 1)  # every node sees the context (the root)


def _tree_bruteforce(parents, tok, g):
    """Deepest node whose whole root path passes the greedy test, ties to the
    lowest index; every node's path is checked from scratch."""
    best, best_d = 0, 0
    for n in range(1, len(parents)):
        path = [n]
        while path[-1] != 0:
            path.append(parents[path[-1]])
        ok = all(tok[c] == g[parents[c]] for c in path[:-1])
        if ok and len(path) - 1 > best_d:
            best, best_d = n, len(path) - 1
    return best, best_d


def test_tree_walk_matches_bruteforce():
    rng = np.random.default_rng(9)
    for trial in range(40):
        N = int(rng.integers(1, 30))
        parents = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)
        depth = np.zeros(N, int)
        for n in range(1, N):
            depth[n] = depth[parents[n]] + 1
        D = int(depth.max())
        B, V = 3, 4
        tgt = rng.normal(0, 1, (B, N, V)).astype(np.float32)
        g = tgt.argmax(axis=2)
        tok = rng.integers(0, V, (B, N)).astype(np.int32)
        res = oracle.verify_tree(tgt, parents, tok, D)
        assert res["errors"] == 0
        for b in range(B):
            best, d = _tree_bruteforce(parents, tok[b], g[b])
            assert res["num_accepted"][b] == d
            path = [best]
            while path[-1] != 0:
                path.append(parents[path[-1]])
            path = path[::-1]
            np.testing.assert_array_equal(res["path"][b, :d + 1], path)
            np.testing.assert_array_equal(res["tokens"][b, :d], tok[b, path[1:]])
            assert res["tokens"][b, d] == g[b, best]
            assert np.all(res["tokens"][b, d + 1:] == -1)


def test_tree_example_path():
    """On the page's tree: a accepted, a2 accepted under a -> depth 2, path
    root, a, a2; bonus = argmax of a2's row."""
    parents = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
    V = 10
    g = [3, 7, 1, 4, 2, 5, 6]  # argmax of each node's row
    tgt = np.zeros((1, 7, V), np.float32)
    for n, t in enumerate(g):
        tgt[0, n, t] = 1.0
    tok = np.array([[0, 3, 9, 0, 7, 8, 1]], np.int32)  # a=3 ok, a2=7 ok, a1 wrong
    res = oracle.verify_tree(tgt, parents, tok, 2)
    assert res["num_accepted"][0] == 2
    np.testing.assert_array_equal(res["path"][0], [0, 1, 4])
    np.testing.assert_array_equal(res["tokens"][0], [3, 7, 2])


def test_greedy_first_maximum():
    tgt = np.array([[[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0]]], np.float32)
    res = oracle.verify_sample(tgt, None, np.array([[2]], np.int32), None, mode=oracle.GREEDY)
    assert res["num_accepted"][0] == 0 and res["tokens"][0, 0] == 1
    res = oracle.verify_sample(tgt, None, np.array([[1]], np.int32), None, mode=oracle.GREEDY)
    assert res["num_accepted"][0] == 1 and list(res["tokens"][0]) == [1, 0]


def test_argmax_row_is_numpys_first_maximum():
    """Reading R5 (the greedy rule's argmax is the first maximum of the raw
    logits) reduces to numpy's argmax, which returns the first occurrence:
    random rows with planted ties, fp32 and bf16, rows holding -inf; a NaN
    or +inf fails the row, and so does a row of -inf only."""
    rng = np.random.default_rng(21)
    for V in (1, 2, 7, 33, 1000):
        for _ in range(20):
            row = np.round(rng.normal(0, 2, V) * 2).astype(np.float32) / 2  # ties
            if V > 2:
                row[rng.integers(0, V, 2)] = -np.inf
                row[rng.integers(0, V)] = row.max()  # a second copy of the max
            if np.isneginf(row).all():
                continue
            st, arg = oracle.argmax_row(row)
            assert st == 0 and arg == int(np.argmax(row)), (V, row)
            bits = workloads.to_bf16_bits(row)
            st, arg = oracle.argmax_row(bits)
            assert st == 0 and arg == int(np.argmax(workloads.as_f32(bits)))
    ok = np.array([0.5, 2.0, -1.0], np.float32)
    for bad in (np.nan, np.inf):
        row = ok.copy()
        row[2] = bad
        assert oracle.argmax_row(row)[0] == 1
    assert oracle.argmax_row(np.full(4, -np.inf, np.float32))[0] == 2


def test_inverse_cdf_against_searchsorted():
    """The draw is the textbook inverse CDF: numpy's searchsorted of u*S in
    the cumulative sums, side='right'."""
    rng = np.random.default_rng(4)
    for _ in range(200):
        V = int(rng.integers(1, 12))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[int(rng.integers(0, V))] = 1.0
        u = float(rng.random())
        tok, (S, c0, c1) = oracle.inverse_cdf(w, u)
        assert tok == int(np.searchsorted(np.cumsum(w), u * w.sum(), side="right"))
        assert w[tok] > 0 and c0 <= u * S < c1


@pytest.mark.parametrize("seed", range(6))
def test_top_p_matches_upper_set_bruteforce(seed):
    """Reading R1 (top-p is never defined on the pages): the kept set is the
    smallest upward-closed set with mass >= top_p, ties kept together."""
    rng = np.random.default_rng(seed)
    V = 8
    l = rng.normal(0, 1, V).astype(np.float32)
    l[rng.integers(0, V, 3)] = l[0]  # forced ties
    for top_p in (0.05, 0.3, 0.5, 0.77, 0.95, 0.999):
        p = softmax_T(l.astype(np.float64), 0.8)
        st, prob, info = oracle.process_row(l, T=0.8, top_p=top_p)
        assert st == 0
        np.testing.assert_allclose(prob, nucleus_upper_set(p, top_p), atol=1e-14)
        assert info[2] < top_p <= info[3] + 1e-15


def test_top_p_limits():
    l = np.array([2.0, 2.0, 1.0, 0.0, -1.0], np.float32)
    st, prob, _ = oracle.process_row(l, top_p=1e-9)  # only the top tie group
    np.testing.assert_allclose(prob, [0.5, 0.5, 0, 0, 0], atol=1e-15)
    st, prob, _ = oracle.process_row(l, top_p=1.0)
    np.testing.assert_allclose(prob, softmax_T(l.astype(np.float64), 1.0), atol=1e-15)


def test_zero_draft_probability_reading():
    """Reading R2 at q(x~) = 0: u*Q < P accepts iff P > 0; with P = Q = 0 the
    draft is rejected and, the residual being empty, the draw falls back to
    p (reading R4)."""
    tgt = _logits_of([[0.5, 0.5, 0.0], [1 / 3, 1 / 3, 1 / 3]])[None]
    u = np.array([[0.99, 0.5]], np.float32)
    res = oracle.verify_sample(tgt, _logits_of([[0.0, 0.5, 0.5]])[None],
                               np.array([[0]], np.int32), u)
    assert res["num_accepted"][0] == 1  # P = 0.5 > 0 = Q
    res = oracle.verify_sample(tgt, _logits_of([[0.5, 0.5, 0.0]])[None],
                               np.array([[2]], np.int32), u)
    assert res["num_accepted"][0] == 0  # P = Q = 0
    assert res["tokens"][0, 0] == 1     # u = 0.5 on p = (0.5, 0.5, 0)


def test_invariants_on_c2():
    wl = workloads.c2()
    res = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T)
    j = res["num_accepted"]
    assert np.all((j >= 0) & (j <= wl.k))
    for b in range(wl.B):
        np.testing.assert_array_equal(res["tokens"][b, :j[b]], wl.draft_tokens[b, :j[b]])
        assert 0 <= res["tokens"][b, j[b]] < wl.V
        assert np.all(res["tokens"][b, j[b] + 1:] == -1)


def test_data_errors():
    rng = np.random.default_rng(0)
    B, k, V = 6, 2, 16
    tgt = rng.normal(0, 1, (B, k + 1, V)).astype(np.float32)
    drf = rng.normal(0, 1, (B, k, V)).astype(np.float32)
    toks = rng.integers(0, V, (B, k)).astype(np.int32)
    u = workloads.uniforms(rng, (B, k + 1))
    tgt[1, 2, 5] = np.nan
    drf[2, 0, 3] = np.inf
    tgt[3, 0, :] = -np.inf
    toks[4, 1] = V
    u[5, 2] = 1.0
    res = oracle.verify_sample(tgt, drf, toks, u)
    want = {1: oracle.ROW_NONFINITE, 2: oracle.ROW_NONFINITE, 3: oracle.ROW_ALL_NEG_INF,
            4: oracle.TOKEN_RANGE, 5: oracle.UNIFORM_RANGE}
    assert res["errors"] == sum(1 << c for c in set(want.values()))
    for b in range(B):
        if b in want:
            assert res["num_accepted"][b] == -1 and np.all(res["tokens"][b] == -1)
        else:
            assert res["num_accepted"][b] >= 0
    # -inf entries alone are fine: probability 0
    tgt2 = tgt[:1].copy()
    tgt2[0, :, :4] = -np.inf
    res = oracle.verify_sample(tgt2, drf[:1], toks[:1], u[:1])
    assert res["errors"] == 0

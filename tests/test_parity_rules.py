"""The parity rule the GPU tests apply (tests/parity_rules.py) and the
oracle's boundary flags it rests on, checked on the CPU: inputs placed
exactly on each kind of decision boundary are flagged with that kind and
no other, and the rule accepts exactly the differences each flag allows.

Uniforms and top_p are put on the boundary by reading the oracle's own
debug values from a first run and rerunning with the uniform (or top_p)
set to the boundary value; the flags must then fire whatever the tie
went to.
"""
import numpy as np
import pytest

import oracle
import parity_rules


def _chain(B=6, k=3, V=40, seed=3):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.5, (B, k + 1, V)).astype(np.float32)
    drf = (tgt[:, :k] + rng.normal(0, 0.6, (B, k, V))).astype(np.float32)
    toks = rng.integers(0, V, (B, k)).astype(np.int32)
    # every draft token the draft's own argmax: q > 0 and a large P/Q span
    toks[:] = np.argmax(drf, axis=2)
    uni = rng.uniform(0.2, 0.8, (B, k + 1)).astype(np.float32)
    return tgt, drf, toks, uni


def _run(tgt, drf, toks, uni, top_p=1.0):
    return oracle.verify_sample(tgt, drf, toks, uni, T=1.0, top_p=top_p, debug=True)


def test_clean_inputs_are_not_flagged():
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni)
    acc, cdf, nuc = oracle.boundary_kinds(res, uni)
    assert not (acc | cdf | nuc).any()


def test_accept_ratio_boundary_is_flagged():
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni)
    k = toks.shape[1]
    P, Q = res["dbg"][:, :k], res["dbg"][:, k:2 * k]
    b = 2
    u = uni.copy()
    u[b, 0] = np.float32(min(P[b, 0] / Q[b, 0], 1.0 - 2.0 ** -24))  # position 1 is always tested
    res2 = _run(tgt, drf, toks, u)
    acc, cdf, nuc = oracle.boundary_kinds(res2, u)
    assert acc[b] and not nuc.any()
    assert not acc[np.arange(len(acc)) != b].any()


def test_cdf_edge_is_flagged():
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni)
    k = toks.shape[1]
    S, c0 = res["dbg"][:, 2 * k], res["dbg"][:, 2 * k + 1]
    b = 4
    u = uni.copy()
    u[b, k] = np.float32(c0[b] / S[b])  # the final uniform on the drawn token's lower edge
    res2 = _run(tgt, drf, toks, u)
    acc, cdf, nuc = oracle.boundary_kinds(res2, u)
    assert cdf[b] and not acc[b] and not nuc.any()


def test_nucleus_boundary_is_flagged():
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni, top_p=0.9)
    # top_p set to one row's mass at and above its threshold: that row's
    # kept set is then exactly at top_p
    b, r = 1, 2
    tp = float(res["row_info"][b, r, 3])
    res2 = _run(tgt, drf, toks, uni, top_p=tp)
    acc, cdf, nuc = oracle.boundary_kinds(res2, uni, top_p=tp)
    assert nuc[b]
    # without top-p nothing is a nucleus boundary
    assert not oracle.boundary_kinds(res2, uni, top_p=1.0)[2].any()


def test_invalid_sequences_are_never_flagged():
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni)
    k = toks.shape[1]
    P, Q = res["dbg"][:, :k], res["dbg"][:, k:2 * k]
    u = uni.copy()
    u[0, 0] = np.float32(min(P[0, 0] / Q[0, 0], 1.0 - 2.0 ** -24))
    tgt2 = tgt.copy()
    tgt2[0, 0, 5] = np.nan  # a data error fails sequence 0
    res2 = _run(tgt2, drf, toks, u)
    assert res2["num_accepted"][0] == -1
    assert not oracle.boundary_flags(res2, u)[0]


# ------------------------------------------------------------ the rule

def _ref_and_flags(kind):
    """An oracle result with exactly one flagged sequence of `kind` (or
    none), and that sequence's index."""
    tgt, drf, toks, uni = _chain()
    res = _run(tgt, drf, toks, uni)
    k = toks.shape[1]
    u, b = uni.copy(), 3
    if kind == "accept":
        P, Q = res["dbg"][:, :k], res["dbg"][:, k:2 * k]
        u[b, 0] = np.float32(min(P[b, 0] / Q[b, 0], 1.0 - 2.0 ** -24))
    elif kind == "cdf":
        u[b, k] = np.float32(res["dbg"][b, 2 * k + 1] / res["dbg"][b, 2 * k])
    ref = _run(tgt, drf, toks, u)
    return ref, u, b


def test_rule_accepts_identical_outputs():
    ref, u, _ = _ref_and_flags(None)
    parity_rules.check("same", ref["tokens"].copy(), ref["num_accepted"].copy(), ref, u, 1.0, 0)


def test_rule_rejects_an_unflagged_accept_count():
    ref, u, b = _ref_and_flags(None)
    n = ref["num_accepted"].copy()
    n[b] = (n[b] + 1) % (ref["tokens"].shape[1])
    with pytest.raises(AssertionError, match="accept counts differ"):
        parity_rules.check("bad n", ref["tokens"].copy(), n, ref, u, 1.0, 10)


def test_rule_rejects_an_unflagged_token():
    ref, u, b = _ref_and_flags(None)
    t = ref["tokens"].copy()
    t[b, ref["num_accepted"][b]] += 1
    with pytest.raises(AssertionError, match="unflagged mismatches"):
        parity_rules.check("bad t", t, ref["num_accepted"].copy(), ref, u, 1.0, 10)


def test_rule_on_a_cdf_edge_excuses_the_drawn_token_only():
    ref, u, b = _ref_and_flags("cdf")
    acc, cdf, nuc = oracle.boundary_kinds(ref, u)
    assert cdf[b] and not acc[b]
    j = ref["num_accepted"][b]
    t = ref["tokens"].copy()
    t[b, j] += 1  # the drawn token may differ
    parity_rules.check("cdf drawn", t, ref["num_accepted"].copy(), ref, u, 1.0, 1)
    n = ref["num_accepted"].copy()
    n[b] = (j + 1) % ref["tokens"].shape[1]  # the accept count may not
    with pytest.raises(AssertionError, match="accept counts differ"):
        parity_rules.check("cdf n", ref["tokens"].copy(), n, ref, u, 1.0, 1)
    assert j > 0  # this seed accepts a draft token there, to alter next
    t = ref["tokens"].copy()
    t[b, 0] += 1  # nor an accepted draft token
    with pytest.raises(AssertionError, match="beyond its drawn token"):
        parity_rules.check("cdf other", t, ref["num_accepted"].copy(), ref, u, 1.0, 1)


def test_rule_on_an_accept_boundary_excuses_the_count():
    ref, u, b = _ref_and_flags("accept")
    assert oracle.boundary_kinds(ref, u)[0][b]
    n = ref["num_accepted"].copy()
    t = ref["tokens"].copy()
    n[b] = 1 if n[b] == 0 else 0
    t[b] = -1
    t[b, 0] = 7
    parity_rules.check("acc", t, n, ref, u, 1.0, 1)
    # the budget still counts it
    with pytest.raises(AssertionError, match="budget"):
        parity_rules.check("acc budget", t, n, ref, u, 1.0, 0)

"""Pins of the oracle's top-k processing (reading R10) on CPU: a sort-based
brute force, the K = 1 reduction to the greedy rule, the no-op cases, and
exactness of the step when target and draft share top-k (and top-p)."""
import numpy as np
import pytest

import oracle
import workloads
from enumeration import cells, laws, nucleus_upper_set, softmax_T


def brute(logits, T, top_k, top_p):
    """Keep the top_k largest logits and all their ties (np.sort), softmax
    over them, then the upper-set nucleus."""
    l = workloads.as_f32(np.asarray(logits)).astype(np.float64)
    V = l.shape[0]
    if 0 < top_k < V:
        kth = np.sort(l)[::-1][top_k - 1]
        l = np.where(l >= kth, l, -np.inf)
    p = softmax_T(l, T)
    return nucleus_upper_set(p, top_p) if top_p < 1.0 else p


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (3, 1.0), (5, 0.8), (7, 0.95), (2, 0.5)])
def test_against_sort(dtype, top_k, top_p):
    rng = np.random.default_rng(top_k * 10 + int(top_p * 10))
    for r in range(6):
        l = (rng.normal(0, 2, 12) if r % 2 else np.round(rng.normal(0, 2, 12))).astype(np.float32)
        row = workloads.to_bf16_bits(l) if dtype == "bf16" else l
        st, p, _ = oracle.process_row(row, 0.9, top_p, top_k)
        assert st == 0
        np.testing.assert_allclose(p, brute(row, 0.9, top_k, top_p), atol=1e-12)
        assert np.count_nonzero(p) >= min(top_k, 12) if top_p == 1.0 else True


def test_ties_at_the_kth_are_kept():
    l = np.array([3.0, 1.0, 2.0, 2.0, 2.0, 0.0], np.float32)
    _, p, _ = oracle.process_row(l, 1.0, 1.0, 2)
    assert np.count_nonzero(p) == 4 and p[1] == 0.0 and p[5] == 0.0


@pytest.mark.parametrize("top_k", [0, -3, 8, 9, 100])
def test_no_op_values(top_k):
    l = np.random.default_rng(1).normal(0, 1, 8).astype(np.float32)
    np.testing.assert_array_equal(oracle.process_row(l, 0.7, 0.9, top_k)[1],
                                  oracle.process_row(l, 0.7, 0.9, 0)[1])


def test_k1_is_the_greedy_rule():
    """With top-k = 1 on target and draft, q is one-hot at the draft's
    argmax and p at the target's: the stochastic step with drafts at the
    draft argmax gives the greedy rule's tokens ("3.5 Speculative
    Decoding", end of the proof: accept iff the argmaxes agree)."""
    rng = np.random.default_rng(4)
    B, k, V = 64, 3, 50
    tgt = rng.normal(0, 1.5, (B, k + 1, V)).astype(np.float32)
    drf = np.where(rng.random((B, k, 1)) < 0.6, tgt[:, :k], rng.normal(0, 1.5, (B, k, V)))
    drf = drf.astype(np.float32)
    toks = drf.argmax(-1).astype(np.int32)
    u = workloads.uniforms(rng, (B, k + 1))
    st = oracle.verify_sample(tgt, drf, toks, u, T=0.8, top_k=1)
    gr = oracle.verify_sample(tgt, None, toks, None, mode=oracle.GREEDY)
    np.testing.assert_array_equal(st["num_accepted"], gr["num_accepted"])
    np.testing.assert_array_equal(st["tokens"], gr["tokens"])


@pytest.mark.parametrize("top_k,top_p", [(2, 1.0), (3, 0.9), (4, 0.7)])
def test_exactness_with_shared_top_k(top_k, top_p):
    """Cell enumeration (V = 6, k = 2): every emitted position has the law
    of the processed target row, and beta = the accept mass."""
    rng = np.random.default_rng(top_k)
    V, k, T = 6, 2, 0.9
    tgt = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    drf = (tgt[:k] + rng.normal(0, 1.0, (k, V))).astype(np.float32)
    P = [brute(tgt[i], T, top_k, top_p) for i in range(k + 1)]
    Q = [brute(drf[i], T, top_k, top_p) for i in range(k)]
    cl = list(cells(P, Q))
    n = len(cl)
    res = oracle.verify_sample(np.broadcast_to(tgt, (n, k + 1, V)).copy(),
                               np.broadcast_to(drf, (n, k, V)).copy(),
                               np.array([c[0] for c in cl], np.int32).reshape(n, k),
                               np.array([c[1] for c in cl], np.float32), T=T, top_p=top_p,
                               top_k=top_k)
    w = np.array([c[2] for c in cl])
    law, reach = laws(P, Q, None, res["num_accepted"], res["tokens"], w)
    assert reach[0] > 0.99
    for pos in range(k + 1):
        if reach[pos] > 1e-9:  # positions the drafts can reach at all
            np.testing.assert_allclose(law[pos] / reach[pos], P[pos], atol=1e-9)
    beta = oracle.acceptance(tgt[None], drf[None], T=T, top_p=top_p, top_k=top_k)["beta"][0, 0]
    assert abs(beta - np.minimum(P[0], Q[0]).sum()) < 1e-12

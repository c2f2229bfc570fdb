"""GPU parity of top-k processing (spec_verify_sample_topk and the top_k
arguments of the probability form and the acceptance rate) against the
oracle: same rules as the other parity tests (exact outside the flagged
near-boundary sequences; the top-k threshold itself is integer work on the
raw logits and has no boundary)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

import oracle  # noqa: E402
import speculative_decoding_verification_top_gb300 as sv  # noqa: E402
import workloads  # noqa: E402
import parity_rules  # noqa: E402
from test_gpu_parity import DEV, _small_chain, dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()
    oracle.build()


def topk_tokens(wl, K, seed):
    """Draft tokens from the draft's top-K (inside q's support)."""
    rng = np.random.default_rng(seed)
    wl.draft_tokens = workloads.gumbel_draw(rng, workloads.as_f32(wl.draft), wl.T,
                                            top=min(K, wl.V)).astype(np.int32)


def run(wl, K, mode=sv.SPEC_STOCHASTIC):
    stoch = mode == sv.SPEC_STOCHASTIC
    t, n, ws = sv.verify_sample(dev(wl.target), dev(wl.draft) if stoch else None,
                                dev(wl.draft_tokens), dev(wl.uniforms) if stoch else None,
                                temperature=wl.T, top_p=wl.top_p, mode=mode, top_k=K)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy(), ws


def check(wl, K, t, n, max_mismatch_frac=0.01):
    ref = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T,
                               top_p=wl.top_p, top_k=K, debug=True)
    parity_rules.check("%s K=%d top_p=%.2f" % (wl.name, K, wl.top_p), t, n, ref, wl.uniforms,
                       wl.top_p, max(2, int(max_mismatch_frac * wl.B)))
    return ref


@pytest.mark.parametrize("case", ["c4_k50", "c4_k20_nop", "c3_k40", "c2_k100_p09"])
def test_workloads(case):
    if case.startswith("c4"):
        wl = workloads.c4(B=32)
        K = 50 if case == "c4_k50" else 20
        if case == "c4_k20_nop":
            wl.top_p = 1.0
    elif case == "c3_k40":
        wl, K = workloads.c3(B=12), 40
    else:
        wl, K = workloads.c2(), 100
        wl.top_p = 0.9
    topk_tokens(wl, K, 3)
    t, n, ws = run(wl, K)
    check(wl, K, t, n)
    assert sv.last_error(ws) == 0


@pytest.mark.parametrize("V", [7, 33, 8193])
@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
@pytest.mark.parametrize("K,top_p", [(1, 1.0), (3, 1.0), (5, 0.9)])
def test_ragged_vocab(V, dtype, K, top_p):
    wl = _small_chain(6, 3, V, dtype, 0.8, top_p, seed=V + K)
    topk_tokens(wl, K, V)
    t, n, _ = run(wl, K)
    check(wl, K, t, n, max_mismatch_frac=0.02)


def test_ties_at_the_kth():
    """Logits rounded to halves (many ties), bf16: every tie of the K-th
    logit is kept."""
    wl = _small_chain(16, 3, 3000, workloads.BF16, 1.0, 1.0, seed=5, ties=True)
    topk_tokens(wl, 10, 5)
    t, n, _ = run(wl, 10)
    check(wl, 10, t, n, max_mismatch_frac=0.02)


def test_k1_equals_greedy():
    wl = _small_chain(32, 4, 5000, workloads.F32, 0.7, 1.0, seed=8)
    wl.draft_tokens = workloads.as_f32(wl.draft).argmax(-1).astype(np.int32)
    t, n, _ = run(wl, 1)
    gt, gn, _ = run(wl, 0, mode=sv.SPEC_GREEDY)
    np.testing.assert_array_equal(n, gn)
    np.testing.assert_array_equal(t, gt)


@pytest.mark.parametrize("K", [3000, 20000])
def test_k_beyond_the_near_max_list(K):
    """K far above the logits captured near the row's max (a few hundred on
    c4's rows): the K-th largest is found from the row, over wider
    windows."""
    wl = workloads.c4(B=6)
    topk_tokens(wl, K, 9)
    t, n, _ = run(wl, K)
    check(wl, K, t, n, max_mismatch_frac=0.02)


@pytest.mark.parametrize("K", [128, 129])
def test_at_the_warp_select_limit(K):
    """K at the largest the warp-per-row select takes (128) and one above
    (the row goes to the per-row CTA select, which bounds the K-th largest
    from the row summary itself)."""
    wl = workloads.c4(B=6)
    topk_tokens(wl, K, 11)
    t, n, ws = run(wl, K)
    check(wl, K, t, n, max_mismatch_frac=0.02)
    assert sv.last_error(ws) == 0


@pytest.mark.parametrize("V", [100003, 200003])
def test_rows_of_many_pieces(V):
    """Few rows of a large vocabulary: the statistics grid's warp segments
    are at their shortest, so a row spans 50 to 100 pieces -- more than the
    warp select maps, and at V = 200003 more than the CTA select stages (it
    then searches the row itself)."""
    wl = _small_chain(2, 1, V, workloads.BF16, 0.8, 0.9, seed=V)
    topk_tokens(wl, 50, 7)
    t, n, ws = run(wl, 50)
    check(wl, 50, t, n, max_mismatch_frac=0.02)
    assert sv.last_error(ws) == 0


def test_flat_rows_overflow_the_list():
    rng = np.random.default_rng(6)
    B, k, V = 6, 2, 20011
    tgt = rng.normal(0, 0.3, (B, k + 1, V)).astype(np.float32)
    drf = (tgt[:, :k] + rng.normal(0, 0.1, (B, k, V))).astype(np.float32)
    wl = workloads.Chain("flat", B, k, V, workloads.F32, 1.0, 0.9, tgt, drf, None,
                         workloads.uniforms(rng, (B, k + 1)))
    for K in (10, 6000):
        topk_tokens(wl, K, K)
        t, n, _ = run(wl, K)
        check(wl, K, t, n, max_mismatch_frac=0.02)


def test_acceptance_and_probability_form():
    wl = workloads.c4(B=8)
    K = 30
    topk_tokens(wl, K, 4)
    tg, dr = dev(wl.target), dev(wl.draft)
    _, _, ws = sv.verify_sample(tg, dr, dev(wl.draft_tokens), dev(wl.uniforms), temperature=wl.T,
                                top_p=wl.top_p, top_k=K)
    beta, tv = sv.acceptance(tg, dr, ws, temperature=wl.T, top_p=wl.top_p, top_k=K)
    torch.cuda.synchronize()
    ref = oracle.acceptance(wl.target, wl.draft, T=wl.T, top_p=wl.top_p, top_k=K)
    err = np.abs(beta.cpu().numpy() - ref["beta"])
    info = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T,
                                top_p=wl.top_p, top_k=K, debug=True)["row_info"]
    near = (np.abs(info[:, :, 2] - wl.top_p) < 1e-5) | (np.abs(info[:, :, 3] - wl.top_p) < 1e-5)
    skip = near[:, :wl.k] | near[:, wl.k + 1:]
    assert np.all((err <= 2e-3 * ref["beta"] + 1e-6) | skip)
    # probabilities form: top-k on the target rows only
    rng = np.random.default_rng(2)
    q, toks = workloads.draft_prob_rows(rng, workloads.as_f32(wl.target), wl.k)
    t, n, _ = sv.verify_sample_probs(tg, dev(q), dev(toks), dev(wl.uniforms), temperature=wl.T,
                                     top_p=wl.top_p, top_k=K)
    torch.cuda.synchronize()
    pref = oracle.verify_sample_probs(wl.target, q, toks, wl.uniforms, T=wl.T, top_p=wl.top_p,
                                      top_k=K, debug=True)
    parity_rules.check("%s probs K=%d" % (wl.name, K), t.cpu().numpy(), n.cpu().numpy(), pref,
                       wl.uniforms, wl.top_p, max(2, int(0.02 * wl.B)))

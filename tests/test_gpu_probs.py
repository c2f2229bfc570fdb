"""GPU parity of the verify step with the draft given as probabilities
(spec_verify_sample_probs) against the oracle's verify_sample_probs.

Same rules as the logits form: accept counts and tokens exact except for
sequences the oracle flags within 1e-5 of an accept-ratio, CDF or top-p
boundary; P_i, Q_i within the intermediate-probability tolerance (Q_i is a
gathered input here, so it must match exactly); S within 1e-5.
"""
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


def with_probs(wl, seed):
    rng = np.random.default_rng(seed)
    q, toks = workloads.draft_prob_rows(rng, workloads.as_f32(wl.target), wl.k)
    wl.draft_tokens = toks
    return q


def run_both(wl, q, target=None, qdev=None):
    t, n, ws = sv.verify_sample_probs(dev(wl.target) if target is None else target,
                                      dev(q) if qdev is None else qdev, dev(wl.draft_tokens),
                                      dev(wl.uniforms), temperature=wl.T, top_p=wl.top_p)
    torch.cuda.synchronize()
    ref = oracle.verify_sample_probs(wl.target, q, wl.draft_tokens, wl.uniforms, T=wl.T,
                                     top_p=wl.top_p, debug=True)
    return t.cpu().numpy(), n.cpu().numpy(), ws, ref


def check(wl, t, n, ws, ref, max_mismatch_frac=0.01):
    flags = parity_rules.check("%s probs" % wl.name, t, n, ref, wl.uniforms, wl.top_p,
                               max(2, int(max_mismatch_frac * wl.B)))
    print("accepted %s" % np.bincount(np.maximum(ref["num_accepted"], 0), minlength=wl.k + 1))
    P, Q, _, S = (x.cpu().numpy().astype(np.float64) for x in sv.intermediates(ws, wl.B, wl.k, wl.V))
    ok = ref["num_accepted"] >= 0
    k = wl.k
    rtol = 1e-5 if wl.dtype == workloads.F32 else 2e-3
    rP, rQ = ref["dbg"][:, :k], ref["dbg"][:, k:2 * k]
    assert np.all(np.abs(P - rP)[ok] <= (rtol * np.abs(rP) + 1e-30)[ok])
    np.testing.assert_array_equal(Q[ok], rQ[ok])
    same_j = ok & ~flags
    assert np.all(np.abs(S - ref["dbg"][:, 2 * k])[same_j] <= 1e-5)


@pytest.mark.parametrize("make", [workloads.c2, lambda: workloads.c3(B=24),
                                  lambda: workloads.c4(B=32)], ids=["c2", "c3", "c4"])
def test_workloads(make):
    wl = make()
    q = with_probs(wl, 11)
    t, n, ws, ref = run_both(wl, q)
    check(wl, t, n, ws, ref)
    assert sv.last_error(ws) == 0


@pytest.mark.parametrize("V", [1, 7, 9, 33, 8193, 40001])
@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_ragged_vocab(V, dtype, top_p):
    wl = _small_chain(6, 3, V, dtype, 0.9 if top_p == 1.0 else 0.3, top_p, seed=V + 3)
    q = with_probs(wl, V)
    t, n, ws, ref = run_both(wl, q)
    check(wl, t, n, ws, ref, max_mismatch_frac=0.02)


def test_large_nucleus_without_lists():
    """A 0.9-nucleus of ~2500 tokens: no nucleus list fits, so the residual
    and bonus draws stream the rows (the fp32 draft row with keys on p)."""
    rng = np.random.default_rng(5)
    B, k, V, H = 8, 2, 30011, 3000
    tgt = rng.normal(-4.0, 1.0, (B, k + 1, V)).astype(np.float32)
    for b in range(B):
        for i in range(k + 1):
            tgt[b, i, rng.choice(V, H, replace=False)] = rng.normal(4.0, 0.3, H)
    wl = workloads.Chain("large_nucleus", B, k, V, workloads.BF16, 1.0, 0.9,
                         workloads.to_bf16_bits(tgt), None, None,
                         workloads.uniforms(rng, (B, k + 1)))
    q = with_probs(wl, 2)
    t, n, ws, ref = run_both(wl, q)
    check(wl, t, n, ws, ref, max_mismatch_frac=0.02)


def test_same_outcome_as_the_logits_form():
    """q = the oracle's processed draft rows (fp32): the probabilities form
    gives the logits form's tokens wherever neither is near a boundary."""
    wl = workloads.c3(B=6)
    q = np.stack([[oracle.process_row(wl.draft[b, i], wl.T, wl.top_p)[1]
                   for i in range(wl.k)] for b in range(wl.B)]).astype(np.float32)
    t, n, ws, ref = run_both(wl, q)
    check(wl, t, n, ws, ref)
    lt, ln, _ = sv.verify_sample(dev(wl.target), dev(wl.draft), dev(wl.draft_tokens),
                                 dev(wl.uniforms), temperature=wl.T)
    lref = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T,
                                debug=True)
    near = oracle.boundary_flags(ref, wl.uniforms) | oracle.boundary_flags(lref, wl.uniforms)
    same = (ln.cpu().numpy() == n) & np.all(lt.cpu().numpy() == t, axis=1)
    assert np.all(same | near)


def test_unaligned_probability_rows():
    """draft_probs 4 bytes past a 16-byte boundary, V odd: element loads."""
    wl = _small_chain(4, 2, 5003, workloads.BF16, 1.0, 1.0, seed=13)
    q = with_probs(wl, 13)
    flat = torch.zeros(q.size + 1, dtype=torch.float32, device=DEV)
    flat[1:] = torch.from_numpy(q.ravel()).to(DEV)
    qd = flat[1:].view(q.shape)
    assert qd.data_ptr() % 16 != 0
    t, n, ws, ref = run_both(wl, q, qdev=qd)
    check(wl, t, n, ws, ref, max_mismatch_frac=0.02)


def test_gathered_probability_errors():
    wl = _small_chain(6, 3, 3000, workloads.F32, 1.0, 1.0, seed=17)
    q = with_probs(wl, 17)
    x = wl.draft_tokens
    q[0, 1, x[0, 1]] = np.nan
    q[1, 0, x[1, 0]] = -0.5
    q[2, 2, x[2, 2]] = 1.25
    t, n, ws, ref = run_both(wl, q)
    np.testing.assert_array_equal(n, ref["num_accepted"])
    np.testing.assert_array_equal(t, ref["tokens"])
    assert list(n[:3]) == [-1, -1, -1] and np.all(n[3:] >= 0)
    assert sv.last_error(ws) == sv.SPEC_DATA_PROB_RANGE


def test_argument_errors():
    wl = _small_chain(2, 2, 64, workloads.F32, 1.0, 1.0, seed=0)
    q = with_probs(wl, 0)
    tg, qd = dev(wl.target), dev(q)
    tk, un = dev(wl.draft_tokens), dev(wl.uniforms)
    ws = sv.new_workspace(sv.spec_verify_workspace_size(2, 2, 64), DEV)
    out_t = torch.empty((2, 3), dtype=torch.int32, device=DEV)
    out_n = torch.empty((2,), dtype=torch.int32, device=DEV)
    args = [tg.data_ptr(), qd.data_ptr(), tk.data_ptr(), un.data_ptr(), 2, 2, 64, 1.0, 1.0, 0,
            sv.SPEC_F32, out_t.data_ptr(), out_n.data_ptr(), ws.data_ptr(), ws.numel()]
    bad = list(args)
    bad[1] = qd.data_ptr() + 2  # not 4-byte aligned
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_sample_probs(*bad)
    bad = list(args)
    bad[7] = -1.0
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_sample_probs(*bad)
    assert sv.spec_verify_sample_probs(*args) == 0

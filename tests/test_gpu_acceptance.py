"""GPU parity of the per-position acceptance rate (spec_verify_acceptance)
against the oracle's beta = sum min(p, q) and TV = (1/2) sum |p - q|.

Tolerance: the intermediate-probability rule of the verification contract,
relative 1e-5 on fp32 inputs and 2e-3 on bf16 inputs, plus 1e-6 absolute
(beta is a sum of probabilities each carrying that relative error; a sum of
non-negative terms keeps it).  TV is compared within the same bound on
beta, since the library reports it as 1 - beta.  With top-p, a pair whose
target or draft row has its nucleus mass within 1e-5 of top_p may keep a
different token set in fp32 than in fp64; such pairs are counted and
skipped.
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
from test_gpu_parity import DEV, _small_chain, dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()
    oracle.build()


def gpu_beta(wl, two_phase=False):
    """Verify call, then the acceptance call on its workspace."""
    tg, dr = dev(wl.target), dev(wl.draft)
    tk, un = dev(wl.draft_tokens), dev(wl.uniforms)
    if two_phase:
        out_t = torch.empty((wl.B, wl.k + 1), dtype=torch.int32, device=DEV)
        out_n = torch.empty((wl.B,), dtype=torch.int32, device=DEV)
        ws = sv.new_workspace(sv.spec_verify_workspace_size(wl.B, wl.k, wl.V), DEV)
        stream = torch.cuda.current_stream().cuda_stream
        dt = sv.SPEC_BF16 if wl.dtype == workloads.BF16 else sv.SPEC_F32
        args = (tg.data_ptr(), dr.data_ptr(), tk.data_ptr(), un.data_ptr(), wl.B, wl.k, wl.V,
                wl.T, wl.top_p, sv.SPEC_STOCHASTIC, dt, out_t.data_ptr(), out_n.data_ptr(),
                ws.data_ptr(), ws.numel(), stream)
        sv.spec_verify_sample_rows(*args)
        beta, tv = sv.acceptance(tg, dr, ws, temperature=wl.T, top_p=wl.top_p)
        sv.spec_verify_sample_finish(*args)
    else:
        out_t, out_n, ws = sv.verify_sample(tg, dr, tk, un, temperature=wl.T, top_p=wl.top_p)
        beta, tv = sv.acceptance(tg, dr, ws, temperature=wl.T, top_p=wl.top_p)
    torch.cuda.synchronize()
    return (beta.cpu().numpy().astype(np.float64), tv.cpu().numpy().astype(np.float64),
            out_t.cpu().numpy(), out_n.cpu().numpy())


def nucleus_edge_pairs(wl, tol=1e-5):
    """[B, k] pairs whose target or draft row sits within tol of top_p."""
    if wl.top_p >= 1.0:
        return np.zeros((wl.B, wl.k), bool)
    res = oracle.verify_sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T=wl.T,
                               top_p=wl.top_p, debug=True)
    info = res["row_info"]
    near = (np.abs(info[:, :, 2] - wl.top_p) < tol) | (np.abs(info[:, :, 3] - wl.top_p) < tol)
    k = wl.k
    return near[:, :k] | near[:, k + 1:2 * k + 1]


def check(wl, beta, tv):
    ref = oracle.acceptance(wl.target, wl.draft, T=wl.T, top_p=wl.top_p)
    rb, rt = ref["beta"], ref["tv"]
    nan = np.isnan(rb)
    np.testing.assert_array_equal(np.isnan(beta), nan)
    np.testing.assert_array_equal(np.isnan(tv), nan)
    skip = nucleus_edge_pairs(wl) | nan
    rtol = 1e-5 if wl.dtype == workloads.F32 else 2e-3
    lim = rtol * np.abs(rb) + 1e-6
    err_b = np.where(skip, 0.0, np.abs(beta - rb))
    err_t = np.where(skip, 0.0, np.abs(tv - rt))
    print("%s B=%d k=%d V=%d: max |beta err| %.3g, max |tv err| %.3g, skipped %d, "
          "mean beta %.4f" % (wl.name, wl.B, wl.k, wl.V, err_b.max(), err_t.max(), skip.sum(),
                              np.nanmean(rb)))
    assert np.all(err_b <= np.where(skip, np.inf, lim))
    assert np.all(err_t <= np.where(skip, np.inf, lim))
    # How many rows sit near the boundary is a property of the inputs (at
    # small V each token moves the cumulative mass by ~1e-4); nearly every
    # pair must still be compared.
    assert skip[~nan].sum() <= max(2, 0.05 * (~nan).sum())
    return rb


@pytest.mark.parametrize("make", [workloads.c2, lambda: workloads.c3(B=64),
                                  lambda: workloads.c4(B=128)], ids=["c2", "c3", "c4"])
def test_workloads(make):
    wl = make()
    beta, tv, _, _ = gpu_beta(wl)
    rb = check(wl, beta, tv)
    assert np.all((rb > 0) & (rb <= 1))


@pytest.mark.parametrize("V", [1, 7, 9, 33, 8193, 40001])
@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_ragged_vocab(V, dtype, top_p):
    """Odd V puts target and draft rows at different offsets from 16-byte
    boundaries (element loads).  With top-p the rows are sharpened (T = 0.3)
    so that the nucleus is small and its mass steps are large: the pairs go
    through the nucleus lists and few sit near the top-p boundary."""
    wl = _small_chain(5, 3, V, dtype, 0.9 if top_p == 1.0 else 0.3, top_p, seed=V + 7)
    beta, tv, _, _ = gpu_beta(wl)
    check(wl, beta, tv)


@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
def test_large_nucleus_streams_the_rows(dtype):
    """Rows whose 0.9-nucleus holds ~2700 tokens (a flat group of 3000 high
    logits over V = 30011): no nucleus list fits, so both rows of every pair
    are streamed with nucleus keys.  Each high token moves the cumulative
    mass by ~3e-4, so few rows sit within 1e-5 of top_p."""
    rng = np.random.default_rng(5)
    B, k, V, H = 8, 2, 30011, 3000
    def rows(n):
        out = rng.normal(-4.0, 1.0, (n, V)).astype(np.float32)
        for r in range(n):
            out[r, rng.choice(V, H, replace=False)] = rng.normal(4.0, 0.3, H)
        return out
    tgt = rows(B * (k + 1)).reshape(B, k + 1, V)
    drf = (tgt[:, :k] + rng.normal(0, 0.2, (B, k, V))).astype(np.float32)
    store = workloads.to_bf16_bits if dtype == workloads.BF16 else (lambda a: a)
    wl = workloads.Chain("large_nucleus", B, k, V, dtype, 1.0, 0.9, store(tgt), store(drf),
                         rng.integers(0, V, (B, k)).astype(np.int32),
                         workloads.uniforms(rng, (B, k + 1)))
    beta, tv, _, _ = gpu_beta(wl)
    check(wl, beta, tv)


def test_between_phases_leaves_the_step_unchanged():
    for wl in (workloads.c4(B=4), workloads.c3(B=6)):
        b1, t1, tok1, n1 = gpu_beta(wl)
        b2, t2, tok2, n2 = gpu_beta(wl, two_phase=True)
        np.testing.assert_array_equal(tok1, tok2)
        np.testing.assert_array_equal(n1, n2)
        np.testing.assert_array_equal(b1, b2)
        np.testing.assert_array_equal(t1, t2)


def test_identical_draft_and_reproducible():
    wl = _small_chain(8, 4, 20000, workloads.BF16, 0.8, 1.0, seed=3)
    wl.draft = np.ascontiguousarray(wl.target[:, :wl.k])
    b1, t1, _, _ = gpu_beta(wl)
    b2, t2, _, _ = gpu_beta(wl)
    np.testing.assert_array_equal(b1, b2)
    assert np.all(np.abs(b1 - 1.0) < 2e-5) and np.all(t1 >= 0)
    check(wl, b1, t1)


def test_data_errors_give_nan():
    wl = _small_chain(4, 3, 3000, workloads.F32, 1.0, 1.0, seed=9)
    wl.target[1, 2, 17] = np.nan
    wl.draft[2, 0, :] = -np.inf
    wl.target[3, 3, 5] = np.inf  # the bonus row is not part of any pair
    beta, tv, _, n = gpu_beta(wl)
    check(wl, beta, tv)
    assert np.isnan(beta[1, 2]) and np.isnan(beta[2, 0])
    assert np.isfinite(beta[3]).all() and n[3] == -1


def test_argument_errors():
    wl = _small_chain(2, 2, 64, workloads.F32, 1.0, 1.0, seed=0)
    tg, dr = dev(wl.target), dev(wl.draft)
    _, _, ws = sv.verify_sample(tg, dr, dev(wl.draft_tokens), dev(wl.uniforms))
    out = torch.empty((2, 2), dtype=torch.float32, device=DEV)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_acceptance(tg.data_ptr(), dr.data_ptr(), 2, 2, 64, 0.0, 1.0, 0, sv.SPEC_F32,
                                  out.data_ptr(), None, ws.data_ptr(), ws.numel())
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_acceptance(tg.data_ptr(), dr.data_ptr(), 2, 2, 64, 1.0, 1.0, 0, sv.SPEC_F32,
                                  out.data_ptr(), None, ws.data_ptr(), 16)
    assert sv.spec_verify_acceptance(None, None, 0, 2, 64, 1.0, 1.0, 0, sv.SPEC_F32, None, None,
                                     None, 0) == 0

"""GPU parity: the CUDA library, called through its C ABI, against the fp64
CPU oracle on identical seeded inputs.

Rules (from the verification contract):
  * accept counts, greedy tokens and tree outputs: bit-exact;
  * sampled tokens: exact, except sequences the oracle flags as lying within
    1e-5 of an accept-ratio, CDF or top-p boundary -- those are counted and
    reported, and must stay rare;
  * intermediates P_i, Q_i, Z: relative error <= 1e-5 on fp32 inputs and
    <= 2e-3 on bf16 inputs; the draw total S within 1e-5 absolute.
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
from stats import position_fits  # noqa: E402
from enumeration import cells, processed  # noqa: E402
import parity_rules  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()
    oracle.build()


def dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_gpu(wl, mode=sv.SPEC_STOCHASTIC, workspace=None):
    stoch = mode == sv.SPEC_STOCHASTIC
    t, n, ws = sv.verify_sample(dev(wl.target), dev(wl.draft) if stoch else None,
                                dev(wl.draft_tokens), dev(wl.uniforms) if stoch else None,
                                temperature=wl.T, top_p=wl.top_p, mode=mode, workspace=workspace)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy(), ws


def run_oracle(wl, mode=oracle.STOCHASTIC):
    stoch = mode == oracle.STOCHASTIC
    return oracle.verify_sample(wl.target, wl.draft if stoch else None, wl.draft_tokens,
                                wl.uniforms if stoch else None, T=wl.T, top_p=wl.top_p,
                                mode=mode, debug=stoch)


def check_stochastic(wl, gpu_t, gpu_n, ref, max_mismatch_frac=0.01):
    """The parity rule (tests/parity_rules.py): accept counts bit-exact off
    accept-ratio and top-p boundaries, tokens exact off every boundary (a
    CDF edge excuses the drawn token alone), mismatches within
    max(2, max_mismatch_frac B)."""
    return parity_rules.check(wl.name, gpu_t, gpu_n, ref, wl.uniforms, wl.top_p,
                              max(2, int(max_mismatch_frac * wl.B)))


def check_intermediates(wl, ws, ref, flags):
    P, Q, Z, S = (x.cpu().numpy().astype(np.float64)
                  for x in sv.intermediates(ws, wl.B, wl.k, wl.V))
    ok = (ref["num_accepted"] >= 0)
    rtol = 1e-5 if wl.dtype == workloads.F32 else 2e-3
    k = wl.k
    rP, rQ = ref["dbg"][:, :k], ref["dbg"][:, k:2 * k]
    # P, Q and the recorded normaliser are taken over the nucleus: on a
    # sequence with a row whose prefix mass lies at top_p (the oracle's
    # nucleus flag) the kept set, and so that normaliser, depends on the
    # order of the sums.
    nuc = oracle.boundary_kinds(ref, wl.uniforms, wl.top_p)[2]
    pq = ok & ~nuc
    print("%s P/Q compared on %d of %d sequences (nucleus-flagged: %d)"
          % (wl.name, pq.sum(), ok.sum(), (ok & nuc).sum()))
    for got, want, name in ((P, rP, "P"), (Q, rQ, "Q")):
        if not pq.any():
            continue
        err = np.abs(got - want)[pq]
        lim = (rtol * np.abs(want) + 1e-30)[pq]
        print("%s %s max rel err %.3g" % (wl.name, name, (err / np.maximum(np.abs(want[pq]), 1e-30)).max()))
        assert np.all(err <= lim), name
    info = ref["row_info"]
    rZ = info[:, :, 0] * info[:, :, 3]
    zerr = (np.abs(Z - rZ) / rZ)[pq]
    print("%s Z max rel err %.3g" % (wl.name, zerr.max() if zerr.size else 0.0))
    assert np.all(zerr <= rtol)
    # S is compared where both sides drew from the same row.
    same_j = ok & ~flags
    serr = np.abs(S - ref["dbg"][:, 2 * k])[same_j]
    print("%s S max abs err %.3g" % (wl.name, serr.max() if serr.size else 0.0))
    assert np.all(serr <= 1e-5)


# ----------------------------------------------------------- workloads

def test_c2_stochastic_greedy_and_intermediates():
    wl = workloads.c2()
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    flags = check_stochastic(wl, t, n, ref)
    check_intermediates(wl, ws, ref, flags)
    gt, gn, _ = run_gpu(wl, sv.SPEC_GREEDY)
    gref = run_oracle(wl, oracle.GREEDY)
    np.testing.assert_array_equal(gn, gref["num_accepted"])
    np.testing.assert_array_equal(gt, gref["tokens"])


def test_c1_exactness_chi_square():
    """10^5 steps of the tiny case: parity with the oracle, and the GPU's own
    tokens pass the chi-square test against p at every position."""
    wl = workloads.c1()
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    check_stochastic(wl, t, n, ref)
    from enumeration import softmax_T
    P = [softmax_T(wl.target[0, i].astype(np.float64), wl.T) for i in range(wl.k + 1)]
    pv = position_fits(t, n, P, wl.V)
    print("c1 GPU chi-square p-values", pv)
    assert min(pv) > 1e-3
    assert np.all((n >= 0) & (n <= wl.k))


@pytest.mark.parametrize("B", [6, 64])
def test_c3(B):
    wl = workloads.c3(B=B)
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    flags = check_stochastic(wl, t, n, ref)
    check_intermediates(wl, ws, ref, flags)


@pytest.mark.parametrize("B", [4, 128])
def test_c4_top_p(B):
    wl = workloads.c4(B=B)
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    flags = check_stochastic(wl, t, n, ref)
    check_intermediates(wl, ws, ref, flags)
    # the top-16 drafter stays inside the draft nucleus (Q > 0) almost always
    assert np.mean(ref["dbg"][:, wl.k:2 * wl.k] == 0) < 0.01


def test_c5_tree():
    tr = workloads.c5()
    t, n, p, ws = sv.verify_tree(dev(tr.target), dev(tr.parents), dev(tr.node_tokens), tr.D)
    ref = oracle.verify_tree(tr.target, tr.parents, tr.node_tokens, tr.D)
    np.testing.assert_array_equal(n.cpu().numpy(), ref["num_accepted"])
    np.testing.assert_array_equal(t.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(p.cpu().numpy(), ref["path"])
    assert sv.last_error(ws) == 0
    print("c5 accepted depths", ref["num_accepted"])


# ------------------------------------------------------------ edge cases

def _small_chain(B, k, V, dtype, T, top_p, seed, ties=False):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    drf = (tgt[:, :k] + rng.normal(0, 1.0, (B, k, V))).astype(np.float32)
    if ties:
        tgt = np.round(tgt * 2) / 2
        drf = np.round(drf * 2) / 2
    store = workloads.to_bf16_bits if dtype == workloads.BF16 else (lambda a: a)
    tgt, drf = store(tgt), store(drf)
    toks = workloads.gumbel_draw(rng, workloads.as_f32(drf), T).astype(np.int32)
    return workloads.Chain("edge", B, k, V, dtype, T, top_p, tgt, drf, toks,
                           workloads.uniforms(rng, (B, k + 1)))


@pytest.mark.parametrize("V", [1, 7, 8, 9, 33, 1000, 1025, 2048, 2049, 8191, 8193, 16383,
                               16384, 16385, 40001])
@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
def test_ragged_vocab(V, dtype):
    for top_p in (1.0, 0.9):
        wl = _small_chain(5, 3, V, dtype, 0.9, top_p, seed=V)
        t, n, ws = run_gpu(wl)
        ref = run_oracle(wl)
        flags = check_stochastic(wl, t, n, ref, max_mismatch_frac=0.02)
        check_intermediates(wl, ws, ref, flags)
    gt, gn, _ = run_gpu(wl, sv.SPEC_GREEDY)
    gref = run_oracle(wl, oracle.GREEDY)
    np.testing.assert_array_equal(gn, gref["num_accepted"])
    np.testing.assert_array_equal(gt, gref["tokens"])


@pytest.mark.parametrize("V,dtype", [(131071, workloads.F32), (262147, workloads.BF16)])
def test_top_p_long_rows(V, dtype):
    """Rows too long for the fused top-p kernel's shared-memory summary
    (fp32 V = 131071, bf16 V = 262147): it keeps the logits near the running
    max as they stream by instead."""
    wl = _small_chain(3, 2, V, dtype, 0.8, 0.9, seed=V)
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    flags = check_stochastic(wl, t, n, ref, max_mismatch_frac=0.02)
    check_intermediates(wl, ws, ref, flags)


@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
def test_unaligned_base(dtype):
    """Logit arrays that start one element past a 16-byte boundary."""
    wl = _small_chain(4, 2, 5003, dtype, 1.0, 0.95, seed=11)
    def shifted(a):
        flat = np.zeros(a.size + 1, a.dtype)
        flat[1:] = a.ravel()
        t = dev(flat)[1:]
        return t.view(a.shape)
    tg, dr = shifted(wl.target), shifted(wl.draft)
    assert tg.data_ptr() % 16 != 0
    t, n, ws = sv.verify_sample(tg, dr, dev(wl.draft_tokens), dev(wl.uniforms),
                                temperature=wl.T, top_p=wl.top_p)
    ref = run_oracle(wl)
    check_stochastic(wl, t.cpu().numpy(), n.cpu().numpy(), ref, max_mismatch_frac=0.02)


@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
@pytest.mark.parametrize("top_p", [0.3, 0.8, 0.97])
def test_top_p_with_ties(dtype, top_p):
    wl = _small_chain(16, 3, 3000, dtype, 1.0, top_p, seed=int(top_p * 100), ties=True)
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    flags = check_stochastic(wl, t, n, ref, max_mismatch_frac=0.02)
    check_intermediates(wl, ws, ref, flags)


@pytest.mark.parametrize("k", [1, 2, 31])
def test_draft_length_limits(k):
    wl = _small_chain(3, k, 2000, workloads.F32, 1.0, 1.0, seed=k)
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    check_stochastic(wl, t, n, ref, max_mismatch_frac=0.02)
    gt, gn, _ = run_gpu(wl, sv.SPEC_GREEDY)
    gref = run_oracle(wl, oracle.GREEDY)
    np.testing.assert_array_equal(gt, gref["tokens"])


def test_identical_draft_accepts_everything():
    wl = _small_chain(32, 4, 5000, workloads.BF16, 0.8, 1.0, seed=3)
    wl.draft = np.ascontiguousarray(wl.target[:, :wl.k])
    t, n, ws = run_gpu(wl)
    assert np.all(n == wl.k)
    ref = run_oracle(wl)
    check_stochastic(wl, t, n, ref)


def test_enumeration_cells_match_exactly():
    """Every cell midpoint of a tiny step (V=6, k=3; far from boundaries):
    the GPU and the oracle agree on every one."""
    rng = np.random.default_rng(21)
    V, k, T = 6, 3, 0.8
    tgt = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    drf = (tgt[:k] + rng.normal(0, 1.0, (k, V))).astype(np.float32)
    P = [processed(tgt[i].astype(np.float64), T, 1.0) for i in range(k + 1)]
    Q = [processed(drf[i].astype(np.float64), T, 1.0) for i in range(k)]
    cl = list(cells(P, Q))
    B = len(cl)
    wl = workloads.Chain("cells", B, k, V, workloads.F32, T, 1.0,
                         np.ascontiguousarray(np.broadcast_to(tgt, (B, k + 1, V))),
                         np.ascontiguousarray(np.broadcast_to(drf, (B, k, V))),
                         np.array([c[0] for c in cl], np.int32).reshape(B, k),
                         np.array([c[1] for c in cl], np.float32))
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    np.testing.assert_array_equal(n, ref["num_accepted"])
    np.testing.assert_array_equal(t, ref["tokens"])


def test_repeated_calls_are_bitwise_reproducible():
    wl = workloads.c3(B=6)
    t1, n1, ws = run_gpu(wl)
    I1 = [x.cpu().numpy() for x in sv.intermediates(ws, wl.B, wl.k, wl.V)]
    t2, n2, _ = run_gpu(wl, workspace=ws)
    I2 = [x.cpu().numpy() for x in sv.intermediates(ws, wl.B, wl.k, wl.V)]
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(n1, n2)
    for a, b in zip(I1, I2):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("make", [
    lambda: workloads.c4(B=4), lambda: workloads.c3(B=6),
    # short rows, one row per warp: the whole call draws inside the rows
    # kernel, the two-phase call in the final kernel (NS = 1 and 2 sub-tiles)
    lambda: _small_chain(40, 3, 1000, workloads.F32, 0.8, 1.0, seed=11),
    lambda: _small_chain(40, 4, 2048, workloads.BF16, 1.2, 1.0, seed=12)],
    ids=["top_p_rows", "stream_rows", "short_rows_f32", "short_rows_bf16"])
def test_two_phase_api_equals_single_call(make):
    wl = make()
    t1, n1, _ = run_gpu(wl)
    tg, dr, tk, un = dev(wl.target), dev(wl.draft), dev(wl.draft_tokens), dev(wl.uniforms)
    out_t = torch.empty((wl.B, wl.k + 1), dtype=torch.int32, device=DEV)
    out_n = torch.empty((wl.B,), dtype=torch.int32, device=DEV)
    nbytes = sv.spec_verify_workspace_size(wl.B, wl.k, wl.V)
    ws = sv.new_workspace(nbytes, DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = (tg.data_ptr(), dr.data_ptr(), tk.data_ptr(), un.data_ptr(), wl.B, wl.k, wl.V, wl.T,
            wl.top_p, sv.SPEC_STOCHASTIC,
            sv.SPEC_BF16 if wl.dtype == workloads.BF16 else sv.SPEC_F32,
            out_t.data_ptr(), out_n.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    sv.spec_verify_sample_rows(*args)
    sv.spec_verify_sample_finish(*args)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_t.cpu().numpy(), t1)
    np.testing.assert_array_equal(out_n.cpu().numpy(), n1)


def test_empty_batch():
    wl = _small_chain(1, 2, 64, workloads.F32, 1.0, 1.0, seed=0)
    t = torch.empty((0, 3, 64), dtype=torch.float32, device=DEV)
    d = torch.empty((0, 2, 64), dtype=torch.float32, device=DEV)
    out_t, out_n, ws = sv.verify_sample(t, d, torch.empty((0, 2), dtype=torch.int32, device=DEV),
                                        torch.empty((0, 3), dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert out_t.shape == (0, 3) and out_n.shape == (0,)


# ----------------------------------------------------------- data errors

def test_data_errors_match_oracle():
    wl = _small_chain(8, 2, 700, workloads.F32, 1.0, 1.0, seed=5)
    wl.target[1, 2, 5] = np.nan
    wl.draft[2, 0, 3] = np.inf
    wl.target[3, 0, :] = -np.inf
    wl.draft_tokens[4, 1] = wl.V
    wl.uniforms[5, 2] = 1.0
    wl.target[6, 1, :10] = -np.inf  # -inf entries alone are fine
    t, n, ws = run_gpu(wl)
    ref = run_oracle(wl)
    np.testing.assert_array_equal(n, ref["num_accepted"])
    np.testing.assert_array_equal(t, ref["tokens"])
    gpu_err = sv.last_error(ws)
    assert gpu_err == ref["errors"], (gpu_err, ref["errors"])
    assert sv.last_error(ws) == 0  # reading clears the word
    gt, gn, gws = run_gpu(wl, sv.SPEC_GREEDY)
    gref = run_oracle(wl, oracle.GREEDY)
    np.testing.assert_array_equal(gn, gref["num_accepted"])
    np.testing.assert_array_equal(gt, gref["tokens"])
    assert sv.last_error(gws) == gref["errors"]


def test_tree_random_shapes_and_errors():
    rng = np.random.default_rng(17)
    for trial in range(12):
        N = int(rng.integers(1, 60))
        parents = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)
        depth = np.zeros(N, int)
        for m in range(1, N):
            depth[m] = depth[parents[m]] + 1
        D = int(depth.max())
        B, V = 3, int(rng.integers(2, 50))
        dtype = (workloads.F32, workloads.BF16)[trial % 2]
        tgt = rng.normal(0, 1, (B, N, V)).astype(np.float32)
        tgt = workloads.to_bf16_bits(tgt) if dtype == workloads.BF16 else tgt
        g = workloads.as_f32(tgt).argmax(axis=2)
        tok = np.where(rng.random((B, N)) < 0.7, g[:, np.maximum(parents, 0)],
                       rng.integers(0, V, (B, N))).astype(np.int32)
        ref = oracle.verify_tree(tgt, parents, tok, D)
        t, n, p, ws = sv.verify_tree(dev(tgt), dev(parents), dev(tok), D)
        np.testing.assert_array_equal(n.cpu().numpy(), ref["num_accepted"])
        np.testing.assert_array_equal(t.cpu().numpy(), ref["tokens"])
        np.testing.assert_array_equal(p.cpu().numpy(), ref["path"])
    # malformed trees, a too-small depth bound, bad tokens
    parents = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
    tgt = rng.normal(0, 1, (2, 7, 16)).astype(np.float32)
    tok = rng.integers(0, 16, (2, 7)).astype(np.int32)
    for par, D, tk in ((np.array([-1, 0, 3, 1, 1, 2, 2], np.int32), 2, tok),
                       (np.array([0, 0, 0, 1, 1, 2, 2], np.int32), 2, tok),
                       (parents, 1, tok),
                       (parents, 2, np.where(np.arange(7) == 4, 16, tok).astype(np.int32))):
        ref = oracle.verify_tree(tgt, par, tk, D)
        t, n, p, ws = sv.verify_tree(dev(tgt), dev(par), dev(tk), D)
        np.testing.assert_array_equal(n.cpu().numpy(), ref["num_accepted"])
        np.testing.assert_array_equal(t.cpu().numpy(), ref["tokens"])
        assert sv.last_error(ws) == ref["errors"]

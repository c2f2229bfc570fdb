"""GPU parity of stochastic tree verification (spec_verify_tree_sample)
against the oracle: tokens, depths and paths exact, except sequences the
oracle reports within 1e-5 of a decision boundary (its margin); plus the
exactness claim checked on the GPU's own outputs by chi-square."""
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
from stats import chi_square_pvalue  # noqa: E402
from test_gpu_parity import DEV, dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()
    oracle.build()


def run(tr, top_p=1.0, top_k=0):
    t, n, p, ws = sv.verify_tree_sample(dev(tr.target), dev(tr.draft), dev(tr.parents),
                                        dev(tr.node_tokens), dev(tr.uniforms), tr.D,
                                        temperature=tr.T, top_p=top_p, top_k=top_k)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy(), p.cpu().numpy(), ws


def check(tr, t, n, p, top_p=1.0, top_k=0, max_mismatch_frac=0.02):
    ref = oracle.verify_tree_sample(tr.target, tr.draft, tr.parents, tr.node_tokens, tr.uniforms,
                                    tr.D, T=tr.T, top_p=top_p, top_k=top_k)
    flags = ref["margin"] < 1e-5
    same = (n == ref["num_accepted"]) & np.all(t == ref["tokens"], 1) & np.all(p == ref["path"], 1)
    print("%s N=%d V=%d: B=%d flagged=%d mismatched=%d depths=%s" % (
        tr.name, tr.N, tr.V, tr.B, flags.sum(), (~same).sum(),
        np.bincount(np.maximum(ref["num_accepted"], 0), minlength=tr.D + 1)))
    assert not (~same & ~flags).any(), np.nonzero(~same & ~flags)[0][:10]
    assert (~same).sum() <= max(2, max_mismatch_frac * tr.B)
    return ref


def test_c5_shaped_tree():
    tr = workloads.c5s(B=64)
    t, n, p, ws = run(tr)
    check(tr, t, n, p)
    assert sv.last_error(ws) == 0


@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
@pytest.mark.parametrize("V,top_p,top_k", [(7, 1.0, 0), (1001, 0.9, 0), (4099, 1.0, 20),
                                           (30011, 0.95, 50)])
def test_shapes_and_processing(dtype, V, top_p, top_k):
    tr = workloads.c5s(seed=V, B=24, V=V, branching=3, depth=2, dtype=dtype, T=0.8, noise=0.7)
    t, n, p, _ = run(tr, top_p, top_k)
    check(tr, t, n, p, top_p, top_k, max_mismatch_frac=0.2)


def test_chain_tree_equals_chain_verify():
    """One child per node: the GPU's tree walk gives the GPU chain verify's
    tokens wherever neither is near a boundary."""
    wl = workloads.c2()
    B, k, V = wl.B, wl.k, wl.V
    parents = np.arange(-1, k, dtype=np.int32)
    tr = workloads.SampledTree("chain", B, k + 1, V, k, workloads.F32, wl.T, wl.target,
                               np.concatenate([wl.draft, wl.draft[:, :1]], axis=1), parents,
                               np.concatenate([np.zeros((B, 1), np.int32), wl.draft_tokens], 1),
                               np.concatenate([wl.uniforms[:, k:], wl.uniforms[:, :k]], 1))
    t, n, p, _ = run(tr)
    ref = check(tr, t, n, p)
    ct, cn, _ = sv.verify_sample(dev(wl.target), dev(wl.draft), dev(wl.draft_tokens),
                                 dev(wl.uniforms), temperature=wl.T)
    same = (cn.cpu().numpy() == n) & np.all(ct.cpu().numpy() == t, 1)
    assert np.all(same | (ref["margin"] < 1e-5))


def test_exactness_chi_square_on_gpu():
    """10^5 trials, three i.i.d. candidates at the root (V = 6): the GPU's
    first emitted token follows p_root."""
    rng = np.random.default_rng(12)
    V, n = 6, 100_000
    parents = np.array([-1, 0, 0, 0, 1], np.int32)
    N = len(parents)
    tgt = rng.normal(0, 1.5, (N, V)).astype(np.float32)
    drf = (tgt + rng.normal(0, 1.2, (N, V))).astype(np.float32)
    st, p0, _ = oracle.process_row(tgt[0])
    _, q0, _ = oracle.process_row(drf[0])
    _, q1, _ = oracle.process_row(drf[1])
    tok = np.zeros((n, N), np.int32)
    tok[:, 1:4] = rng.choice(V, size=(n, 3), p=q0)
    tok[:, 4] = rng.choice(V, size=n, p=q1)
    tr = workloads.SampledTree("mc", n, N, V, 2, workloads.F32, 1.0,
                               np.ascontiguousarray(np.broadcast_to(tgt, (n, N, V))),
                               np.ascontiguousarray(np.broadcast_to(drf, (n, N, V))), parents, tok,
                               workloads.uniforms(rng, (n, N)))
    t, nacc, _, _ = run(tr)
    counts = np.bincount(t[:, 0], minlength=V)
    print("first-token p-value", chi_square_pvalue(counts, p0))
    assert chi_square_pvalue(counts, p0) > 1e-4


def test_data_errors_and_wide_nodes():
    tr = workloads.c5s(seed=3, B=6, V=500, branching=2, depth=2)
    tr.target[0, 3, 7] = np.nan
    tr.node_tokens[1, 4] = tr.V
    tr.uniforms[2, 0] = 1.0
    tr.draft[3, 2, :] = -np.inf
    t, n, p, ws = run(tr)
    ref = check(tr, t, n, p)
    assert list(n[:4]) == [-1] * 4 and np.all(n[4:] >= 0)
    # a node with 65 children is refused
    N = 67
    par = np.zeros(N, np.int32)
    par[0] = -1
    par[66] = 1
    wide = workloads.SampledTree("wide", 2, N, 50, 2, workloads.F32, 1.0,
                                 np.zeros((2, N, 50), np.float32), np.zeros((2, N, 50), np.float32),
                                 par, np.ones((2, N), np.int32), np.full((2, N), 0.5, np.float32))
    _, wn, _, ws2 = run(wide)
    assert list(wn) == [-1, -1] and sv.last_error(ws2) == sv.SPEC_DATA_TREE_SHAPE

"""GPU parity of the tree attention mask / bias / position builder
(spec_verify_tree_mask) against the oracle's tree_mask: bit-exact."""
import os

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
from test_oracle_tree_mask import random_tree  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()
    oracle.build()


def run(par, pos0=None, bias=True):
    p = torch.from_numpy(np.ascontiguousarray(par, np.int32)).to(DEV)
    p0 = None if pos0 is None else torch.from_numpy(np.asarray(pos0, np.int32)).to(DEV)
    m, b, pos = sv.tree_mask(p, p0, bias=bias)
    torch.cuda.synchronize()
    return m.cpu().numpy(), None if b is None else b.cpu().numpy(), pos.cpu().numpy()


def check(par, pos0=None):
    m, b, pos = run(par, pos0)
    ref = oracle.tree_mask(par, pos0)
    np.testing.assert_array_equal(m, ref["mask"])
    np.testing.assert_array_equal(pos, ref["pos"])
    np.testing.assert_array_equal(b, np.where(ref["mask"] == 1, 0.0, -np.inf).astype(np.float32))
    return ref


def test_page_tree():
    g = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "lz_tree_mask.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                g[k] = v
    par = np.array(g["parents"], np.int32)[None]
    check(par, [7])


@pytest.mark.parametrize("N", [1, 2, 15, 16, 31, 32, 33, 85, 100, 512, 1024])
def test_random_trees(N):
    rng = np.random.default_rng(N)
    B = 5
    par = np.stack([random_tree(rng, N, max_children=4 if b % 2 else None) for b in range(B)])
    check(par, rng.integers(0, 4096, B))


def test_c5_tree_broadcast():
    tr = workloads.c5()
    par = np.broadcast_to(tr.parents, (tr.B, tr.N)).copy()
    check(par)


def test_chain_tree_full_depth():
    N = 1024
    par = (np.arange(N, dtype=np.int32) - 1)[None]
    ref = check(par, [3])
    assert ref["pos"][0, -1] == 3 + N - 1


def test_malformed_trees_in_a_batch():
    good = np.array([-1, 0, 0, 1, 1, 2, 2, 3], np.int32)
    par = np.stack([good, [0, 0, 0, 1, 1, 2, 2, 3], [-1, 0, 0, 3, 1, 2, 2, 3],
                    [-1, 0, 0, 1, -5, 2, 2, 3], good]).astype(np.int32)
    ref = check(par, [1, 2, 3, 4, 5])
    assert ref["errors"] == 1 << oracle.TREE_SHAPE


def test_outputs_optional_and_unaligned():
    rng = np.random.default_rng(4)
    N = 37  # odd N: element stores
    par = np.stack([random_tree(rng, N) for _ in range(3)])
    m, b, pos = run(par, bias=False)
    ref = oracle.tree_mask(par)
    assert b is None
    np.testing.assert_array_equal(m, ref["mask"])
    np.testing.assert_array_equal(pos, ref["pos"])
    p = torch.from_numpy(par).to(DEV)
    assert sv.spec_verify_tree_mask(p.data_ptr(), None, 3, N, None, None, None) == 0
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_tree_mask(p.data_ptr(), None, 3, 0, None, None, None)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_tree_mask(p.data_ptr(), None, 3, 1025, None, None, None)

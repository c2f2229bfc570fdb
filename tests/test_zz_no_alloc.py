"""spec_verify_sample_noalloc -- the entry point for callers that cannot
allocate device memory (an engine that plans all device memory ahead and
forbids allocation on its decode path, a plugin given no allocator) -- must
give exactly what spec_verify_sample gives with a caller-owned workspace,
call after call, through the C ABI.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test; it also passes on its own
in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

import speculative_decoding_verification_top_gb300 as sv  # noqa: E402
import workloads  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build()


def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _args(wl, mode):
    stoch = mode == sv.SPEC_STOCHASTIC
    tg, dr = _dev(wl.target), _dev(wl.draft)
    tk, un = _dev(wl.draft_tokens), _dev(wl.uniforms)
    dtype = sv.SPEC_BF16 if wl.dtype == workloads.BF16 else sv.SPEC_F32
    keep = (tg, dr, tk, un)
    return keep, (tg.data_ptr(), dr.data_ptr() if stoch else None, tk.data_ptr(),
                  un.data_ptr() if stoch else None, wl.B, wl.k, wl.V, wl.T, wl.top_p, mode, dtype)


def _outputs(wl):
    return (torch.full((wl.B, wl.k + 1), -7, dtype=torch.int32, device=DEV),
            torch.full((wl.B,), -7, dtype=torch.int32, device=DEV))


CASES = {
    "c2": lambda: workloads.c2(),
    "c3_B6": lambda: workloads.c3(B=6),
    "c4_B4_top_p": lambda: workloads.c4(B=4),
}


@pytest.mark.parametrize("mode", [sv.SPEC_STOCHASTIC, sv.SPEC_GREEDY])
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_workspace_entry_point(case, mode):
    wl = CASES[case]()
    keep, args = _args(wl, mode)
    stream = torch.cuda.current_stream().cuda_stream

    ref_t, ref_n = _outputs(wl)
    ws = sv.new_workspace(sv.spec_verify_workspace_size(wl.B, wl.k, wl.V), DEV)
    sv.spec_verify_sample(*args, ref_t.data_ptr(), ref_n.data_ptr(), ws.data_ptr(), ws.numel(),
                          stream)

    for _ in range(2):  # the shared scratch must come back clean every call
        out_t, out_n = _outputs(wl)
        sv.spec_verify_sample_noalloc(*args, out_t.data_ptr(), out_n.data_ptr(), stream)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out_n.cpu().numpy(), ref_n.cpu().numpy())
        np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t.cpu().numpy())
    assert np.all(ref_n.cpu().numpy() >= 0)


def test_noalloc_rejects_what_it_cannot_hold():
    """Batches whose workspace exceeds the fixed scratch, and bad arguments,
    are refused synchronously (fake pointers: nothing may be launched)."""
    fake = 4096
    big = sv.lib().spec_verify_sample_noalloc(fake, fake, fake, fake, 2048, 31, 1 << 22, 1.0, 1.0,
                                              sv.SPEC_STOCHASTIC, sv.SPEC_BF16, fake, fake, None)
    assert big == -7
    bad_mode = sv.lib().spec_verify_sample_noalloc(fake, fake, fake, fake, 2, 3, 100, 1.0, 1.0, 9,
                                                   sv.SPEC_F32, fake, fake, None)
    assert bad_mode == -5
    assert sv.lib().spec_verify_sample_noalloc(None, None, None, None, 0, 3, 100, 1.0, 1.0,
                                               sv.SPEC_STOCHASTIC, sv.SPEC_F32, None, None,
                                               None) == 0

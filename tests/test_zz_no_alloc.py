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
# include/spec_verify.h's status codes
SPEC_ERR_PARAM, SPEC_ERR_DTYPE, SPEC_ERR_MODE, SPEC_ERR_WORKSPACE = -3, -4, -5, -7


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


def _probe(B, k, V):
    """What the no-alloc entry point answers for batch B without launching
    anything: an invalid temperature makes it stop after the size check
    (SPEC_ERR_PARAM when the batch fits the scratch, SPEC_ERR_WORKSPACE when
    it does not); the pointers are never touched."""
    fake = 4096
    return sv.lib().spec_verify_sample_noalloc(fake, fake, fake, fake, B, k, V, -1.0, 1.0,
                                               sv.SPEC_STOCHASTIC, sv.SPEC_F32, fake, fake, None)


def test_noalloc_at_and_just_past_the_scratch_limit():
    """The largest batch the fixed scratch holds runs and matches the
    workspace entry point; one sequence more is refused with
    SPEC_ERR_WORKSPACE, before anything is enqueued."""
    k, V = 3, 32000
    lo, hi = 1, 4096
    assert _probe(lo, k, V) == SPEC_ERR_PARAM and _probe(hi, k, V) == SPEC_ERR_WORKSPACE
    while hi - lo > 1:  # lo fits, hi does not
        mid = (lo + hi) // 2
        if _probe(mid, k, V) == SPEC_ERR_PARAM:
            lo = mid
        else:
            hi = mid
    B = lo
    g = torch.Generator(device=DEV).manual_seed(1234)
    tgt = torch.randn((B, k + 1, V), generator=g, device=DEV) * 2.0
    drf = tgt[:, :k] + torch.randn((B, k, V), generator=g, device=DEV) * 0.5
    tok = torch.randint(0, V, (B, k), generator=g, device=DEV, dtype=torch.int32)
    uni = torch.rand((B, k + 1), generator=g, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = (tgt.data_ptr(), drf.data_ptr(), tok.data_ptr(), uni.data_ptr(), B, k, V, 0.8, 1.0,
            sv.SPEC_STOCHASTIC, sv.SPEC_F32)
    ref_t = torch.full((B, k + 1), -7, dtype=torch.int32, device=DEV)
    ref_n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    ws = sv.new_workspace(sv.spec_verify_workspace_size(B, k, V), DEV)
    sv.spec_verify_sample(*args, ref_t.data_ptr(), ref_n.data_ptr(), ws.data_ptr(), ws.numel(),
                          stream)
    out_t = torch.full((B, k + 1), -7, dtype=torch.int32, device=DEV)
    out_n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    sv.spec_verify_sample_noalloc(*args, out_t.data_ptr(), out_n.data_ptr(), stream)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_n.cpu().numpy(), ref_n.cpu().numpy())
    np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t.cpu().numpy())
    # one sequence more: refused, and the outputs are left alone
    B1 = B + 1
    tgt1 = torch.zeros((B1, k + 1, V), device=DEV)
    drf1 = torch.zeros((B1, k, V), device=DEV)
    tok1 = torch.zeros((B1, k), dtype=torch.int32, device=DEV)
    uni1 = torch.zeros((B1, k + 1), device=DEV)
    o_t = torch.full((B1, k + 1), -7, dtype=torch.int32, device=DEV)
    o_n = torch.full((B1,), -7, dtype=torch.int32, device=DEV)
    rc = sv.lib().spec_verify_sample_noalloc(tgt1.data_ptr(), drf1.data_ptr(), tok1.data_ptr(),
                                             uni1.data_ptr(), B1, k, V, 0.8, 1.0,
                                             sv.SPEC_STOCHASTIC, sv.SPEC_F32, o_t.data_ptr(),
                                             o_n.data_ptr(), stream)
    torch.cuda.synchronize()
    assert rc == SPEC_ERR_WORKSPACE
    assert np.all(o_n.cpu().numpy() == -7)


def test_noalloc_empty_batch_still_checks_mode_and_dtype():
    """B = 0 enqueues nothing, but a bad mode or dtype is still an error."""
    assert sv.lib().spec_verify_sample_noalloc(None, None, None, None, 0, 3, 100, 1.0, 1.0, 9,
                                               sv.SPEC_F32, None, None, None) == SPEC_ERR_MODE
    assert sv.lib().spec_verify_sample_noalloc(None, None, None, None, 0, 3, 100, 1.0, 1.0,
                                               sv.SPEC_GREEDY, 7, None, None,
                                               None) == SPEC_ERR_DTYPE

"""The C ABI on the CPU: the library builds for sm_103a, loads, exports every
function include/spec_verify.h declares, and rejects bad arguments before
touching the GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_top_gb300 as sv

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:int|const char \*)\s*(spec_\w+)\s*\(", text, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    sv.build()
    return sv.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared, "no declarations parsed"
    raw = ctypes.CDLL(sv.LIB_PATH)
    for name in declared:
        assert hasattr(raw, name), name
    assert declared == set(sv.EXPORTED)


def test_workspace_sizes(lib):
    a = sv.spec_verify_workspace_size(64, 5, 151936)
    b = sv.spec_verify_workspace_size(128, 5, 151936)
    assert 0 < a < b
    assert sv.spec_verify_workspace_size(0, 1, 1) > 0
    assert sv.spec_verify_tree_workspace_size(16, 85, 32000) > 0
    for args in [(1, 0, 10), (1, 32, 10), (1, 3, 0), (1, 3, (1 << 22) + 1), (-1, 3, 10)]:
        with pytest.raises(sv.SpecVerifyError):
            sv.spec_verify_workspace_size(*args)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_tree_workspace_size(1, 1025, 10)


def _call(**kw):
    """spec_verify_sample with fake (never dereferenced) pointers: every case
    below fails validation on the host, before any CUDA call.  The default
    workspace size is too small on purpose: the workspace check runs last, so
    a case that slipped through every other check is still refused before
    anything is enqueued."""
    a = dict(target=4096, draft=8192, toks=12288, uni=16384, B=2, k=3, V=100, T=1.0, top_p=1.0,
             mode=0, dtype=0, out_t=20480, out_n=24576, ws=32768, ws_bytes=16, stream=None)
    a.update(kw)
    rc = sv.lib().spec_verify_sample(a["target"], a["draft"], a["toks"], a["uni"], a["B"],
                                       a["k"], a["V"], a["T"], a["top_p"], a["mode"], a["dtype"],
                                       a["out_t"], a["out_n"], a["ws"], a["ws_bytes"], a["stream"])
    # The fake pointers must never reach a kernel: only a rejected call or an
    # empty batch is allowed here.
    assert rc < 0 or a["B"] == 0
    return rc


def test_argument_errors_are_synchronous(lib):
    assert _call(mode=2) == -5
    assert _call(dtype=3) == -4
    assert _call(k=0) == -2
    assert _call(k=32) == -2
    assert _call(V=0) == -2
    assert _call(B=-1) == -2
    assert _call(target=None) == -1
    assert _call(draft=None) == -1
    assert _call(uni=None) == -1
    assert _call(T=0.0) == -3
    assert _call(T=float("nan")) == -3
    assert _call(T=float("inf")) == -3
    assert _call(top_p=0.0) == -3
    assert _call(top_p=1.5) == -3
    assert _call(target=4097) == -6         # misaligned for fp32
    assert _call(ws_bytes=16) == -7
    assert _call(B=0, ws_bytes=1 << 20) == 0  # nothing to do, nothing enqueued
    assert _call(B=0, target=None, draft=None, toks=None, uni=None, out_t=None, out_n=None,
                 ws=None) == 0
    # greedy ignores the draft logits, uniforms and the sampling parameters
    assert _call(mode=1, draft=None, uni=None, T=0.0, top_p=7.0, B=0, ws_bytes=1 << 20) == 0


def test_bf16_alignment_rule(lib):
    # 2-byte aligned logits pass the bf16 check and stop at the (too small)
    # workspace; the same pointers are misaligned for fp32.
    assert _call(target=4098, draft=8194, dtype=1) == -7
    assert _call(target=4098, draft=8194, dtype=0) == -6


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, 2, 4, 8, 16, 32):
        s = sv.spec_verify_status_string(code)
        assert s and s != "unknown status", code
    assert sv.spec_verify_status_string(12345) == "unknown status"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        sv.lib()

"""GB300 (sm_103a) speculative-decoding verification: Python binding.

The compute lives in ``libspecverify.so`` (hand-written CUDA, C ABI declared
in ``include/spec_verify.h``).  This module only loads it with ctypes and
marshals arguments: every step of the verification runs in the library's
kernels.  There is no CPU fallback -- if the library is not built, every
call raises.

Entry points (same names as the C ABI):
    spec_verify_workspace_size, spec_verify_tree_workspace_size,
    spec_verify_workspace_init, spec_verify_sample, spec_verify_tree,
    spec_verify_last_error, spec_verify_intermediates,
    spec_verify_acceptance, spec_verify_sample_probs, spec_verify_tree_mask,
    spec_verify_status_string
plus tensor-level helpers ``verify_sample`` / ``verify_sample_probs`` /
``verify_tree`` / ``acceptance`` that take
torch CUDA tensors, allocate outputs and a zeroed workspace, and raise on a
negative status.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
LIB_PATH = os.path.join(_PKG, "libspecverify.so")
CSRC = os.path.join(_PKG, "csrc")
SOURCES = [os.path.join(CSRC, f)
           for f in ("api.cu", "rows.cu", "topp.cu", "final.cu", "noalloc.cu",
                     "accept.cu", "treemask.cu", "treesample.cu", "select.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("common.cuh", "stream.cuh", "draw.cuh")]
INCLUDE = os.path.join(_ROOT, "include")
HEADER = os.path.join(INCLUDE, "spec_verify.h")
BUILD_DIR = os.path.join(_PKG, "_build")

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_STOCHASTIC, SPEC_GREEDY = 0, 1
SPEC_OK = 0
SPEC_DATA_ROW_NONFINITE = 1 << 1
SPEC_DATA_ROW_ALL_NEG_INF = 1 << 2
SPEC_DATA_TOKEN_RANGE = 1 << 3
SPEC_DATA_UNIFORM_RANGE = 1 << 4
SPEC_DATA_TREE_SHAPE = 1 << 5
SPEC_DATA_PROB_RANGE = 1 << 6
SPEC_MAX_K = 31

EXPORTED = (
    "spec_verify_workspace_size",
    "spec_verify_tree_workspace_size",
    "spec_verify_workspace_init",
    "spec_verify_sample",
    "spec_verify_sample_topk",
    "spec_verify_sample_rows",
    "spec_verify_sample_finish",
    "spec_verify_sample_noalloc",
    "spec_verify_tree",
    "spec_verify_last_error",
    "spec_verify_intermediates",
    "spec_verify_acceptance",
    "spec_verify_sample_probs",
    "spec_verify_tree_mask",
    "spec_verify_tree_sample_workspace_size",
    "spec_verify_tree_sample",
    "spec_verify_status_string",
)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden"]


class SpecVerifyError(RuntimeError):
    """A negative status from the library."""


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (one nvcc per translation unit,
    in parallel) and link libspecverify.so in-tree."""
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS + [HEADER])
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = "%d" % os.getpid()
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + "." + tag + ".o")
        cmd = ["nvcc", *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("nvcc failed")
    tmp = LIB_PATH + "." + tag + ".tmp"
    subprocess.check_call(["nvcc", *ARCH, "-shared", *objs, "-o", tmp])
    os.replace(tmp, LIB_PATH)
    for obj in objs:
        os.unlink(obj)
    return LIB_PATH


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libspecverify.so is not built (run speculative_decoding_verification_top_gb300"
                ".build()); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.spec_verify_workspace_size.argtypes = [I, I, I, ctypes.POINTER(Z)]
        L.spec_verify_tree_workspace_size.argtypes = [I, I, I, ctypes.POINTER(Z)]
        L.spec_verify_workspace_init.argtypes = [P, Z, P]
        for name in ("spec_verify_sample", "spec_verify_sample_rows", "spec_verify_sample_finish"):
            getattr(L, name).argtypes = [P, P, P, P, I, I, I, F, F, I, I, P, P, P, Z, P]
        L.spec_verify_sample_topk.argtypes = [P, P, P, P, I, I, I, F, F, I, I, I, P, P, P, Z, P]
        L.spec_verify_sample_noalloc.argtypes = [P, P, P, P, I, I, I, F, F, I, I, P, P, P]
        L.spec_verify_tree.argtypes = [P, P, P, I, I, I, I, I, P, P, P, P, Z, P]
        L.spec_verify_last_error.argtypes = [P, Z, P]
        L.spec_verify_intermediates.argtypes = [P, Z, I, I, I, P, P, P, P, P]
        L.spec_verify_acceptance.argtypes = [P, P, I, I, I, F, F, I, I, P, P, P, Z, P]
        L.spec_verify_sample_probs.argtypes = [P, P, P, P, I, I, I, F, F, I, I, P, P, P, Z, P]
        L.spec_verify_tree_mask.argtypes = [P, P, I, I, P, P, P, P]
        L.spec_verify_tree_sample_workspace_size.argtypes = [I, I, I, ctypes.POINTER(Z)]
        L.spec_verify_tree_sample.argtypes = [P, P, P, P, P, I, I, I, I, F, F, I, I, P, P, P, P,
                                              Z, P]
        L.spec_verify_status_string.argtypes = [I]
        L.spec_verify_status_string.restype = ctypes.c_char_p
        for name in EXPORTED[:-1]:
            getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(rc):
    if rc < 0:
        raise SpecVerifyError("%d: %s" % (rc, spec_verify_status_string(rc)))
    return rc


# ----------------------------------------------------- C ABI, same names

def spec_verify_workspace_size(B, k, V):
    out = ctypes.c_size_t(0)
    _check(lib().spec_verify_workspace_size(B, k, V, ctypes.byref(out)))
    return out.value


def spec_verify_tree_workspace_size(B, N, V):
    out = ctypes.c_size_t(0)
    _check(lib().spec_verify_tree_workspace_size(B, N, V, ctypes.byref(out)))
    return out.value


def spec_verify_workspace_init(workspace_ptr, nbytes, stream=0):
    return _check(lib().spec_verify_workspace_init(workspace_ptr, nbytes, stream))


def spec_verify_sample(target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, temperature,
                       top_p, mode, dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
                       workspace_bytes, stream=0):
    return _check(lib().spec_verify_sample(
        target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), mode, dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
        workspace_bytes, stream))


def spec_verify_sample_topk(target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V,
                            temperature, top_p, top_k, mode, dtype, out_tokens_ptr, out_num_ptr,
                            workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_sample_topk(
        target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), int(top_k), mode, dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
        workspace_bytes, stream))


def spec_verify_sample_rows(target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V,
                            temperature, top_p, mode, dtype, out_tokens_ptr, out_num_ptr,
                            workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_sample_rows(
        target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), mode, dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
        workspace_bytes, stream))


def spec_verify_sample_finish(target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V,
                              temperature, top_p, mode, dtype, out_tokens_ptr, out_num_ptr,
                              workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_sample_finish(
        target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), mode, dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
        workspace_bytes, stream))


def spec_verify_sample_noalloc(target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V,
                               temperature, top_p, mode, dtype, out_tokens_ptr, out_num_ptr,
                               stream=0):
    """spec_verify_sample without a workspace, for callers that cannot
    allocate device memory: the library's fixed 4 MiB per-device scratch is
    used instead (calls that overlap on the GPU race on it)."""
    return _check(lib().spec_verify_sample_noalloc(
        target_ptr, draft_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), mode, dtype, out_tokens_ptr, out_num_ptr, stream))


def spec_verify_tree(target_ptr, parents_ptr, node_tokens_ptr, B, N, V, D, dtype,
                     out_tokens_ptr, out_num_ptr, out_path_ptr, workspace_ptr, workspace_bytes,
                     stream=0):
    return _check(lib().spec_verify_tree(
        target_ptr, parents_ptr, node_tokens_ptr, B, N, V, D, dtype, out_tokens_ptr,
        out_num_ptr, out_path_ptr, workspace_ptr, workspace_bytes, stream))


def spec_verify_last_error(workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_last_error(workspace_ptr, workspace_bytes, stream))


def spec_verify_intermediates(workspace_ptr, workspace_bytes, B, k, V, P_ptr, Q_ptr, Z_ptr,
                              S_ptr, stream=0):
    return _check(lib().spec_verify_intermediates(workspace_ptr, workspace_bytes, B, k, V,
                                                  P_ptr, Q_ptr, Z_ptr, S_ptr, stream))


def spec_verify_acceptance(target_ptr, draft_ptr, B, k, V, temperature, top_p, top_k, dtype,
                           out_beta_ptr, out_tv_ptr, workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_acceptance(
        target_ptr, draft_ptr, B, k, V, float(temperature), float(top_p), int(top_k), dtype,
        out_beta_ptr, out_tv_ptr, workspace_ptr, workspace_bytes, stream))


def spec_verify_sample_probs(target_ptr, draft_probs_ptr, tokens_ptr, uniforms_ptr, B, k, V,
                             temperature, top_p, top_k, dtype, out_tokens_ptr, out_num_ptr,
                             workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_sample_probs(
        target_ptr, draft_probs_ptr, tokens_ptr, uniforms_ptr, B, k, V, float(temperature),
        float(top_p), int(top_k), dtype, out_tokens_ptr, out_num_ptr, workspace_ptr,
        workspace_bytes, stream))


def spec_verify_tree_mask(parents_ptr, pos0_ptr, B, N, out_mask_ptr, out_bias_ptr, out_pos_ptr,
                          stream=0):
    return _check(lib().spec_verify_tree_mask(parents_ptr, pos0_ptr, B, N, out_mask_ptr,
                                              out_bias_ptr, out_pos_ptr, stream))


def spec_verify_tree_sample_workspace_size(B, N, V):
    out = ctypes.c_size_t(0)
    _check(lib().spec_verify_tree_sample_workspace_size(B, N, V, ctypes.byref(out)))
    return out.value


def spec_verify_tree_sample(target_ptr, draft_ptr, parents_ptr, node_tokens_ptr, uniforms_ptr,
                            B, N, V, D, temperature, top_p, top_k, dtype, out_tokens_ptr,
                            out_num_ptr, out_path_ptr, workspace_ptr, workspace_bytes, stream=0):
    return _check(lib().spec_verify_tree_sample(
        target_ptr, draft_ptr, parents_ptr, node_tokens_ptr, uniforms_ptr, B, N, V, D,
        float(temperature), float(top_p), int(top_k), dtype, out_tokens_ptr, out_num_ptr,
        out_path_ptr, workspace_ptr, workspace_bytes, stream))


def spec_verify_status_string(status):
    return lib().spec_verify_status_string(int(status)).decode()


# ------------------------------------------------- torch tensor helpers

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError("logits must be torch.float32 or torch.bfloat16, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, name, dtype, shape):
    torch = _torch()
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s, got %s %s"
                         % (name, dtype, tuple(shape), t.dtype, tuple(t.shape)))


def new_workspace(nbytes, device):
    """A zero-filled workspace tensor (zeroing is the required first-use init)."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def verify_sample(target, draft, draft_tokens, uniforms, temperature=1.0, top_p=1.0,
                  mode=SPEC_STOCHASTIC, out_tokens=None, out_num=None, workspace=None,
                  stream=None, top_k=0):
    """Tensor-level spec_verify_sample.  Returns (out_tokens [B, k+1],
    out_num_accepted [B], workspace)."""
    torch = _torch()
    B, k1, V = target.shape
    k = k1 - 1
    dt = _dtype_code(target)
    _need(target, "target", target.dtype, (B, k + 1, V))
    if mode == SPEC_STOCHASTIC:
        _need(draft, "draft", target.dtype, (B, k, V))
        _need(uniforms, "uniforms", torch.float32, (B, k + 1))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num is None:
        out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_size(B, k, V)
    if workspace is None:
        workspace = new_workspace(nbytes, dev)
    stoch = mode == SPEC_STOCHASTIC
    args = (_ptr(target), _ptr(draft) if stoch else None, _ptr(draft_tokens),
            _ptr(uniforms) if stoch else None, B, k, V, temperature, top_p)
    tail = (mode, dt, _ptr(out_tokens), _ptr(out_num), _ptr(workspace), workspace.numel(),
            _stream(stream))
    if top_k:
        spec_verify_sample_topk(*args, top_k, *tail)
    else:
        spec_verify_sample(*args, *tail)
    return out_tokens, out_num, workspace


def verify_sample_probs(target, draft_probs, draft_tokens, uniforms, temperature=1.0, top_p=1.0,
                        out_tokens=None, out_num=None, workspace=None, stream=None, top_k=0):
    """Tensor-level spec_verify_sample_probs (draft given as fp32
    probabilities [B, k, V]).  Returns (out_tokens, out_num_accepted,
    workspace)."""
    torch = _torch()
    B, k1, V = target.shape
    k = k1 - 1
    dt = _dtype_code(target)
    _need(target, "target", target.dtype, (B, k + 1, V))
    _need(draft_probs, "draft_probs", torch.float32, (B, k, V))
    _need(uniforms, "uniforms", torch.float32, (B, k + 1))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num is None:
        out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(spec_verify_workspace_size(B, k, V), dev)
    spec_verify_sample_probs(_ptr(target), _ptr(draft_probs), _ptr(draft_tokens), _ptr(uniforms),
                             B, k, V, temperature, top_p, top_k, dt, _ptr(out_tokens),
                             _ptr(out_num),
                             _ptr(workspace), workspace.numel(), _stream(stream))
    return out_tokens, out_num, workspace


def verify_tree(target, parents, node_tokens, depth, out_tokens=None, out_num=None,
                out_path=None, workspace=None, stream=None):
    """Tensor-level spec_verify_tree.  Returns (out_tokens [B, D+1],
    out_num_accepted [B], out_path [B, D+1], workspace)."""
    torch = _torch()
    B, N, V = target.shape
    dt = _dtype_code(target)
    _need(target, "target", target.dtype, (B, N, V))
    _need(parents, "parents", torch.int32, (N,))
    _need(node_tokens, "node_tokens", torch.int32, (B, N))
    dev = target.device
    W = depth + 1
    if out_tokens is None:
        out_tokens = torch.empty((B, W), dtype=torch.int32, device=dev)
    if out_num is None:
        out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_path is None:
        out_path = torch.empty((B, W), dtype=torch.int32, device=dev)
    nbytes = spec_verify_tree_workspace_size(B, N, V)
    if workspace is None:
        workspace = new_workspace(nbytes, dev)
    spec_verify_tree(_ptr(target), _ptr(parents), _ptr(node_tokens), B, N, V, depth, dt,
                     _ptr(out_tokens), _ptr(out_num), _ptr(out_path), _ptr(workspace),
                     workspace.numel(), _stream(stream))
    return out_tokens, out_num, out_path, workspace


def last_error(workspace, stream=None):
    return spec_verify_last_error(_ptr(workspace), workspace.numel(), _stream(stream))


def intermediates(workspace, B, k, V, stream=None):
    """(P [B, k], Q [B, k], Z [B, 2k+1], S [B]) of the last stochastic call."""
    torch = _torch()
    dev = workspace.device
    P = torch.empty((B, k), dtype=torch.float32, device=dev)
    Q = torch.empty((B, k), dtype=torch.float32, device=dev)
    Z = torch.empty((B, 2 * k + 1), dtype=torch.float32, device=dev)
    S = torch.empty((B,), dtype=torch.float32, device=dev)
    spec_verify_intermediates(_ptr(workspace), workspace.numel(), B, k, V, _ptr(P), _ptr(Q),
                              _ptr(Z), _ptr(S), _stream(stream))
    return P, Q, Z, S


def acceptance(target, draft, workspace, temperature=1.0, top_p=1.0, out_beta=None, out_tv=None,
               stream=None, top_k=0):
    """Tensor-level spec_verify_acceptance: (beta [B, k], tv [B, k]) of the
    last stochastic verify call made on `workspace` with these arguments."""
    torch = _torch()
    B, k1, V = target.shape
    k = k1 - 1
    dt = _dtype_code(target)
    _need(target, "target", target.dtype, (B, k + 1, V))
    _need(draft, "draft", target.dtype, (B, k, V))
    dev = target.device
    if out_beta is None:
        out_beta = torch.empty((B, k), dtype=torch.float32, device=dev)
    if out_tv is None:
        out_tv = torch.empty((B, k), dtype=torch.float32, device=dev)
    spec_verify_acceptance(_ptr(target), _ptr(draft), B, k, V, temperature, top_p, top_k, dt,
                           _ptr(out_beta), _ptr(out_tv), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    return out_beta, out_tv


def tree_mask(parents, pos0=None, mask=True, bias=False, pos=True, stream=None):
    """Tensor-level spec_verify_tree_mask: parents [B, N] int32 (CUDA).
    Returns (mask [B, N, N] uint8 or None, bias [B, N, N] fp32 or None,
    pos [B, N] int32 or None)."""
    torch = _torch()
    B, N = parents.shape
    _need(parents, "parents", torch.int32, (B, N))
    if pos0 is not None:
        _need(pos0, "pos0", torch.int32, (B,))
    dev = parents.device
    m = torch.empty((B, N, N), dtype=torch.uint8, device=dev) if mask else None
    bs = torch.empty((B, N, N), dtype=torch.float32, device=dev) if bias else None
    p = torch.empty((B, N), dtype=torch.int32, device=dev) if pos else None
    spec_verify_tree_mask(_ptr(parents), _ptr(pos0), B, N, _ptr(m), _ptr(bs), _ptr(p),
                          _stream(stream))
    return m, bs, p


def verify_tree_sample(target, draft, parents, node_tokens, uniforms, depth, temperature=1.0,
                       top_p=1.0, top_k=0, workspace=None, stream=None):
    """Tensor-level spec_verify_tree_sample.  Returns (out_tokens [B, D+1],
    out_num_accepted [B], out_path [B, D+1], workspace)."""
    torch = _torch()
    B, N, V = target.shape
    dt = _dtype_code(target)
    _need(target, "target", target.dtype, (B, N, V))
    _need(draft, "draft", target.dtype, (B, N, V))
    _need(parents, "parents", torch.int32, (N,))
    _need(node_tokens, "node_tokens", torch.int32, (B, N))
    _need(uniforms, "uniforms", torch.float32, (B, N))
    dev = target.device
    W = depth + 1
    out_t = torch.empty((B, W), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    out_p = torch.empty((B, W), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(spec_verify_tree_sample_workspace_size(B, N, V), dev)
    spec_verify_tree_sample(_ptr(target), _ptr(draft), _ptr(parents), _ptr(node_tokens),
                            _ptr(uniforms), B, N, V, depth, temperature, top_p, top_k, dt,
                            _ptr(out_t), _ptr(out_n), _ptr(out_p), _ptr(workspace),
                            workspace.numel(), _stream(stream))
    return out_t, out_n, out_p, workspace
